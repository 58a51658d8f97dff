"""Helpers shared by the GPU tests: upload a synth.DecodeCase, run the library,
and compare with the fp64 oracle."""
from __future__ import annotations

import numpy as np
import torch

import mla_latent_kv_15_gb300 as mla
import oracle

LKV, DQK = 512, 576
TOL_OUT_BF16 = 2e-2     # max abs error of the bf16 latent output
TOL_LSE = 1e-3          # max abs error of the LSE
TOL_OUT_FP8 = 6e-2      # fp8 cache, against the oracle on dequantised values


def bf16_tensor(bits: np.ndarray, dev="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev).view(torch.bfloat16)


class GpuCase:
    """Device copies of a case; the cache is prepared by the library itself
    (bf16: a copy of the drawn pool; fp8: mla_cache_write of every referenced
    row), then the step's new rows are written with mla_cache_write."""

    def __init__(self, case, write_new: bool = True, num_splits_max: int = 0):
        self.case = case
        dev = "cuda"
        if case.cache_dtype == "bf16":
            self.cache = bf16_tensor(case.pool, dev)
        else:
            self.cache = torch.full(case.pool.shape, 0x7F, dtype=torch.uint8, device=dev).view(torch.float8_e4m3fn)
            slots = torch.from_numpy(case.referenced_slots).to(dev)
            flat = case.pool.reshape(-1, DQK)
            rows = flat[case.referenced_slots]
            mla.cache_write(bf16_tensor(np.ascontiguousarray(rows[:, :LKV])),
                            bf16_tensor(np.ascontiguousarray(rows[:, LKV:])), slots, self.cache, case.kv_scale)
        self.q_abs = bf16_tensor(case.q_abs, dev)
        self.q_pe = bf16_tensor(case.q_pe, dev)
        self.block_table = torch.from_numpy(case.block_table).to(dev)
        self.seq_lens = torch.from_numpy(case.seq_lens).to(dev)
        self.qsl = torch.from_numpy(case.query_start_loc).to(dev)
        self.new_kv_c = bf16_tensor(case.new_kv_c, dev)
        self.new_k_pe = bf16_tensor(case.new_k_pe, dev)
        self.slots = torch.from_numpy(case.slot_mapping).to(dev)
        T, N = case.total_q, case.num_heads
        self.out = torch.full((T, N, LKV), float("nan"), dtype=torch.bfloat16, device=dev)
        self.lse = torch.full((T, N), float("nan"), dtype=torch.float32, device=dev)
        ws = mla.decode_workspace_size(case.batch, T, N, num_splits_max)
        self.workspace = torch.empty(ws, dtype=torch.uint8, device=dev)
        if write_new:
            self.write_new()

    def write_new(self):
        mla.cache_write(self.new_kv_c, self.new_k_pe, self.slots, self.cache, self.case.kv_scale)

    def decode(self, num_splits: int = 0):
        c = self.case
        mla.decode(self.q_abs, self.q_pe, self.cache, self.block_table, self.seq_lens, self.out, self.workspace,
                   scale=c.scale, query_start_loc=self.qsl, lse=self.lse, num_splits=num_splits,
                   kv_scale=c.kv_scale)
        torch.cuda.synchronize()
        return self.out, self.lse


def compare(case, gpu: GpuCase, rows=None, cache_host=None, tol_out=None):
    """Max |gpu - oracle| over the given flattened query rows (default all)."""
    if cache_host is None:
        cache_host = oracle.prepare_cache(case)
    ref_o, ref_lse, _ = oracle.decode_case(case, cache_host, rows=rows)
    out = gpu.out.float().reshape(-1, LKV).cpu().numpy().astype(np.float64)
    lse = gpu.lse.reshape(-1).cpu().numpy().astype(np.float64)
    if rows is not None:
        out, lse = out[rows], lse[rows]
    assert np.all(np.isfinite(out)), "non-finite latent output"
    err_o = float(np.max(np.abs(out - ref_o))) if out.size else 0.0
    fin = np.isfinite(ref_lse)
    assert np.array_equal(np.isfinite(lse), fin), "LSE finiteness differs from the oracle"
    assert np.all(lse[~fin] == -np.inf)
    err_l = float(np.max(np.abs(lse[fin] - ref_lse[fin]))) if fin.any() else 0.0
    tol = tol_out if tol_out is not None else (TOL_OUT_BF16 if case.cache_dtype == "bf16" else TOL_OUT_FP8)
    assert err_o <= tol, f"latent output error {err_o:.3g} > {tol}"
    assert err_l <= TOL_LSE, f"LSE error {err_l:.3g} > {TOL_LSE}"
    return err_o, err_l


def sample_rows(case, n: int, seed: int = 0) -> np.ndarray:
    """n flattened query rows spread over all requests (first/last head of
    every request plus random ones)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    N = case.num_heads
    qsl = case.query_start_loc
    rows = set()
    for b in range(case.batch):
        for t in range(qsl[b], qsl[b + 1]):
            rows.add(t * N)
            rows.add(t * N + N - 1)
    total = case.total_q * N
    extra = rng.choice(total, size=min(n, total), replace=False)
    rows.update(int(r) for r in extra)
    return np.array(sorted(rows), dtype=np.int64)
