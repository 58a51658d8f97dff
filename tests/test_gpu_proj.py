"""GPU parity of the per-head projections (query absorption and value
up-projection, tcgen05) against the fp64 oracle's einsums.

Bar: every element within 2^-8 * |ref| + 1e-4 of the fp64 result on the same
bf16 inputs.  The kernels accumulate in float32 and round the result to bf16
once (nearest even: at most half a bf16 ulp, 2^-8 relative); the float32
accumulation of <= 1024 products of values below 4 stays far below 1e-4.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import synth
from oracle import expanded

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import mla_latent_kv_15_gb300 as mla
    from gpu_case import GpuCase, bf16_tensor, LKV


def f64(bits):
    return oracle.bf16_to_f64(bits)


def check(got: torch.Tensor, ref: np.ndarray):
    g = got.float().cpu().numpy().astype(np.float64)
    assert g.shape == ref.shape
    assert np.all(np.isfinite(g))
    err = np.abs(g - ref)
    bound = 2.0 ** -8 * np.abs(ref) + 1e-4
    worst = np.unravel_index(np.argmax(err - bound), err.shape)
    assert np.all(err <= bound), f"error {err[worst]:.3g} > {bound[worst]:.3g} at {worst}"


@pytest.mark.parametrize("T,N,V", [(1, 1, 128), (5, 16, 128), (64, 128, 128), (130, 3, 64), (257, 2, 192),
                                   (33, 4, 256), (7, 2, 512), (70, 2, 1024), (600, 4, 128)])
def test_v_up_proj(T, N, V):
    """out[t, n, :] = o_lat[t, n, :] @ W_UV[n]: token tiles with ragged tails,
    every supported width (one and several column tiles)."""
    _, w_uv = synth.projection_weights(T + N + V, N, v=V)          # [L, N, V]
    o_lat = synth.bf16_normal(T * 7 + N, (T, N, LKV))
    ref = expanded.up_project(f64(o_lat), f64(w_uv))
    out = torch.full((T, N, V), float("nan"), dtype=torch.bfloat16, device="cuda")
    w_dev = bf16_tensor(np.ascontiguousarray(w_uv.transpose(1, 0, 2)))   # (N, L, V) as stored for the bmm
    mla.v_up_proj(bf16_tensor(o_lat), w_dev, out)
    torch.cuda.synchronize()
    check(out, ref)
    assert mla.proj_status() == 0


@pytest.mark.parametrize("T,N,P,stride", [(1, 1, 128, 128), (64, 128, 128, 192), (130, 16, 128, 192),
                                          (9, 3, 64, 64), (200, 2, 256, 320), (3, 2, 1024, 1024),
                                          (300, 8, 512, 576)])
def test_q_absorb(T, N, P, stride):
    """ql_nope[t, n, :] = q_nope[t, n, :] @ W_UK_T[n], q_nope read as the first
    P columns of wider rows (q = [q_nope | q_pe]) when stride > P."""
    w_uk, _ = synth.projection_weights(T + N + P, N, p=P)           # [L, N, P]
    q = synth.bf16_normal(T * 5 + P, (T, N, stride))
    ref = expanded.absorb_query(f64(q[:, :, :P]), f64(w_uk))
    q_dev = bf16_tensor(q)
    ql = torch.full((T, N, LKV), float("nan"), dtype=torch.bfloat16, device="cuda")
    w_dev = bf16_tensor(np.ascontiguousarray(w_uk.transpose(1, 2, 0)))   # (N, P, L) as stored for the bmm
    mla.q_absorb(q_dev[:, :, :P], w_dev, ql)
    torch.cuda.synchronize()
    check(ql, ref)
    assert mla.proj_status() == 0


def test_projection_empty_batch_is_a_no_op():
    w = torch.zeros((2, 512, 128), dtype=torch.bfloat16, device="cuda")
    x = torch.zeros((0, 2, 512), dtype=torch.bfloat16, device="cuda")
    y = torch.zeros((0, 2, 128), dtype=torch.bfloat16, device="cuda")
    mla.v_up_proj(x, w, y)
    mla.q_absorb(torch.zeros((0, 2, 128), dtype=torch.bfloat16, device="cuda"),
                 torch.zeros((2, 128, 512), dtype=torch.bfloat16, device="cuda"),
                 torch.zeros((0, 2, 512), dtype=torch.bfloat16, device="cuda"))
    torch.cuda.synchronize()
    assert mla.proj_status() == 0


def test_projection_output_tail_untouched():
    """Rows past num_tokens (the zero-filled tail of the last token tile) are
    never written."""
    T, N, V = 3, 2, 128
    _, w_uv = synth.projection_weights(1, N, v=V)
    o_lat = synth.bf16_normal(2, (T, N, LKV))
    buf = torch.full((T + 125, N, V), 7.0, dtype=torch.bfloat16, device="cuda")
    mla.v_up_proj(bf16_tensor(o_lat), bf16_tensor(np.ascontiguousarray(w_uv.transpose(1, 0, 2))), buf[:T])
    torch.cuda.synchronize()
    assert torch.all(buf[T:] == 7.0)
    check(buf[:T], expanded.up_project(f64(o_lat), f64(w_uv)))


def test_absorbed_chain_matches_expanded_mha():
    """q_absorb -> cache write -> decode -> v_up_proj on the GPU against the
    oracle's compute-friendly MHA (expanded keys and values): the two
    approaches of the MLA pages agree.  Bar: 2e-2 on the up-projected output
    (the decode's bf16 output bar; W_UV columns have unit expected norm) and
    1e-3 on the LSE."""
    N, P, V = 16, 128, 128
    case = synth.make_decode_case(num_heads=N, batch=3, ctx=(100, 400), sq=[1, 3, 2], page_size=64, seed=61,
                                  poison=False)
    w_uk, w_uv = synth.projection_weights(61, N, p=P, v=V)
    T = case.total_q
    q_nope = synth.bf16_normal(62, (T, N, P))
    g = GpuCase(case)
    # replace the drawn absorbed query with the absorption of q_nope
    mla.q_absorb(bf16_tensor(q_nope), bf16_tensor(np.ascontiguousarray(w_uk.transpose(1, 2, 0))), g.q_abs)
    g.decode()
    out = torch.empty((T, N, V), dtype=torch.bfloat16, device="cuda")
    mla.v_up_proj(g.out, bf16_tensor(np.ascontiguousarray(w_uv.transpose(1, 0, 2))), out)
    torch.cuda.synchronize()
    assert mla.decode_status(g.workspace) == 0 and mla.proj_status() == 0

    cache = oracle.prepare_cache(case)
    got = out.float().cpu().numpy().astype(np.float64)
    lse = g.lse.cpu().numpy().astype(np.float64)
    q_pe = f64(case.q_pe)
    for b in range(case.batch):
        L = int(case.seq_lens[b])
        pos = np.arange(L)
        rows = f64(cache[case.block_table[b, pos // case.page_size], pos % case.page_size])
        t0, t1 = int(case.query_start_loc[b]), int(case.query_start_loc[b + 1])
        sq = t1 - t0
        visible = [L - sq + 1 + t for t in range(sq)]
        o_exp, lse_exp = expanded.expanded_mha(f64(q_nope[t0:t1]), q_pe[t0:t1], rows[:, :LKV], rows[:, LKV:],
                                               f64(w_uk), f64(w_uv), case.scale, visible)
        assert np.max(np.abs(got[t0:t1] - o_exp)) <= 2e-2
        assert np.max(np.abs(lse[t0:t1] - lse_exp)) <= 1e-3
