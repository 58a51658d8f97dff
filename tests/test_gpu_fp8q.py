"""GPU parity of the e4m3-query decode (fp8 x fp8 score MMAs over an e4m3
cache) against the fp64 oracle run on the same quantised query and the
dequantised cache.  Bar: the e4m3-cache bar, 6e-2 on the latent output and
1e-3 on the LSE."""
import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import mla_latent_kv_15_gb300 as mla
    from gpu_case import GpuCase, sample_rows, LKV, DQK


def q_rows(case):
    """bf16 bits of [q_abs | q_pe], [T, N, 576]."""
    return np.ascontiguousarray(np.concatenate([case.q_abs, case.q_pe], axis=-1))


def run_fp8q(case, num_splits=0, rows=None, quantize_on_gpu=False):
    g = GpuCase(case, num_splits_max=num_splits)
    qb = q_rows(case)
    q_scale = float(np.float32(np.abs(oracle.bf16_to_f64(qb)).max() / 448.0))
    codes = oracle.quantize_fp8(qb, q_scale)                     # the oracle's own quantisation
    if quantize_on_gpu:
        # the library's scaled_fp8_quant straight into [q_abs | q_pe] rows (bit-identical codes)
        g8 = torch.empty(codes.shape, dtype=torch.uint8, device="cuda")
        mla.quantize_fp8(g.q_abs, q_scale, g8[..., :LKV])
        mla.quantize_fp8(g.q_pe, q_scale, g8[..., LKV:])
        torch.cuda.synchronize()
        assert np.array_equal(g8.cpu().numpy(), codes)
    q8 = torch.from_numpy(codes).cuda()
    mla.decode_fp8q(q8, q_scale, g.cache, g.block_table, g.seq_lens, g.out, g.workspace, scale=case.scale,
                    query_start_loc=g.qsl, lse=g.lse, num_splits=num_splits, kv_scale=case.kv_scale)
    torch.cuda.synchronize()
    assert mla.decode_status(g.workspace) == 0
    # oracle on the dequantised query (codes x q_scale) and the dequantised cache
    qf = oracle.e4m3_to_f64(codes) * np.float64(np.float32(q_scale))
    cache = oracle.prepare_cache(case)
    ref_o, ref_lse, _ = oracle.decode(qf, cache, case.page_size, oracle.CACHE_E4M3, case.kv_scale, case.block_table,
                                      case.seq_lens, case.query_start_loc, case.num_heads, case.scale, rows=rows)
    out = g.out.float().reshape(-1, LKV).cpu().numpy().astype(np.float64)
    lse = g.lse.reshape(-1).cpu().numpy().astype(np.float64)
    if rows is not None:
        out, lse = out[rows], lse[rows]
    assert np.all(np.isfinite(out))
    fin = np.isfinite(ref_lse)
    assert np.array_equal(np.isfinite(lse), fin)
    err_o = float(np.max(np.abs(out - ref_o)))
    err_l = float(np.max(np.abs(lse[fin] - ref_lse[fin]))) if fin.any() else 0.0
    assert err_o <= 6e-2, err_o
    assert err_l <= 1e-3, err_l
    return err_o, err_l


@pytest.mark.parametrize("num_heads,sq,page_size,num_splits", [
    (16, 1, 64, 0), (128, 1, 64, 0), (128, 4, 64, 0), (128, [4, 1, 1, 2, 1, 3], 16, 2), (20, 2, 32, 3),
])
def test_decode_fp8q_small(num_heads, sq, page_size, num_splits):
    case = synth.make_decode_case(num_heads=num_heads, batch=6, ctx=(60, 700), sq=sq, page_size=page_size,
                                  cache_dtype="fp8", seed=500 + num_heads + page_size + num_splits)
    run_fp8q(case, num_splits)


def test_decode_fp8q_full_size():
    case = synth.workload("dsv3_n128_b64_ctx1k-8k_fp8")
    run_fp8q(case, 0, rows=sample_rows(case, 300, seed=9), quantize_on_gpu=True)


def test_decode_fp8q_negative_scale():
    case = synth.make_decode_case(num_heads=16, batch=4, ctx=(60, 500), page_size=64, cache_dtype="fp8", seed=46)
    case.scale = -case.scale
    run_fp8q(case)


@pytest.mark.parametrize("seed", range(12))
def test_random_configuration_fp8q(seed):
    """The randomized sweep's configurations (head counts, page sizes,
    multi-token mixes, splits, ragged pools) through the e4m3-query decode."""
    from test_gpu_random import draw
    kw, splits = draw(100 + seed)
    kw["cache_dtype"] = "fp8"
    case = synth.make_decode_case(**kw)
    rows = sample_rows(case, 400, seed=seed) if case.total_q * case.num_heads > 3000 else None
    run_fp8q(case, splits, rows=rows)


@pytest.mark.parametrize("num_heads,sq,num_splits", [(128, 1, 0), (16, [1, 3, 2], 2)])
def test_decode_fp8q_step(num_heads, sq, num_splits):
    """mla_decode_fp8q_step: its cache rows and query codes equal those of
    mla_cache_write and mla_quantize_fp8 byte for byte, and its decode meets
    the e4m3 bar against the oracle on its quantised query."""
    case = synth.make_decode_case(num_heads=num_heads, batch=3, ctx=(200, 1200), sq=sq, page_size=64,
                                  cache_dtype="fp8", seed=730 + num_heads, poison=False)
    qb = q_rows(case)
    q_scale = float(np.float32(np.abs(oracle.bf16_to_f64(qb)).max() / 448.0))
    codes = oracle.quantize_fp8(qb, q_scale)
    ref = GpuCase(case, write_new=False, num_splits_max=num_splits)
    mla.cache_write(ref.new_kv_c, ref.new_k_pe, ref.slots, ref.cache, case.kv_scale)
    g = GpuCase(case, write_new=False, num_splits_max=num_splits)
    q8 = torch.zeros(codes.shape, dtype=torch.uint8, device="cuda")
    mla.decode_fp8q_step(g.new_kv_c, g.new_k_pe, g.slots, g.q_abs, g.q_pe, q_scale, q8, g.cache, g.block_table,
                         g.seq_lens, g.out, g.workspace, scale=case.scale, query_start_loc=g.qsl, lse=g.lse,
                         num_splits=num_splits, kv_scale=case.kv_scale)
    torch.cuda.synchronize()
    assert mla.decode_status(g.workspace) == 0
    assert torch.equal(g.cache.view(torch.uint8), ref.cache.view(torch.uint8))
    assert np.array_equal(q8.cpu().numpy(), codes)
    qf = oracle.e4m3_to_f64(codes) * np.float64(np.float32(q_scale))
    ref_o, ref_lse, _ = oracle.decode(qf, oracle.prepare_cache(case), case.page_size, oracle.CACHE_E4M3,
                                      case.kv_scale, case.block_table, case.seq_lens, case.query_start_loc,
                                      case.num_heads, case.scale)
    out = g.out.float().reshape(-1, LKV).cpu().numpy().astype(np.float64)
    lse = g.lse.reshape(-1).cpu().numpy().astype(np.float64)
    fin = np.isfinite(ref_lse)
    assert np.array_equal(np.isfinite(lse), fin)
    assert float(np.max(np.abs(out - ref_o))) <= 6e-2
    assert (float(np.max(np.abs(lse[fin] - ref_lse[fin]))) if fin.any() else 0.0) <= 1e-3


def test_decode_fp8q_step_full_size():
    """The e4m3-query step at the full DeepSeek-V3-shaped size (the query's
    quantisation blocks stride over 589 824 vectors): every query code equals
    the oracle's, the cache equals mla_cache_write's, and sampled rows meet the
    e4m3 bar."""
    case = synth.workload("dsv3_n128_b64_ctx1k-8k_fp8")
    qb = q_rows(case)
    q_scale = float(np.float32(np.abs(oracle.bf16_to_f64(qb)).max() / 448.0))
    codes = oracle.quantize_fp8(qb, q_scale)
    g = GpuCase(case, write_new=False)
    ref_cache = g.cache.clone()
    mla.cache_write(g.new_kv_c, g.new_k_pe, g.slots, ref_cache, case.kv_scale)
    q8 = torch.zeros(codes.shape, dtype=torch.uint8, device="cuda")
    mla.decode_fp8q_step(g.new_kv_c, g.new_k_pe, g.slots, g.q_abs, g.q_pe, q_scale, q8, g.cache, g.block_table,
                         g.seq_lens, g.out, g.workspace, scale=case.scale, query_start_loc=g.qsl, lse=g.lse,
                         kv_scale=case.kv_scale)
    torch.cuda.synchronize()
    assert mla.decode_status(g.workspace) == 0
    assert np.array_equal(q8.cpu().numpy(), codes)
    assert torch.equal(g.cache.view(torch.uint8), ref_cache.view(torch.uint8))
    rows = sample_rows(case, 300, seed=10)
    qf = oracle.e4m3_to_f64(codes) * np.float64(np.float32(q_scale))
    ref_o, ref_lse, _ = oracle.decode(qf, oracle.prepare_cache(case), case.page_size, oracle.CACHE_E4M3,
                                      case.kv_scale, case.block_table, case.seq_lens, case.query_start_loc,
                                      case.num_heads, case.scale, rows=rows)
    out = g.out.float().reshape(-1, LKV).cpu().numpy().astype(np.float64)[rows]
    lse = g.lse.reshape(-1).cpu().numpy().astype(np.float64)[rows]
    fin = np.isfinite(ref_lse)
    assert np.array_equal(np.isfinite(lse), fin)
    assert float(np.max(np.abs(out - ref_o))) <= 6e-2
    assert (float(np.max(np.abs(lse[fin] - ref_lse[fin]))) if fin.any() else 0.0) <= 1e-3
