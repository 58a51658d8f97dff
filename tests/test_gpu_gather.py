"""GPU parity of the paged context gather (gather_and_maybe_dequant_cache):
bit-exact against the oracle for bf16 and e4m3 caches, chunk starts inside
pages, every page size, bad positions and pages flagged and zero-filled."""
import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import mla_latent_kv_15_gb300 as mla
    from gpu_case import GpuCase


def chunks(case, seed, max_chunk):
    """Chunk starts (any offset, page aligned or not) and lengths per request."""
    rng = np.random.Generator(np.random.PCG64(seed))
    lens = case.seq_lens.astype(np.int64)
    starts = np.array([rng.integers(0, max(1, L)) for L in lens], dtype=np.int32)
    n = np.array([min(int(L - s), max_chunk) for L, s in zip(lens, starts)], dtype=np.int64)
    n[0] = 0                                                  # a request with an empty chunk
    cu = np.concatenate([[0], np.cumsum(n)]).astype(np.int32)
    return starts, cu


def run(g, case, cu, starts, extra=3):
    total = int(cu[-1])
    dst = torch.full((total + extra, 576), -7.0, dtype=torch.bfloat16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    mla.gather_cache(g.cache, g.block_table, torch.from_numpy(cu).cuda(), dst,
                     seq_starts=None if starts is None else torch.from_numpy(starts).cuda(),
                     kv_scale=case.kv_scale, status=status)
    torch.cuda.synchronize()
    return dst.view(torch.int16).cpu().numpy().view(np.uint16), int(status.item())


@pytest.mark.parametrize("dtype,page_size", [("bf16", 16), ("bf16", 64), ("bf16", 256), ("fp8", 64), ("fp8", 32)])
def test_gather_bitexact(dtype, page_size):
    case = synth.make_decode_case(num_heads=2, batch=7, ctx=(40, 900), page_size=page_size, cache_dtype=dtype,
                                  seed=70 + page_size, poison=False)
    g = GpuCase(case)
    cache_host = oracle.prepare_cache(case)
    starts, cu = chunks(case, 71, 300)
    got, status = run(g, case, cu, starts)
    want = oracle.gather_cache(cache_host, page_size, oracle.CACHE_BF16 if dtype == "bf16" else oracle.CACHE_E4M3,
                               case.kv_scale, case.block_table, cu, starts, int(cu[-1]))
    assert status == 0
    assert np.array_equal(got[:cu[-1]], want)
    assert np.all(got[cu[-1]:] == np.uint16(0xC0E0))          # bf16 -7.0: rows past the chunk untouched


def test_gather_fp8_into_16_byte_aligned_dst():
    """A destination that is 16- but not 32-byte aligned (the e4m3 path then
    stores 16 bytes at a time)."""
    case = synth.make_decode_case(num_heads=2, batch=4, ctx=(40, 300), page_size=64, cache_dtype="fp8", seed=75,
                                  poison=False)
    g = GpuCase(case)
    starts, cu = chunks(case, 76, 200)
    total = int(cu[-1])
    buf = torch.zeros((total + 1) * 576 + 8, dtype=torch.bfloat16, device="cuda")
    dst = buf[8:8 + total * 576].view(total, 576)               # 16 bytes past a 256-byte boundary
    assert dst.data_ptr() % 32 == 16
    mla.gather_cache(g.cache, g.block_table, torch.from_numpy(cu).cuda(), dst,
                     seq_starts=torch.from_numpy(starts).cuda(), kv_scale=case.kv_scale)
    torch.cuda.synchronize()
    got = dst.view(torch.int16).cpu().numpy().view(np.uint16)
    want = oracle.gather_cache(oracle.prepare_cache(case), 64, oracle.CACHE_E4M3, case.kv_scale, case.block_table,
                               cu, starts, total)
    assert np.array_equal(got, want)


def test_gather_whole_contexts_from_zero():
    """seq_starts = NULL: every request's context from position 0."""
    case = synth.make_decode_case(num_heads=2, batch=5, ctx=(1, 700), page_size=64, seed=73, poison=False)
    g = GpuCase(case)
    cu = np.concatenate([[0], np.cumsum(case.seq_lens.astype(np.int64))]).astype(np.int32)
    got, status = run(g, case, cu, None, extra=0)
    want = oracle.gather_cache(oracle.prepare_cache(case), 64, oracle.CACHE_BF16, 1.0, case.block_table, cu, None,
                               int(cu[-1]))
    assert status == 0 and np.array_equal(got, want)


def test_gather_flags_bad_rows_and_zero_fills():
    case = synth.make_decode_case(num_heads=2, batch=3, ctx=(100, 200), page_size=64, seed=74, poison=False)
    g = GpuCase(case)
    bt = g.block_table.clone()
    bt[1, 0] = case.num_blocks + 3                            # a page id out of range
    g.block_table = bt
    cu = np.array([0, 10, 30, 40], dtype=np.int32)
    starts = np.array([0, 0, case.max_pages * 64 - 5], dtype=np.int32)   # request 2 runs past its table
    got, status = run(g, case, cu, starts, extra=0)
    assert status & mla.DEVERR_BAD_BLOCK and status & mla.DEVERR_BAD_SEQ_LEN
    assert not got[10:30].any()                               # request 1: page 0 is bad
    assert not got[35:40].any()                               # request 2: positions past the table
    cache_host = oracle.prepare_cache(case)
    ok = oracle.gather_cache(cache_host, 64, oracle.CACHE_BF16, 1.0, case.block_table, cu[:2], starts[:1], 10)
    assert np.array_equal(got[:10], ok)


def test_gather_full_dsv3_contexts():
    """The whole DeepSeek-V3-shaped batch (64 requests, 1k-8k contexts,
    ~295k rows), bf16 and e4m3, bit-exact on every row."""
    for name in ("dsv3_n128_b64_ctx1k-8k", "dsv3_n128_b64_ctx1k-8k_fp8"):
        case = synth.workload(name, poison=False)
        g = GpuCase(case)
        cu = np.concatenate([[0], np.cumsum(case.seq_lens.astype(np.int64))]).astype(np.int32)
        got, status = run(g, case, cu, None, extra=0)
        want = oracle.gather_cache(oracle.prepare_cache(case), case.page_size,
                                   oracle.CACHE_BF16 if case.cache_dtype == "bf16" else oracle.CACHE_E4M3,
                                   case.kv_scale, case.block_table, cu, None, int(cu[-1]))
        assert status == 0 and np.array_equal(got, want)
        del g


@pytest.mark.parametrize("rows,width", [(1, 8), (3, 64), (1000, 512), (64 * 128, 576)])
def test_quantize_fp8_bitexact(rows, width):
    """scaled_fp8_quant on the GPU equals the oracle's float32 divide + e4m3
    encoding bit for bit (values past the range saturate)."""
    x = synth.bf16_normal(80 + rows % 97, (rows, width), std=2.0)
    scale = float(np.float32(3.0 / 448.0))
    dev = torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16)
    out = torch.full((rows, width), 0x55, dtype=torch.uint8, device="cuda")
    mla.quantize_fp8(dev, scale, out)
    torch.cuda.synchronize()
    assert np.array_equal(out.cpu().numpy(), oracle.quantize_fp8(x, scale))


def test_quantize_fp8_into_query_rows():
    """q_abs and q_pe quantised straight into the two column ranges of
    [q_abs | q_pe] rows (strided output), the rest of each row untouched."""
    T, N = 7, 16
    qa = synth.bf16_normal(90, (T, N, 512))
    qp = synth.bf16_normal(91, (T, N, 64))
    scale = float(np.float32(2.5 / 448.0))
    q8 = torch.full((T, N, 576), 0x55, dtype=torch.uint8, device="cuda")
    mla.quantize_fp8(torch.from_numpy(qa.view(np.int16)).cuda().view(torch.bfloat16), scale, q8[..., :512])
    mla.quantize_fp8(torch.from_numpy(qp.view(np.int16)).cuda().view(torch.bfloat16), scale, q8[..., 512:])
    torch.cuda.synchronize()
    want = np.concatenate([oracle.quantize_fp8(qa, scale), oracle.quantize_fp8(qp, scale)], axis=-1)
    assert np.array_equal(q8.cpu().numpy(), want)
