"""GPU parity of the CUDA library (through its C ABI) against the fp64 oracle.

Bars: cache write and paged gather bit-exact; latent output max abs error
<= 2e-2 (bf16 cache) or <= 6e-2 (fp8 cache, against the oracle on dequantised
values); LSE max abs error <= 1e-3.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import mla_latent_kv_15_gb300 as mla
    from gpu_case import GpuCase, compare, sample_rows, bf16_tensor, LKV, DQK, TOL_OUT_BF16, TOL_LSE


# ----------------------------------------------------------------- cache write

@pytest.mark.parametrize("dtype", ["bf16", "fp8"])
@pytest.mark.parametrize("page_size", [16, 64])
def test_cache_write_bitexact(dtype, page_size):
    case = synth.make_decode_case(num_heads=4, batch=37, ctx=(1, 300), sq=[1, 3] * 18 + [2], page_size=page_size,
                                  cache_dtype=dtype, seed=31, poison=False)
    slots = case.slot_mapping.copy()
    slots[5] = -1                                             # a padding token
    g = GpuCase(case, write_new=False)
    before = g.cache.view(torch.uint8).cpu().numpy().copy()
    mla.cache_write(g.new_kv_c, g.new_k_pe, torch.from_numpy(slots).cuda(), g.cache, case.kv_scale)
    torch.cuda.synchronize()
    got = g.cache.view(torch.uint8).cpu().numpy()
    # oracle: the same write applied on the host to the same starting bytes
    if dtype == "bf16":
        ref = before.view(np.uint16).reshape(case.pool.shape).copy()
        oracle.cache_write(case.new_kv_c, case.new_k_pe, slots, ref, page_size, oracle.CACHE_BF16)
        ref = ref.view(np.uint8)
    else:
        ref = before.reshape(case.pool.shape).copy()
        oracle.cache_write(case.new_kv_c, case.new_k_pe, slots, ref, page_size, oracle.CACHE_E4M3, case.kv_scale)
    assert np.array_equal(got.reshape(-1), ref.reshape(-1))


@pytest.mark.parametrize("dtype", ["bf16", "fp8"])
def test_cache_write_skips_slots_past_the_cache(dtype):
    """Slots at or past num_blocks * page_size are skipped like padding ones
    (device data is not checked on the host): the cache equals the oracle's
    write with those tokens marked as padding."""
    case = synth.make_decode_case(num_heads=4, batch=9, ctx=(1, 300), page_size=64, cache_dtype=dtype, seed=33,
                                  poison=False)
    num_slots = case.pool.shape[0] * case.pool.shape[1]
    slots = case.slot_mapping.copy()
    past = [1, 4, 7]
    slots[past] = [num_slots, num_slots + 12345, 1 << 40]
    g = GpuCase(case, write_new=False)
    before = g.cache.view(torch.uint8).cpu().numpy().copy()
    mla.cache_write(g.new_kv_c, g.new_k_pe, torch.from_numpy(slots).cuda(), g.cache, case.kv_scale)
    torch.cuda.synchronize()
    got = g.cache.view(torch.uint8).cpu().numpy()
    pad = slots.copy()
    pad[past] = -1
    if dtype == "bf16":
        ref = before.view(np.uint16).reshape(case.pool.shape).copy()
        oracle.cache_write(case.new_kv_c, case.new_k_pe, pad, ref, case.page_size, oracle.CACHE_BF16)
        ref = ref.view(np.uint8)
    else:
        ref = before.reshape(case.pool.shape).copy()
        oracle.cache_write(case.new_kv_c, case.new_k_pe, pad, ref, case.page_size, oracle.CACHE_E4M3, case.kv_scale)
    assert np.array_equal(got.reshape(-1), ref.reshape(-1))


def test_cache_write_preparation_matches_oracle_fp8():
    """The whole fp8 cache the decode tests read (every referenced row
    quantised on the GPU) is bit-identical to the oracle's."""
    case = synth.make_decode_case(num_heads=2, batch=6, ctx=(50, 400), page_size=64, cache_dtype="fp8", seed=32)
    g = GpuCase(case)
    torch.cuda.synchronize()
    ref = oracle.prepare_cache(case)
    got = g.cache.view(torch.uint8).cpu().numpy()
    used = np.unique(case.referenced_slots // 64)
    assert np.array_equal(got[used], ref[used])


# ----------------------------------------------------------------------- merge

@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_merge_states(dtype):
    rows = 3000
    o_a, lse_a, o_b, lse_b = synth.random_partials(5, rows, 512, neg_inf_frac=0.05)
    ta, tb = torch.from_numpy(o_a).cuda().to(dtype), torch.from_numpy(o_b).cuda().to(dtype)
    la, lb = torch.from_numpy(lse_a).cuda(), torch.from_numpy(lse_b).cuda()
    out = torch.empty_like(ta)
    lo = torch.empty_like(la)
    mla.merge_states(ta, la, tb, lb, out, lo)
    torch.cuda.synchronize()
    ref_o, ref_l = oracle.merge(ta.float().cpu().numpy(), lse_a, tb.float().cpu().numpy(), lse_b)
    got = out.float().cpu().numpy()
    tol = 1e-5 if dtype == torch.float32 else 1e-2
    assert np.max(np.abs(got - ref_o)) <= tol
    fin = np.isfinite(ref_l)
    gl = lo.cpu().numpy()
    assert np.array_equal(np.isfinite(gl), fin)
    assert np.max(np.abs(gl[fin] - ref_l[fin])) <= 1e-5
    # in place: out aliases o_a
    mla.merge_states(ta, la, tb, lb, ta, None)
    torch.cuda.synchronize()
    assert torch.equal(ta, out)


# ---------------------------------------------------------------------- decode

def test_decode_tiny_config_all_rows():
    """N=16, ctx 256, page 64, 4 of 8 pages permuted: every row vs the oracle."""
    case = synth.workload("tiny_n16_ctx256")
    g = GpuCase(case)
    g.decode()
    compare(case, g)
    assert mla.decode_status(g.workspace) == 0


@pytest.mark.parametrize("num_heads,sq,page_size,num_splits", [
    (16, 1, 64, 0), (16, 1, 64, 3), (128, 1, 64, 0), (128, 1, 64, 1), (128, 1, 16, 2),
    (128, 4, 64, 0), (16, 4, 32, 0), (16, [4, 1, 2, 1, 3, 1], 64, 0), (128, [4, 1, 1, 4, 2, 1], 64, 2),
    (20, 2, 64, 0), (1, 1, 128, 0), (256, 1, 256, 0), (64, 3, 64, 5),
])
def test_decode_small_cases(num_heads, sq, page_size, num_splits):
    """Several tiles with a ragged tail; splits, multi-token causal groups,
    head counts that do not divide 128, every page size."""
    batch = 6
    case = synth.make_decode_case(num_heads=num_heads, batch=batch, ctx=(60, 700), sq=sq, page_size=page_size,
                                  seed=100 + num_heads + page_size + num_splits)
    g = GpuCase(case, num_splits_max=num_splits)
    g.decode(num_splits)
    compare(case, g)
    assert mla.decode_status(g.workspace) == 0


@pytest.mark.parametrize("num_heads,sq,page_size,num_splits", [
    (128, 1, 64, 0), (16, 1, 64, 3), (128, 4, 64, 0), (128, [4, 1, 1, 2, 1, 3], 16, 2),
])
def test_decode_fp8_cache(num_heads, sq, page_size, num_splits):
    """e4m3 cache with a per-tensor scale, dequantised inside the decode; against
    the oracle run on the dequantised values."""
    case = synth.make_decode_case(num_heads=num_heads, batch=6, ctx=(60, 700), sq=sq, page_size=page_size,
                                  cache_dtype="fp8", seed=200 + num_heads + page_size + num_splits)
    g = GpuCase(case, num_splits_max=num_splits)
    g.decode(num_splits)
    compare(case, g)
    assert mla.decode_status(g.workspace) == 0


@pytest.mark.parametrize("num_heads,sq,num_splits", [
    (16, [1] * 8, 0), (32, [2, 0, 1, 1, 2, 0, 1, 1], 0), (24, [3, 0, 0, 1, 1, 1, 1, 1], 2), (20, [1] * 8, 3),
])
def test_decode_small_head_count(num_heads, sq, num_splits):
    """Small head counts with as many query tokens as requests run the
    small-rows kernel variant (32-row groups); requests with several tokens
    span several groups there."""
    batch = len(sq)
    assert sum(sq) == batch
    case = synth.make_decode_case(num_heads=num_heads, batch=batch, ctx=(60, 900), sq=sq, page_size=64,
                                  seed=300 + num_heads + num_splits)
    g = GpuCase(case, num_splits_max=num_splits)
    g.decode(num_splits)
    compare(case, g)
    assert mla.decode_status(g.workspace) == 0


@pytest.mark.parametrize("num_heads,sq", [(1024, 1), (1000, [2, 1]), (384, 3)])
def test_decode_large_head_counts(num_heads, sq):
    """Head counts up to the 1024 the ABI accepts: a token spans several
    128-row groups, the last one partial when N is not a multiple of 128."""
    case = synth.make_decode_case(num_heads=num_heads, batch=2, ctx=(100, 600), sq=sq, page_size=64,
                                  seed=400 + num_heads)
    g = GpuCase(case)
    g.decode()
    compare(case, g, rows=sample_rows(case, 600, seed=num_heads))
    assert mla.decode_status(g.workspace) == 0


def test_decode_negative_scale():
    """A negative softmax scale (the kernel negates q and works with |scale|)."""
    case = synth.make_decode_case(num_heads=16, batch=4, ctx=(60, 500), page_size=64, seed=45)
    case.scale = -case.scale
    g = GpuCase(case)
    g.decode()
    compare(case, g)
    assert mla.decode_status(g.workspace) == 0


def test_decode_edge_lengths():
    """seq_len 0 (padding request), Sq > seq_len, one-token contexts, exact
    multiples of the tile, lengths one past a tile."""
    lens = [0, 1, 2, 63, 64, 65, 128, 129, 1, 3]
    sq = [1, 1, 4, 1, 2, 1, 1, 3, 1, 4]
    case = synth.make_decode_case(num_heads=16, batch=len(lens), ctx=(1, 1), sq=sq, seq_lens=lens,
                                  page_size=64, seed=41)
    g = GpuCase(case)
    g.decode()
    compare(case, g)


def test_one_token_context_returns_kv_c_bitexact():
    """seq_len 1 on every physical page: out == kv_c of the page's first row
    bit for bit (p = 1, l = 1), which also pins the paged gather."""
    nb = 16
    case = synth.make_decode_case(num_heads=32, batch=nb, ctx=(1, 1), page_size=64, num_blocks=nb, seed=42,
                                  poison=False)
    case.block_table[:, 0] = np.arange(nb, dtype=np.int32)[::-1]
    case.slot_mapping[:] = -1                                  # keep the drawn rows
    g = GpuCase(case)
    g.decode()
    got = g.out.view(torch.int16).cpu().numpy().view(np.uint16)       # [nb, 32, 512]
    want = case.pool[case.block_table[:, 0], 0, :LKV]                 # [nb, 512]
    assert np.array_equal(got, np.broadcast_to(want[:, None, :], got.shape))


def test_split_counts_agree():
    """Automatic and forced splits (1, 2, 7 pieces) give the same result within
    the rounding of the stored partials and of the merge."""
    case = synth.make_decode_case(num_heads=128, batch=5, ctx=(500, 2000), page_size=64, seed=43)
    g = GpuCase(case, num_splits_max=7)
    res = []
    for k in (0, 1, 2, 7):
        o, l = g.decode(k)
        res.append((o.float().clone(), l.clone()))
        compare(case, g)
    for o, l in res[1:]:
        assert torch.max(torch.abs(o - res[0][0])).item() <= 1.6e-2
        assert torch.max(torch.abs(l - res[0][1])).item() <= 1e-4


def _scale_bf16(bits: np.ndarray, k: int) -> np.ndarray:
    """bf16 bits of x * 2^k (exact: asserted)."""
    f = (bits.astype(np.uint32) << 16).view(np.float32) * np.float32(2.0 ** k)
    out = (f.view(np.uint32) >> 16).astype(np.uint16)
    assert np.array_equal((out.astype(np.uint32) << 16).view(np.float32), f)
    return out


@pytest.mark.parametrize("num_heads", [128, 16])
@pytest.mark.parametrize("k", [20, -30])
def test_split_partials_at_any_magnitude(num_heads, k):
    """Split partials keep their precision whatever the values' magnitude
    (they are stored as fp16 codes with a power-of-two scale per 32-dim
    chunk; plain fp16 would overflow at 2^20 and lose everything at 2^-30).
    kv_c is scaled by 2^k and q_abs by 2^-k: every score, hence the LSE, is
    unchanged and the output scales by exactly 2^k, so 2^-k times the output
    meets the bar against the oracle of the unscaled case."""
    case = synth.make_decode_case(num_heads=num_heads, batch=5, ctx=(500, 2000), page_size=64, seed=45,
                                  poison=False)
    big = dataclasses.replace(case, pool=case.pool.copy(), new_kv_c=_scale_bf16(case.new_kv_c, k),
                              q_abs=_scale_bf16(case.q_abs, -k))
    big.pool[..., :LKV] = _scale_bf16(case.pool[..., :LKV], k)
    g = GpuCase(big, num_splits_max=7)
    ref_o, ref_lse, _ = oracle.decode_case(case, oracle.prepare_cache(case))
    for splits in (0, 7):
        g.decode(splits)
        out = g.out.float().reshape(-1, LKV).cpu().numpy().astype(np.float64) * 2.0 ** -k
        lse = g.lse.reshape(-1).cpu().numpy().astype(np.float64)
        assert np.all(np.isfinite(out)) and np.all(np.isfinite(lse))
        assert np.max(np.abs(out - ref_o)) <= TOL_OUT_BF16
        assert np.max(np.abs(lse - ref_lse)) <= TOL_LSE
        assert mla.decode_status(g.workspace) == 0


def test_block_id_out_of_range_flags_and_does_not_fault():
    case = synth.make_decode_case(num_heads=16, batch=2, ctx=(100, 200), page_size=64, seed=44, poison=False)
    g = GpuCase(case)
    bt = g.block_table.clone()
    bt[0, 0] = case.num_blocks + 5
    g.block_table = bt
    g.decode()
    assert mla.decode_status(g.workspace) & mla.DEVERR_BAD_BLOCK


def test_seq_len_beyond_the_block_table_flags_and_clamps():
    """A request whose seq_len exceeds max_pages * page_size: the scheduler
    flags DEVERR_BAD_SEQ_LEN and clamps the request to the keys its block
    table reaches (its unused entries are -1, so they are flagged too and read
    as zeros), and the other requests keep the oracle's result."""
    case = synth.make_decode_case(num_heads=32, batch=3, ctx=(300, 900), page_size=64, seed=45, poison=False)
    g = GpuCase(case)
    sl = g.seq_lens.clone()
    sl[1] = case.block_table.shape[1] * case.page_size + 100
    g.seq_lens = sl
    g.decode()
    assert mla.decode_status(g.workspace) & mla.DEVERR_BAD_SEQ_LEN
    N, qsl = case.num_heads, case.query_start_loc
    rows = np.array([t * N + h for b in (0, 2) for t in range(qsl[b], qsl[b + 1]) for h in range(N)])
    compare(case, g, rows=rows)


# --------------------------------------------------------- full-size workloads

FULL = [("dsv3_n128_b64_ctx1k-8k", (0,)), ("dsv3_n128_b64_ctx1k-8k_fp8", (0,)), ("n16_b128_ctx8k-32k", (0, 4, 16)),
        ("mtp_n128_sq4_b32_ctx2k-16k", (0,)), ("mtp_mixed_n128_b32_ctx2k-16k", (0,))]


@pytest.mark.parametrize("name,splits", FULL)
def test_full_size_sampled_rows(name, splits):
    """Serving-shaped batches at full size in the launch configuration the
    benchmark uses (automatic split; forced 4 and 16 splits for the long
    contexts); sampled rows against the oracle."""
    case = synth.workload(name)
    g = GpuCase(case, num_splits_max=max(splits))
    cache_host = oracle.prepare_cache(case)
    rows = sample_rows(case, 300, seed=7)
    for k in splits:
        g.out.fill_(float("nan"))
        g.decode(k)
        compare(case, g, rows=rows, cache_host=cache_host)
        assert mla.decode_status(g.workspace) == 0
