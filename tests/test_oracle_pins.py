"""Pins of the fp64 oracle against facts the MLA pages and mathematics fix.

Each check is independent of the oracle's own code path: the compute-friendly
MHA path (a different formula the pages state is equivalent), closed forms,
library routines (scipy logsumexp, torch's float8/bf16 casts), the OCP E4M3
definition, and brute force on tiny inputs with an independent gather.
"""
import math

import numpy as np
import pytest
import torch
from scipy.special import logsumexp

import oracle
import synth
from oracle import expanded

LKV, DQK = 512, 576


def _rows_in_order(case, b):
    """Latent rows of request b in position order (test-side gather)."""
    L = int(case.seq_lens[b])
    pos = np.arange(L)
    pages = case.block_table[b, pos // case.page_size]
    return case.pool[pages, pos % case.page_size]          # [L, 576] bf16 bits


# ------------------------------------------------------------ two-path identity

def test_projections_select_with_one_hot_weights():
    """A one-hot W_UV / W_UK picks one input column per output column, and
    zero columns give zeros: pins which operand axis each einsum contracts."""
    rng = np.random.Generator(np.random.PCG64(11))
    T, N, L, P, V = 3, 4, 512, 128, 64
    o_lat = rng.standard_normal((T, N, L))
    pick = rng.permutation(L)[:V]
    w_uv = np.zeros((L, N, V))
    for n in range(N):
        w_uv[pick, n, np.arange(V)] = 1.0
    w_uv[:, 2, :] = 0.0
    o = expanded.up_project(o_lat, w_uv)
    want = o_lat[:, :, pick].copy()
    want[:, 2, :] = 0.0
    assert np.array_equal(o, want)
    q_nope = rng.standard_normal((T, N, P))
    w_uk = np.zeros((L, N, P))
    src = rng.integers(0, P, size=L)
    for n in range(N):
        w_uk[np.arange(L), n, src] = n + 1.0
    ql = expanded.absorb_query(q_nope, w_uk)
    assert np.array_equal(ql, q_nope[:, :, src] * (np.arange(N) + 1.0)[None, :, None])


@pytest.mark.parametrize("sq", [1, 4])
def test_two_path_identity(sq):
    """Absorbed MQA + W_UV up-projection == expanded MHA (common.py docstring,
    both approaches), fp64 difference <= 1e-10; pins scores (both terms),
    the scale 1/sqrt(P+R), V = kv_c, the block-table gather and the causal rule."""
    N, P, V = 16, 128, 128
    case = synth.make_decode_case(num_heads=N, batch=1, ctx=(256, 256), sq=sq, page_size=64,
                                  num_blocks=8, seed=1)
    rows = oracle.bf16_to_f64(_rows_in_order(case, 0))      # [256, 576]
    kv_c, k_pe = rows[:, :LKV], rows[:, LKV:]
    w_uk, w_uv = synth.expanded_weights(1, N, p=P, v=V)
    rng = np.random.Generator(np.random.PCG64(7))
    q_nope = rng.standard_normal((sq, N, P)) * 0.5
    q_pe = oracle.bf16_to_f64(case.q_pe)
    scale = 1.0 / math.sqrt(P + 64)
    assert case.scale == scale

    ql_nope = expanded.absorb_query(q_nope, w_uk)           # [Sq, N, 512]
    q = np.concatenate([ql_nope, q_pe], axis=-1)
    o_lat, lse_abs, _ = oracle.decode(q, case.pool, 64, oracle.CACHE_BF16, 1.0, case.block_table,
                                      case.seq_lens, case.query_start_loc, N, scale)
    o_abs = expanded.up_project(o_lat.reshape(sq, N, LKV), w_uv)

    # page statement: verify token t sees seq_len - (Sq - 1) + t entries
    visible = [int(case.seq_lens[0]) - (sq - 1) + t for t in range(sq)]
    o_exp, lse_exp = expanded.expanded_mha(q_nope, q_pe, kv_c, k_pe, w_uk, w_uv, scale, visible)
    assert np.max(np.abs(o_abs - o_exp)) <= 1e-10
    assert np.max(np.abs(lse_abs.reshape(sq, N) - lse_exp)) <= 1e-10


def test_two_path_identity_fails_with_sdpa_default_scale():
    """The identity is not vacuous: with the SDPA default 1/sqrt(576) on the
    absorbed side it breaks."""
    N, P, V = 16, 128, 128
    case = synth.make_decode_case(num_heads=N, batch=1, ctx=(64, 64), page_size=64, num_blocks=2, seed=3)
    rows = oracle.bf16_to_f64(_rows_in_order(case, 0))
    w_uk, w_uv = synth.expanded_weights(3, N, p=P, v=V)
    q_nope = np.random.Generator(np.random.PCG64(8)).standard_normal((1, N, P)) * 0.5
    q_pe = oracle.bf16_to_f64(case.q_pe)
    q = np.concatenate([expanded.absorb_query(q_nope, w_uk), q_pe], axis=-1)
    o_lat, _, _ = oracle.decode(q, case.pool, 64, oracle.CACHE_BF16, 1.0, case.block_table,
                                case.seq_lens, case.query_start_loc, N, 1.0 / math.sqrt(576))
    o_abs = expanded.up_project(o_lat.reshape(1, N, LKV), w_uv)
    o_exp, _ = expanded.expanded_mha(q_nope, q_pe, rows[:, :LKV], rows[:, LKV:], w_uk, w_uv,
                                     1.0 / math.sqrt(192), [64])
    assert np.max(np.abs(o_abs - o_exp)) > 1e-3


# ------------------------------------------------------------------ invariants

def test_softmax_rows_sum_to_one():
    """A value column that is 1 for every key returns sum_j p_j = 1 (<= 1e-12)."""
    case = synth.make_decode_case(num_heads=16, batch=3, ctx=(100, 300), page_size=64, seed=11)
    pool = case.pool.copy()
    pool[..., 5] = np.uint16(0x3F80)                       # bf16 1.0
    pool[..., 300] = np.uint16(0xC040)                     # bf16 -3.0
    out, _, _ = oracle.decode_case(case, pool)
    assert np.max(np.abs(out[:, 5] - 1.0)) <= 1e-12
    assert np.max(np.abs(out[:, 300] + 3.0)) <= 1e-12


def test_one_token_context_returns_kv_c_exactly():
    """seq_len 1: p = 1, l = 1, so o is kv_c of position 0 bit for bit, and the
    LSE is the single score; checked for every physical page of the pool."""
    nb = 8
    case = synth.make_decode_case(num_heads=16, batch=nb, ctx=(1, 1), page_size=64, num_blocks=nb, seed=12)
    case.block_table[:, 0] = np.arange(nb, dtype=np.int32)     # request b reads page b
    pool = case.pool.copy()
    pool[:, 0] = synth.to_bf16_bits(np.random.Generator(np.random.PCG64(5)).standard_normal((nb, DQK)).astype(np.float32))
    out, lse, _ = oracle.decode_case(case, pool)
    rows = oracle.bf16_to_f64(pool[:, 0])                      # [nb, 576]
    q = np.concatenate([oracle.bf16_to_f64(case.q_abs), oracle.bf16_to_f64(case.q_pe)], -1)
    for b in range(nb):
        for h in range(16):
            r = b * 16 + h
            assert np.array_equal(out[r], rows[b, :LKV])
            assert abs(lse[r] - case.scale * float(q[b, h] @ rows[b])) <= 1e-12


def test_split_then_merge_equals_unsplit():
    """Attention over [0,k) merged with [k,L) equals attention over [0,L)."""
    case = synth.make_decode_case(num_heads=16, batch=4, ctx=(130, 400), page_size=64, seed=13)
    full, lse_full, _ = oracle.decode_case(case, case.pool)
    for k in (1, 64, 100, 129):
        a, la, _ = oracle.decode_case(case, case.pool, key_end=k)
        b, lb, _ = oracle.decode_case(case, case.pool, key_begin=k)
        m, lm = oracle.merge(a, la, b, lb)
        assert np.max(np.abs(m - full)) <= 1e-12
        assert np.max(np.abs(lm - lse_full)) <= 1e-12
    # three pieces, merged left to right
    a, la, _ = oracle.decode_case(case, case.pool, key_end=64)
    b, lb, _ = oracle.decode_case(case, case.pool, key_begin=64, key_end=128)
    c, lc, _ = oracle.decode_case(case, case.pool, key_begin=128)
    m, lm = oracle.merge(*oracle.merge(a, la, b, lb), c, lc)
    assert np.max(np.abs(m - full)) <= 1e-12 and np.max(np.abs(lm - lse_full)) <= 1e-12


def test_brute_force_tiny_against_scipy():
    """Tiny contexts: scores from an independent gather and numpy dot, softmax
    and LSE from scipy; page size 4 with a permuted table."""
    case = synth.make_decode_case(num_heads=3, batch=4, ctx=(1, 9), sq=[1, 2, 1, 3], page_size=4,
                                  num_blocks=16, seed=14)
    out, lse, _ = oracle.decode_case(case, case.pool)
    q = np.concatenate([oracle.bf16_to_f64(case.q_abs), oracle.bf16_to_f64(case.q_pe)], -1)
    qsl = case.query_start_loc
    for b in range(case.batch):
        rows = oracle.bf16_to_f64(_rows_in_order(case, b))
        sq = qsl[b + 1] - qsl[b]
        for tl in range(sq):
            t = qsl[b] + tl
            L = case.seq_lens[b] - sq + 1 + tl
            for h in range(3):
                s = case.scale * (rows[:L] @ q[t, h])
                w = np.exp(s - logsumexp(s))
                r = t * 3 + h
                assert abs(lse[r] - logsumexp(s)) <= 1e-12
                assert np.max(np.abs(out[r] - w @ rows[:L, :LKV])) <= 1e-12


def test_brute_force_tiny_e4m3_cache_against_scipy():
    """The e4m3 branch of the decode: keys and values are the stored codes'
    OCP values times kv_scale.  Tiny contexts through a permuted table of
    4-row pages, against numpy dots and scipy's logsumexp on rows decoded
    independently of the decode (an unscaled value, a scale applied to the
    keys only or twice, or a wrong gather fails)."""
    case = synth.make_decode_case(num_heads=3, batch=4, ctx=(1, 9), sq=[1, 2, 1, 3], page_size=4,
                                  num_blocks=16, seed=24, cache_dtype="fp8", poison=False)
    cache = oracle.prepare_cache(case, with_new_rows=False)
    out, lse, _ = oracle.decode_case(case, cache)
    kvs = float(np.float32(case.kv_scale))
    q = np.concatenate([oracle.bf16_to_f64(case.q_abs), oracle.bf16_to_f64(case.q_pe)], -1)
    qsl = case.query_start_loc
    for b in range(case.batch):
        pos = np.arange(int(case.seq_lens[b]))
        codes = cache[case.block_table[b, pos // case.page_size], pos % case.page_size]
        rows = oracle.e4m3_to_f64(codes) * kvs
        sq = qsl[b + 1] - qsl[b]
        for tl in range(sq):
            t = qsl[b] + tl
            L = case.seq_lens[b] - sq + 1 + tl
            for h in range(3):
                s = case.scale * (rows[:L] @ q[t, h])
                w = np.exp(s - logsumexp(s))
                r = t * 3 + h
                assert abs(lse[r] - logsumexp(s)) <= 1e-12
                assert np.max(np.abs(out[r] - w @ rows[:L, :LKV])) <= 1e-12


def test_causal_rule_closed_form():
    """q = 0 makes every visible score 0, so o is the mean of the visible rows
    and lse = ln L.  With kv_c[:, 0] = position, o[0] = (L - 1) / 2, where the
    page gives L = seq_len - (Sq - 1) + t for verify token t."""
    sq, seq_len = 4, 70
    case = synth.make_decode_case(num_heads=2, batch=1, ctx=(seq_len, seq_len), sq=sq, page_size=64,
                                  num_blocks=4, seed=15)
    pool = case.pool.copy()
    for j in range(seq_len):
        pool[case.block_table[0, j // 64], j % 64, 0] = synth.to_bf16_bits(np.float32([j]))[0]
    case.q_abs[:] = 0
    case.q_pe[:] = 0
    out, lse, _ = oracle.decode_case(case, pool)
    for t in range(sq):
        L = seq_len - (sq - 1) + t
        for h in range(2):
            assert out[t * 2 + h, 0] == (L - 1) / 2
            assert abs(lse[t * 2 + h] - math.log(L)) <= 1e-12


def test_gather_and_scale_geometric_closed_form():
    """q_pe = c*e_0 and k_pe[:, 0] = j/64 give s_j = scale*c*j/64, so weights
    are geometric in the position j; with kv_c[:, 0] = j the output is the
    geometric mean position.  Pins the paged gather order and the scale."""
    L, c = 200, 8.0
    case = synth.make_decode_case(num_heads=1, batch=1, ctx=(L, L), page_size=16, num_blocks=20, seed=16)
    pool = case.pool.copy()
    for j in range(L):
        page, off = case.block_table[0, j // 16], j % 16
        pool[page, off, 0] = synth.to_bf16_bits(np.float32([j]))[0]
        pool[page, off, LKV] = synth.to_bf16_bits(np.float32([j / 64]))[0]
        pool[page, off, 1:LKV] = 0
        pool[page, off, LKV + 1:] = 0
    case.q_abs[:] = 0
    case.q_pe[:] = 0
    case.q_pe[0, 0, 0] = synth.to_bf16_bits(np.float32([c]))[0]
    out, lse, _ = oracle.decode_case(case, pool)
    r = math.exp(case.scale * c / 64)
    w = np.array([r ** j for j in range(L)])
    assert abs(out[0, 0] - (np.arange(L) @ w) / w.sum()) <= 1e-9
    assert abs(lse[0] - math.log(w.sum())) <= 1e-9


def test_head_padding_invariance():
    """Extra (padding) heads cannot change heads [0:N] (rocm_aiter_mla module notes)."""
    case = synth.make_decode_case(num_heads=16, batch=2, ctx=(50, 150), page_size=64, seed=17)
    out, lse, _ = oracle.decode_case(case, case.pool)
    pad = 4
    rng = np.random.Generator(np.random.PCG64(9))
    q = np.concatenate([oracle.bf16_to_f64(case.q_abs), oracle.bf16_to_f64(case.q_pe)], -1)
    qp = np.concatenate([q, rng.standard_normal((q.shape[0], pad, DQK))], axis=1)
    out_p, lse_p, _ = oracle.decode(qp, case.pool, 64, oracle.CACHE_BF16, 1.0, case.block_table,
                                    case.seq_lens, case.query_start_loc, 16 + pad, case.scale)
    out_p = out_p.reshape(-1, 16 + pad, LKV)[:, :16].reshape(-1, LKV)
    lse_p = lse_p.reshape(-1, 16 + pad)[:, :16].ravel()
    assert np.array_equal(out_p, out) and np.array_equal(lse_p, lse)


def test_empty_rows_zero_output_neg_inf_lse():
    """seq_len 0 (padding request) and verify tokens with no visible key give
    o = 0, lse = -inf (zero-fill of unwritten lanes, AiterMLAImpl.forward_mqa)."""
    case = synth.make_decode_case(num_heads=4, batch=3, ctx=(1, 1), sq=[1, 3, 1],
                                  seq_lens=[0, 2, 5], page_size=64, num_blocks=4, seed=18, poison=False)
    out, lse, _ = oracle.decode_case(case, case.pool)
    out = out.reshape(-1, 4, LKV)
    lse = lse.reshape(-1, 4)
    assert np.all(out[0] == 0) and np.all(np.isneginf(lse[0]))           # seq_len 0
    assert np.all(out[1] == 0) and np.all(np.isneginf(lse[1]))           # L = 2-2+0 = 0
    assert np.all(np.isfinite(lse[2])) and np.all(np.isfinite(lse[3]))   # L = 1, 2
    assert np.all(np.isfinite(lse[4]))


# ----------------------------------------------------------------------- merge

def test_merge_special_cases():
    o_a, lse_a, o_b, lse_b = synth.random_partials(1, 64)
    o_a, o_b = o_a.astype(np.float64), o_b.astype(np.float64)
    lse_a, lse_b = lse_a.astype(np.float64), lse_b.astype(np.float64)
    # one side empty: the other side is returned unchanged
    m, l = oracle.merge(o_a, lse_a, o_b, np.full(64, -np.inf))
    assert np.array_equal(m, o_a) and np.array_equal(l, lse_a)
    # equal LSE: plain average, lse + ln 2
    m, l = oracle.merge(o_a, lse_a, o_b, lse_a)
    assert np.max(np.abs(m - 0.5 * (o_a + o_b))) <= 1e-15
    assert np.max(np.abs(l - (lse_a + math.log(2)))) <= 1e-14
    # both empty
    m, l = oracle.merge(o_a, np.full(64, -np.inf), o_b, np.full(64, -np.inf))
    assert np.all(m == 0) and np.all(np.isneginf(l))
    # general: lse is logsumexp of the pair (scipy)
    _, l = oracle.merge(o_a, lse_a, o_b, lse_b)
    assert np.max(np.abs(l - logsumexp(np.stack([lse_a, lse_b]), axis=0))) <= 1e-13


# ---------------------------------------------------------------- number formats

def test_bf16_decode_matches_torch_all_patterns():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = oracle.bf16_to_f64(bits)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])


def test_e4m3_golden_values():
    """Values fixed by the OCP E4M3 definition (tests/golden/e4m3_values.txt)."""
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "e4m3_values.txt")
    for line in open(path):
        line = line.split("#")[0].strip()
        if not line:
            continue
        code, val = line.split()
        code, val = int(code, 16), float(val)
        got = oracle.e4m3_to_f64(np.array([code], np.uint8))[0]
        assert got == val and math.copysign(1, got) == math.copysign(1, val), (hex(code), got, val)
        assert oracle.f32_to_e4m3(np.array([val], np.float32))[0] == code


def test_e4m3_exhaustive_round_trip_and_torch():
    codes = np.arange(256, dtype=np.uint8)
    vals = oracle.e4m3_to_f64(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert list(np.nonzero(nan)[0]) == [0x7F, 0xFF]
    assert np.array_equal(np.isnan(vals), nan) and np.array_equal(vals[~nan], ref[~nan])
    back = oracle.f32_to_e4m3(vals[~nan].astype(np.float32))
    assert np.array_equal(back, codes[~nan])


def test_e4m3_encoder_matches_torch_cast_on_grid():
    """RNE incl. ties, subnormals and signed zero, against torch's cast, for every
    bf16 value in [-448, 448] and random float32 values."""
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    x = synth.bf16_bits_to_f32(bits)
    x = x[np.isfinite(x) & (np.abs(x) <= 448)]
    rng = np.random.Generator(np.random.PCG64(3))
    x = np.concatenate([x, (rng.standard_normal(200000) * 50).astype(np.float32),
                        (rng.standard_normal(50000) * 0.01).astype(np.float32)])
    x = x[np.abs(x) <= 448]
    ours = oracle.f32_to_e4m3(x)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)


def test_e4m3_saturates():
    x = np.array([449.0, 463.9, 464.0, 1e6, np.inf, -500.0, -np.inf], np.float32)
    assert list(oracle.f32_to_e4m3(x)) == [0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0xFE]
    assert oracle.f32_to_e4m3(np.array([np.nan], np.float32))[0] & 0x7F == 0x7F


# ----------------------------------------------------------------- cache write

def test_cache_write_bf16_places_rows():
    case = synth.make_decode_case(num_heads=2, batch=3, ctx=(10, 130), page_size=16, seed=19, poison=False)
    cache = case.pool.copy()
    slots = case.slot_mapping.copy()
    slots[1] = -1                                              # padding token
    oracle.cache_write(case.new_kv_c, case.new_k_pe, slots, cache, 16, oracle.CACHE_BF16)
    flat, before = cache.reshape(-1, DQK), case.pool.reshape(-1, DQK)
    for i, s in enumerate(slots):
        if s < 0:
            continue
        assert np.array_equal(flat[s, :LKV], case.new_kv_c[i])
        assert np.array_equal(flat[s, LKV:], case.new_k_pe[i])
    untouched = np.setdiff1d(np.arange(flat.shape[0]), slots[slots >= 0])
    assert np.array_equal(flat[untouched], before[untouched])


def test_cache_write_fp8_is_rne_of_x_over_scale():
    """fp8 code = e4m3(fp32(x) / fp32(kv_scale)); checked against torch's
    float32 divide and float8 cast, and dequant x*scale within half an ulp."""
    case = synth.make_decode_case(num_heads=2, batch=4, ctx=(40, 200), page_size=64, seed=20,
                                  cache_dtype="fp8", poison=False)
    cache = np.zeros(case.pool.shape, np.uint8)
    oracle.cache_write(case.new_kv_c, case.new_k_pe, case.slot_mapping, cache, 64, oracle.CACHE_E4M3,
                       case.kv_scale)
    x = np.concatenate([synth.bf16_bits_to_f32(case.new_kv_c), synth.bf16_bits_to_f32(case.new_k_pe)], 1)
    ref = (torch.from_numpy(x) / torch.tensor(case.kv_scale, dtype=torch.float32)).to(torch.float8_e4m3fn)
    got = cache.reshape(-1, DQK)[case.slot_mapping]
    assert np.array_equal(got, ref.view(torch.uint8).numpy())
    deq = oracle.e4m3_to_f64(got) * case.kv_scale
    assert np.max(np.abs(deq - x)) <= case.kv_scale * 16      # half ulp at the top binade (32/2)


# -------------------------------------------------------------- context gather

def _golden_e4m3():
    """code -> value from the OCP E4M3 table of tests/golden/e4m3_values.txt."""
    import os
    vals = {}
    for line in open(os.path.join(os.path.dirname(__file__), "golden", "e4m3_values.txt")):
        line = line.split("#")[0].strip()
        if not line:
            continue
        code, val = line.split()[:2]
        vals[int(code, 0)] = float(val)
    return vals


def test_gather_bf16_is_the_position_ordered_rows():
    """Gathering whole contexts from position 0 returns each request's rows in
    position order (the test-side gather), bit for bit; a chunk that starts
    mid-page returns the same rows shifted."""
    case = synth.make_decode_case(num_heads=2, batch=5, ctx=(30, 300), page_size=16, seed=51, poison=False)
    lens = case.seq_lens.astype(np.int64)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    got = oracle.gather_cache(case.pool, 16, oracle.CACHE_BF16, 1.0, case.block_table, cu, None, int(cu[-1]) + 3)
    for b in range(case.batch):
        assert np.array_equal(got[cu[b]:cu[b + 1]], _rows_in_order(case, b))
    assert not got[cu[-1]:].any()
    starts = np.array([7, 0, 21, 3, 16], dtype=np.int32)
    n = np.minimum(lens - starts, 40)
    cu2 = np.concatenate([[0], np.cumsum(n)]).astype(np.int32)
    got2 = oracle.gather_cache(case.pool, 16, oracle.CACHE_BF16, 1.0, case.block_table, cu2, starts, int(cu2[-1]))
    for b in range(case.batch):
        assert np.array_equal(got2[cu2[b]:cu2[b + 1]], _rows_in_order(case, b)[starts[b]:starts[b] + n[b]])


def test_gather_e4m3_dequantises_to_table_values():
    """With a power-of-two scale the dequantised value code * scale is exact in
    bf16: every gathered element equals the OCP table value times the scale
    (NaN codes stay NaN).  Codes are drawn from the golden table's entries."""
    table = _golden_e4m3()
    nb, ps = 4, 16
    rng = np.random.Generator(np.random.PCG64(52))
    codes = np.array(sorted(table) + [0x7F, 0xFF], dtype=np.uint8)     # table values and the two NaNs
    cache = rng.choice(codes, size=(nb, ps, DQK))
    bt = np.array([[2, 0], [3, 1]], dtype=np.int32)
    cu = np.array([0, 20, 45], dtype=np.int32)
    got = oracle.gather_cache(cache, ps, oracle.CACHE_E4M3, 0.125, bt, cu, np.array([5, 0], np.int32), 45)
    vals = oracle.bf16_to_f64(got)
    for b, (lo, hi) in enumerate([(0, 20), (20, 45)]):
        start = 5 if b == 0 else 0
        for j in range(hi - lo):
            pos = start + j
            codes = cache[bt[b, pos // ps], pos % ps]
            want = np.array([table[c] * 0.125 if c in table else np.nan for c in codes])
            row = vals[lo + j]
            assert np.array_equal(np.isnan(row), np.isnan(want))
            assert np.array_equal(row[~np.isnan(want)], want[~np.isnan(want)])


def test_gather_e4m3_rounding_matches_torch():
    """With an arbitrary scale the float32 product is rounded to bf16: the
    oracle agrees bit for bit with torch's float8 -> float32 multiply ->
    bfloat16 cast on every finite code."""
    nb, ps = 2, 32
    finite = np.array([c for c in range(256) if c & 0x7F != 0x7F], dtype=np.uint8)
    rng = np.random.Generator(np.random.PCG64(53))
    cache = rng.choice(finite, size=(nb, ps, DQK))
    scale = np.float32(0.0137)
    bt = np.array([[1, 0]], dtype=np.int32)
    got = oracle.gather_cache(cache, ps, oracle.CACHE_E4M3, float(scale), bt, np.array([0, 64], np.int32), None, 64)
    rows = np.concatenate([cache[1], cache[0]])
    t = torch.from_numpy(rows).view(torch.float8_e4m3fn).float() * torch.tensor(scale)
    want = t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, want)


def test_query_quantisation_matches_torch_casts():
    """scaled_fp8_quant of a bf16 query: float32 divide by the scale, then the
    e4m3 cast; bit-identical to torch's float32 division and float8_e4m3fn
    cast (with saturation) on random queries, including values past the
    range."""
    rng = np.random.Generator(np.random.PCG64(54))
    x = rng.standard_normal(20000, dtype=np.float32) * np.float32(3.0)
    bits = synth.to_bf16_bits(x)
    scale = float(np.float32(0.0071))
    got = oracle.quantize_fp8(bits, scale)
    t = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).float() / torch.tensor(np.float32(scale))
    want = t.clamp(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(got, want)
