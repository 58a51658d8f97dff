"""The sharp-attention inputs really leave the flat-softmax regime (host only).

Scores are computed here directly from the drawn bf16 values (numpy dot
products over the gathered rows of one request), independently of the
oracle and of the library, to check what the GPU sharp-score tests rely on:
the rising-key inputs make the running maximum of a row grow past the lazy
rescale threshold (8 in log2 units) several times, and the widened query
draws spread a row's scores over tens of nats.
"""
import math

import numpy as np

import synth


def _scores(case, b=0, h=0):
    rows = []
    L = int(case.seq_lens[b])
    for j in range(L):
        blk = case.block_table[b, j // case.page_size]
        rows.append(case.pool[blk, j % case.page_size])
    # the step's new rows overwrite the last Sq positions
    t0, t1 = case.query_start_loc[b], case.query_start_loc[b + 1]
    new = np.concatenate([case.new_kv_c, case.new_k_pe], axis=1)
    for k, t in enumerate(range(t0, t1)):
        rows[L - (t1 - t0) + k] = new[t]
    kv = synth.bf16_bits_to_f32(np.stack(rows)).astype(np.float64)
    q = synth.bf16_bits_to_f32(np.concatenate([case.q_abs[t1 - 1, h], case.q_pe[t1 - 1, h]])).astype(np.float64)
    return case.scale * kv @ q


def test_rising_keys_force_repeated_rescales():
    case = synth.make_decode_case(num_heads=2, batch=2, ctx=(4000, 5000), page_size=64, seed=3, rising=0.03)
    s = _scores(case) / math.log(2.0)                     # log2 units, as the kernel's running maximum
    m, rescales = -np.inf, 0
    for t in range(0, s.size, 64):                       # the kernel's 64-key tiles
        tmax = s[t:t + 64].max()
        if tmax > m + 8.0:
            rescales += m > -np.inf
            m = tmax
    assert rescales >= 3, rescales
    assert s[-64:].max() == s.max()                       # the row maximum sits in the last tile


def test_wide_query_spreads_scores():
    case = synth.make_decode_case(num_heads=2, batch=1, ctx=(3000, 3000), page_size=64, seed=4, q_std=8.0)
    s = _scores(case)
    assert s.max() - np.median(s) > 10.0                  # nats
    p = np.exp(s - s.max())
    assert p.sum() < 50.0                                 # a few keys carry the row
