"""Seeded synthetic inputs for absorbed-MLA decode over a paged latent KV cache.

This module only draws inputs: random values, context lengths, block tables
and slot mappings.  It holds none of the method's arithmetic (no scores, no
softmax, no quantisation), so both the fp64 oracle and the CUDA library can be
fed from it without sharing code.

Shapes and distributions follow the serving-shaped workloads the MLA pages
describe (vllm/v1/attention/backends/mla/common.py, module docstring, "More
Extent Definitions": Lkv=512, R=64; cache layout (num_blocks, block_size,
head_size) from ``get_kv_cache_shape``):

* latent rows ``[kv_c | k_pe]`` (576 wide) and absorbed queries
  ``[q_abs | q_pe]`` are N(0,1)*0.5 drawn in float32, rounded to bf16 (RNE);
* context lengths are uniform integers in [lo, hi] and include the new query
  tokens of the step (the sequence-length convention of the AITER MLA
  backend, ``forward_mqa``, multi-token verify path);
* block tables are disjoint slices of one random permutation of the page pool;
  unused table entries are -1;
* the new latent rows of the step (one per query token) go to the slots of the
  last ``Sq`` positions of each sequence, so ``slot_mapping`` is as random as
  the block tables are.

Arrays are numpy; bf16 values are carried as their uint16 bit patterns.
"""
from __future__ import annotations

import math
import os
from dataclasses import dataclass, field

import numpy as np

LKV = 512
ROPE = 64
DQK = LKV + ROPE
BF16_NAN = np.uint16(0x7FC0)

# Named workloads (head count, batch, context range, query tokens, page size,
# page pool).  "tiny" is the small case the oracle finishes in well under a
# second; the others are the serving-shaped decode batches.
WORKLOADS = {
    "tiny_n16_ctx256": dict(num_heads=16, batch=1, ctx=(256, 256), sq=1,
                            page_size=64, num_blocks=8, cache_dtype="bf16", seed=1),
    "dsv3_n128_b64_ctx1k-8k": dict(num_heads=128, batch=64, ctx=(1024, 8192), sq=1,
                                   page_size=64, num_blocks=40000, cache_dtype="bf16", seed=2),
    "n16_b128_ctx8k-32k": dict(num_heads=16, batch=128, ctx=(8192, 32768), sq=1,
                               page_size=64, num_blocks=52000, cache_dtype="bf16", seed=3),
    "dsv3_n128_b64_ctx1k-8k_fp8": dict(num_heads=128, batch=64, ctx=(1024, 8192), sq=1,
                                       page_size=64, num_blocks=40000, cache_dtype="fp8", seed=4),
    "mtp_n128_sq4_b32_ctx2k-16k": dict(num_heads=128, batch=32, ctx=(2048, 16384), sq=4,
                                       page_size=64, num_blocks=40000, cache_dtype="bf16", seed=5),
    "mtp_mixed_n128_b32_ctx2k-16k": dict(num_heads=128, batch=32, ctx=(2048, 16384),
                                         sq=[4] * 16 + [1] * 16, page_size=64,
                                         num_blocks=40000, cache_dtype="bf16", seed=6),
}


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (round-to-nearest-even) and return the bits."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def _normal_bf16_pages(seed: int, npages: int, page_size: int, std: float = 0.5) -> np.ndarray:
    """N(0,1)*std latent rows for `npages` pages as bf16 bits, drawn in chunks of
    256 pages, each from its own PCG64 stream spawned from `seed` (the result
    does not depend on how many threads draw them)."""
    import concurrent.futures as cf
    chunk = 256
    n = (npages + chunk - 1) // chunk
    seqs = np.random.SeedSequence([seed, 0x5EED]).spawn(n)
    out = np.empty((npages, page_size, DQK), dtype=np.uint16)

    def fill(i):
        lo, hi = i * chunk, min(npages, (i + 1) * chunk)
        g = np.random.Generator(np.random.PCG64(seqs[i]))
        v = g.standard_normal((hi - lo, page_size, DQK), dtype=np.float32)
        v *= np.float32(std)
        out[lo:hi] = to_bf16_bits(v)

    with cf.ThreadPoolExecutor(max_workers=min(32, os.cpu_count() or 4)) as ex:
        list(ex.map(fill, range(n)))
    return out


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to float32 (exact)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


@dataclass
class DecodeCase:
    num_heads: int
    page_size: int
    num_blocks: int
    cache_dtype: str                 # "bf16" or "fp8": how the cache is stored
    seq_lens: np.ndarray             # int32 [B]
    query_start_loc: np.ndarray      # int32 [B+1]
    block_table: np.ndarray          # int32 [B, max_pages]; -1 = unused
    q_abs: np.ndarray                # uint16 (bf16 bits) [T, N, 512]
    q_pe: np.ndarray                 # uint16 (bf16 bits) [T, N, 64]
    pool: np.ndarray                 # uint16 (bf16 bits) [num_blocks, page, 576]
    new_kv_c: np.ndarray             # uint16 [T, 512] latent rows written this step
    new_k_pe: np.ndarray             # uint16 [T, 64]
    slot_mapping: np.ndarray         # int64 [T]
    referenced_slots: np.ndarray     # int64: every slot a sequence can read
    scale: float                     # softmax scale 1/sqrt(P+R)
    kv_scale: float                  # per-tensor fp8 scale (1.0 for bf16)
    name: str = ""
    extra: dict = field(default_factory=dict)

    @property
    def batch(self) -> int:
        return int(self.seq_lens.shape[0])

    @property
    def total_q(self) -> int:
        return int(self.query_start_loc[-1])

    @property
    def max_pages(self) -> int:
        return int(self.block_table.shape[1])


def make_decode_case(*, num_heads: int, batch: int, ctx: tuple[int, int], sq=1,
                     page_size: int = 64, num_blocks: int | None = None,
                     cache_dtype: str = "bf16", seed: int = 0, poison: bool = True,
                     seq_lens=None, qk_nope_dim: int = 128, qk_rope_dim: int = ROPE,
                     max_pages: int | None = None, name: str = "", q_std: float = 0.5,
                     kv_std: float = 0.5, rising: float = 0.0, rising_q: float = 4.0) -> DecodeCase:
    """Draw one decode batch.

    ``sq`` is an int (same number of query tokens for every request) or a list
    of per-request counts.  ``seq_lens`` may be given explicitly (edge cases);
    otherwise lengths are uniform in ``ctx``.  With ``poison`` the pages no
    request references hold bf16 NaN, so a wrong gather cannot go unnoticed.

    Sharper attention: ``q_std`` and ``kv_std`` are the standard deviations of
    the query and latent-row draws (0.5 by default).  ``rising`` > 0 writes
    ``rising * j`` into the first rope dimension of the row at context
    position j of every request (the step's new rows included) and sets the
    first rope dimension of every query to ``rising_q``, so that scores grow
    along the context and the running maximum of a row keeps rising.
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    sqs = np.asarray([sq] * batch if np.isscalar(sq) else list(sq), dtype=np.int64)
    assert sqs.shape == (batch,)
    if seq_lens is None:
        lens = rng.integers(ctx[0], ctx[1] + 1, size=batch).astype(np.int64)
    else:
        lens = np.asarray(seq_lens, dtype=np.int64)
    pages = (lens + page_size - 1) // page_size
    need = int(pages.sum())
    if num_blocks is None:
        num_blocks = max(need, 1)
    assert need <= num_blocks, f"pool of {num_blocks} pages cannot hold {need}"
    mp = max(int(pages.max()) if batch else 1, 1) if max_pages is None else max_pages
    perm = rng.permutation(num_blocks).astype(np.int32)
    table = np.full((batch, mp), -1, dtype=np.int32)
    off = 0
    for b in range(batch):
        table[b, :pages[b]] = perm[off:off + pages[b]]
        off += int(pages[b])

    qsl = np.zeros(batch + 1, dtype=np.int32)
    qsl[1:] = np.cumsum(sqs)
    total_q = int(qsl[-1])

    q = rng.standard_normal((total_q, num_heads, DQK), dtype=np.float32) * np.float32(q_std)
    if rising > 0:
        q[:, :, LKV] = np.float32(rising_q)
    qb = to_bf16_bits(q)
    pool = np.empty((num_blocks, page_size, DQK), dtype=np.uint16)
    used = table[table >= 0]
    if poison:
        pool[...] = BF16_NAN
    else:
        pool[...] = 0
    if used.size:
        pool[used] = _normal_bf16_pages(seed, used.size, page_size, kv_std)
    new = rng.standard_normal((total_q, DQK), dtype=np.float32) * np.float32(kv_std)
    if rising > 0:
        # position of each new row: the last Sq positions of its request
        pos_new = np.concatenate([np.arange(int(lens[b]) - int(sqs[b]), int(lens[b])) for b in range(batch)]) \
            if total_q else np.zeros(0, dtype=np.int64)
        new[:, LKV] = np.float32(rising) * np.maximum(pos_new, 0).astype(np.float32)
        for b in range(batch):
            for lp in range(int(pages[b])):
                pos = lp * page_size + np.arange(page_size)
                pool[table[b, lp], :, LKV] = to_bf16_bits(np.float32(rising) * pos.astype(np.float32))
    newb = to_bf16_bits(new)

    # slots of the new tokens: the last Sq positions of each sequence
    slots = np.empty(total_q, dtype=np.int64)
    for b in range(batch):
        for t in range(int(sqs[b])):
            pos = int(lens[b]) - int(sqs[b]) + t
            if pos < 0:
                slots[qsl[b] + t] = -1           # nothing to write (padding token)
            else:
                slots[qsl[b] + t] = int(table[b, pos // page_size]) * page_size + pos % page_size
    # every slot of every referenced page (used to prepare an fp8 cache from
    # the bf16 pool; whole pages, so rows past seq_len in a last page are
    # finite values too, as a real writer leaves them)
    ref_slots = (used.astype(np.int64)[:, None] * page_size
                 + np.arange(page_size, dtype=np.int64)[None, :]).ravel()

    kv_scale = 1.0
    if cache_dtype == "fp8":
        # Per-tensor calibration of the config: the largest magnitude the fp8
        # cache will hold maps to the e4m3 maximum (448).
        live = np.concatenate([bf16_bits_to_f32(pool[used]).ravel(), bf16_bits_to_f32(newb).ravel()])
        kv_scale = float(np.float32(np.abs(live).max()) / np.float32(448.0)) if live.size else 1.0

    return DecodeCase(
        num_heads=num_heads, page_size=page_size, num_blocks=num_blocks,
        cache_dtype=cache_dtype, seq_lens=lens.astype(np.int32), query_start_loc=qsl,
        block_table=table, q_abs=np.ascontiguousarray(qb[..., :LKV]),
        q_pe=np.ascontiguousarray(qb[..., LKV:]), pool=pool,
        new_kv_c=np.ascontiguousarray(newb[:, :LKV]), new_k_pe=np.ascontiguousarray(newb[:, LKV:]),
        slot_mapping=slots, referenced_slots=ref_slots,
        scale=1.0 / math.sqrt(qk_nope_dim + qk_rope_dim), kv_scale=kv_scale, name=name)


def workload(name: str, **over) -> DecodeCase:
    """Draw a named workload (see ``WORKLOADS``); keyword overrides allowed."""
    cfg = dict(WORKLOADS[name])
    cfg.update(over)
    return make_decode_case(name=name, **cfg)


def expanded_weights(seed: int, num_heads: int, lkv: int = LKV, p: int = 128, v: int = 128):
    """W_UK [Lkv, N, P] and W_UV [Lkv, N, V] drawn N(0, 1/Lkv) in float64, plus
    q_nope [T, N, P] drawn later by the caller; used for the two-path check."""
    rng = np.random.Generator(np.random.PCG64(10_000 + seed))
    sd = 1.0 / math.sqrt(lkv)
    w_uk = rng.standard_normal((lkv, num_heads, p)) * sd
    w_uv = rng.standard_normal((lkv, num_heads, v)) * sd
    return w_uk, w_uv


def random_partials(seed: int, rows: int, dim: int = LKV, neg_inf_frac: float = 0.0):
    """Two partial attention results (o, lse) for the merge: o ~ N(0, 0.25) in
    float32, lse ~ N(0, 4); a fraction of lse entries set to -inf (empty
    partials)."""
    rng = np.random.Generator(np.random.PCG64(20_000 + seed))
    o_a = (rng.standard_normal((rows, dim), dtype=np.float32) * np.float32(0.5))
    o_b = (rng.standard_normal((rows, dim), dtype=np.float32) * np.float32(0.5))
    lse_a = (rng.standard_normal(rows) * 2.0).astype(np.float32)
    lse_b = (rng.standard_normal(rows) * 2.0).astype(np.float32)
    if neg_inf_frac > 0:
        lse_a[rng.random(rows) < neg_inf_frac] = -np.inf
        lse_b[rng.random(rows) < neg_inf_frac] = -np.inf
    return o_a, lse_a, o_b, lse_b


def projection_weights(seed: int, num_heads: int, lkv: int = LKV, p: int = 128, v: int = 128):
    """bf16 bit patterns of W_UK [Lkv, N, P] and W_UV [Lkv, N, V] (the split of
    kv_b_proj's transposed weight, common.py process_weights_after_loading),
    drawn N(0, 1/Lkv) in float32 and rounded to bf16 (RNE)."""
    rng = np.random.Generator(np.random.PCG64(30_000 + seed))
    sd = np.float32(1.0 / math.sqrt(lkv))
    w_uk = rng.standard_normal((lkv, num_heads, p), dtype=np.float32) * sd
    w_uv = rng.standard_normal((lkv, num_heads, v), dtype=np.float32) * sd
    return to_bf16_bits(w_uk), to_bf16_bits(w_uv)


def bf16_normal(seed: int, shape, std: float = 0.5) -> np.ndarray:
    """bf16 bit patterns of N(0, std^2) float32 draws (RNE)."""
    rng = np.random.Generator(np.random.PCG64(40_000 + seed))
    return to_bf16_bits(rng.standard_normal(shape, dtype=np.float32) * np.float32(std))
