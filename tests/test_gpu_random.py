"""Seeded randomized sweep of decode configurations on the GPU against the
fp64 oracle: head counts, query tokens per request (including zero),
context lengths from 1 to a few thousand, every page size, cache dtype,
forced and automatic splits, extra pool pages and wider block tables.  Each
case checks every row (small) or sampled rows, and the device status word."""
import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import mla_latent_kv_15_gb300 as mla
    from gpu_case import GpuCase, compare, sample_rows


def draw(seed):
    rng = np.random.Generator(np.random.PCG64(1000 + seed))
    N = int(rng.choice([1, 2, 8, 16, 20, 32, 48, 64, 100, 128, 160, 256]))
    batch = int(rng.integers(1, 12))
    multi = rng.random() < 0.4
    sq = [int(rng.integers(0 if multi else 1, 5 if multi else 2)) for _ in range(batch)]
    if sum(sq) == 0:
        sq[0] = 1
    page = int(rng.choice([16, 32, 64, 128, 256]))
    lo = int(rng.integers(1, 400))
    hi = lo + int(rng.integers(0, 3000))
    dtype = "fp8" if rng.random() < 0.3 else "bf16"
    splits = int(rng.choice([0, 0, 0, 1, 2, 3, 5]))
    lens = rng.integers(lo, hi + 1, size=batch)
    lens = np.maximum(lens, np.array(sq))                     # a request's context holds its new tokens
    extra_pages = int(rng.integers(0, 20))
    pages_needed = int(sum((int(L) + page - 1) // page for L in lens))
    max_pages = int(max((int(L) + page - 1) // page for L in lens)) + int(rng.integers(0, 3))
    return dict(num_heads=N, batch=batch, ctx=(lo, hi), sq=sq, page_size=page, cache_dtype=dtype,
                seed=2000 + seed, seq_lens=lens, num_blocks=pages_needed + extra_pages,
                max_pages=max_pages), splits


@pytest.mark.parametrize("seed", range(24))
def test_random_configuration(seed):
    kw, splits = draw(seed)
    case = synth.make_decode_case(**kw)
    g = GpuCase(case, num_splits_max=splits)
    g.decode(splits)
    rows = None
    if case.total_q * case.num_heads > 3000:
        rows = sample_rows(case, 400, seed=seed)
    compare(case, g, rows=rows)
    assert mla.decode_status(g.workspace) == 0


@pytest.mark.parametrize("seed", range(100, 116))
def test_random_configuration_step_sharper(seed):
    """Drawn configurations through mla_decode_step (the cache write in the
    plan's launch) with the query times 2^k, k in 1..4 (exact in bf16), so
    that scores are sharper than the drawn ones."""
    kw, splits = draw(seed)
    case = synth.make_decode_case(**kw)
    k = 1 + seed % 4
    for name in ("q_abs", "q_pe"):
        bits = getattr(case, name)
        f = (bits.astype(np.uint32) << 16).view(np.float32) * np.float32(2.0 ** k)
        setattr(case, name, (f.view(np.uint32) >> 16).astype(np.uint16))
    g = GpuCase(case, write_new=False, num_splits_max=splits)
    g.out.fill_(float("nan"))
    mla.decode_step(g.new_kv_c, g.new_k_pe, g.slots, g.q_abs, g.q_pe, g.cache, g.block_table, g.seq_lens, g.out,
                    g.workspace, scale=case.scale, query_start_loc=g.qsl, lse=g.lse, num_splits=splits,
                    kv_scale=case.kv_scale)
    torch.cuda.synchronize()
    rows = sample_rows(case, 400, seed=seed) if case.total_q * case.num_heads > 3000 else None
    compare(case, g, rows=rows)
    assert mla.decode_status(g.workspace) == 0
