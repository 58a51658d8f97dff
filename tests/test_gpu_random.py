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
