"""mla_decode_no_alloc: the decode for callers that cannot allocate device
memory (graph capture, frameworks that own every device buffer).  Its scratch
is the library's own fixed device array instead of a caller workspace, so it
must give the same results as mla_decode with a workspace.

This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test.
"""
import numpy as np
import pytest
import torch

import synth

if torch.cuda.is_available():
    import mla_latent_kv_15_gb300 as mla
    from gpu_case import GpuCase, TOL_OUT_BF16, TOL_LSE


def _no_alloc(g, out, lse, num_splits=0):
    c = g.case
    mla.decode_no_alloc(g.q_abs, g.q_pe, g.cache, g.block_table, g.seq_lens, out, scale=c.scale,
                        query_start_loc=g.qsl, lse=lse, num_splits=num_splits, kv_scale=c.kv_scale)
    torch.cuda.synchronize()


@pytest.mark.gpu
def test_no_alloc_matches_workspace_decode_on_two_calls():
    cases = [
        synth.make_decode_case(num_heads=128, batch=8, ctx=(300, 3000), sq=[1, 2] * 4, page_size=64, seed=77),
        synth.make_decode_case(num_heads=16, batch=12, ctx=(50, 5000), sq=1, page_size=32, seed=78),
    ]
    for k, case in enumerate(cases):            # two calls in a row, different shapes
        g = GpuCase(case)
        ref_out, ref_lse = (t.clone() for t in g.decode(0))
        out = torch.full_like(ref_out, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        _no_alloc(g, out, lse)
        assert torch.isfinite(out.float()).all()
        err_o = torch.max(torch.abs(out.float() - ref_out.float())).item()
        fin = torch.isfinite(ref_lse)
        assert torch.equal(torch.isfinite(lse), fin)
        err_l = torch.max(torch.abs(lse[fin] - ref_lse[fin])).item() if fin.any() else 0.0
        assert err_o <= TOL_OUT_BF16, (k, err_o)
        assert err_l <= TOL_LSE, (k, err_l)


def test_no_alloc_rejects_batches_beyond_its_scratch():
    """A batch whose scratch need exceeds the fixed array is refused before
    anything is enqueued (no device access: the pointers are never used)."""
    import ctypes
    from mla_latent_kv_15_gb300 import _build
    _build.build()
    import mla_latent_kv_15_gb300 as m
    lib = m.load()
    batch, total_q, heads = 4096, 4096, 128
    assert lib.mla_decode_workspace_size(batch, total_q, heads, 0) > m.NO_ALLOC_SCRATCH_BYTES
    fake = ctypes.c_void_p(1 << 20)
    rc = lib.mla_decode_no_alloc(fake, fake, fake, 100, 64, 0, 1.0, fake, 8, fake, batch, fake, total_q, heads,
                                 0.07, 0, fake, None, None)
    assert rc == -4 and b"static scratch" in lib.mla_last_error()


@pytest.mark.gpu
def test_no_alloc_status_reports_bad_block_ids():
    """Callers without a workspace read the device error word through
    mla_decode_no_alloc_status: a block-table entry past the cache sets
    MLA_DEVERR_BAD_BLOCK, a clean call leaves 0."""
    case = synth.make_decode_case(num_heads=16, batch=3, ctx=(100, 300), page_size=64, seed=79, poison=False)
    g = GpuCase(case)
    out = torch.empty_like(g.out)
    lse = torch.empty_like(g.lse)
    _no_alloc(g, out, lse)
    assert mla.decode_no_alloc_status() == 0
    bad = g.block_table.clone()
    bad[1, 0] = case.num_blocks + 3
    g.block_table = bad
    _no_alloc(g, out, lse)
    assert mla.decode_no_alloc_status(clear=True) & mla.DEVERR_BAD_BLOCK
    assert mla.decode_no_alloc_status() == 0                 # cleared
