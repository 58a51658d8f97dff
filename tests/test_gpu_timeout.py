"""Failure detection of the decode kernels: every on-chip wait is bounded.

The test makes one wait run out without faulting, trapping or hanging the
GPU: with the library's test setting, the first CTA of the grid never loads
its first cache tile, so its MMA issuer's bounded wait for that tile expires
(limit 2 ms instead of the default 1 s).  The CTA then records
MLA_DEVERR_TIMEOUT in the device error word, stops waiting on its own
pipeline, still takes the partial scores its peer sends, and both CTAs of the
pair run to the end.  The call must return promptly, the host must read the
timeout bit, and the next ordinary decode on the same stream must be clean
and match the oracle: the context stays usable.
"""
import time

import numpy as np
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import mla_latent_kv_15_gb300 as mla
    from gpu_case import GpuCase, compare


@pytest.mark.parametrize("cache_dtype,heads", [("bf16", 128), ("fp8", 128), ("bf16", 16)])
def test_expired_wait_reports_timeout_and_context_stays_usable(cache_dtype, heads):
    # enough tiles that the first CTA pair of the grid owns real work
    case = synth.make_decode_case(num_heads=heads, batch=8, ctx=(2000, 4000), page_size=64,
                                  cache_dtype=cache_dtype, seed=81 + heads)
    g = GpuCase(case)
    torch.cuda.synchronize()
    mla.set_decode_wait_test(skip_first_tile=True, wait_limit_ns=2_000_000)
    try:
        t0 = time.perf_counter()
        g.decode()                                      # synchronises
        elapsed = time.perf_counter() - t0
    finally:
        mla.set_decode_wait_test(False, 0)
    assert mla.decode_status(g.workspace) & mla.DEVERR_TIMEOUT
    assert elapsed < 5.0, elapsed
    # the same stream, an ordinary decode: clean status, oracle-correct
    g.out.fill_(float("nan"))
    g.lse.fill_(float("nan"))
    g.decode()
    assert mla.decode_status(g.workspace) == 0
    rows = None if case.total_q * heads <= 2000 else np.arange(0, case.total_q * heads, 7)
    compare(case, g, rows=rows)


def test_wait_test_setting_is_validated():
    with pytest.raises(mla.MLAError):
        mla.set_decode_wait_test(True, 10)              # below 0.1 ms
    mla.set_decode_wait_test(False, 0)
