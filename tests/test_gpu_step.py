"""mla_decode_step (the step's cache write done by extra blocks of the
scheduler's launch, then the decode) against the oracle, and its cache bytes
against a separate mla_cache_write."""
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import mla_latent_kv_15_gb300 as mla
    from gpu_case import GpuCase, compare


def _step(g, case, slots=None, num_splits=0):
    mla.decode_step(g.new_kv_c, g.new_k_pe, g.slots if slots is None else slots, g.q_abs, g.q_pe, g.cache,
                    g.block_table, g.seq_lens, g.out, g.workspace, scale=case.scale, query_start_loc=g.qsl,
                    lse=g.lse, num_splits=num_splits, kv_scale=case.kv_scale)
    torch.cuda.synchronize()


@pytest.mark.parametrize("num_heads,sq,cache_dtype,num_splits", [
    (128, 1, "bf16", 0), (16, 1, "bf16", 0), (128, [1, 3, 2, 1, 4], "bf16", 3), (128, 1, "fp8", 0),
    (16, 2, "fp8", 2)])
def test_decode_step_matches_oracle(num_heads, sq, cache_dtype, num_splits):
    case = synth.make_decode_case(num_heads=num_heads, batch=5, ctx=(200, 1500), sq=sq, page_size=64,
                                  cache_dtype=cache_dtype, seed=700 + num_heads + num_splits, poison=False)
    g = GpuCase(case, write_new=False, num_splits_max=num_splits)
    g.out.fill_(float("nan"))
    _step(g, case, num_splits=num_splits)
    compare(case, g)
    assert mla.decode_status(g.workspace) == 0


@pytest.mark.parametrize("cache_dtype", ["bf16", "fp8"])
def test_decode_step_cache_bytes_equal_cache_write(cache_dtype):
    case = synth.make_decode_case(num_heads=32, batch=37, ctx=(1, 300), sq=[1, 3] * 18 + [2], page_size=16,
                                  cache_dtype=cache_dtype, seed=710, poison=False)
    slots = torch.from_numpy(case.slot_mapping.copy())
    slots[5] = -1                                             # a padding token
    slots = slots.cuda()
    a = GpuCase(case, write_new=False)
    b = GpuCase(case, write_new=False)
    mla.cache_write(a.new_kv_c, a.new_k_pe, slots, a.cache, case.kv_scale)
    _step(b, case, slots=slots)
    torch.cuda.synchronize()
    assert torch.equal(a.cache.view(torch.uint8), b.cache.view(torch.uint8))


def test_decode_step_without_new_rows_is_a_decode():
    case = synth.make_decode_case(num_heads=64, batch=4, ctx=(100, 900), page_size=64, seed=720, poison=False)
    g = GpuCase(case)                                         # new rows already written
    empty = torch.empty(0, dtype=torch.int64, device="cuda")
    mla.decode_step(g.new_kv_c[:0], g.new_k_pe[:0], empty, g.q_abs, g.q_pe, g.cache, g.block_table, g.seq_lens,
                    g.out, g.workspace, scale=case.scale, query_start_loc=g.qsl, lse=g.lse)
    torch.cuda.synchronize()
    compare(case, g)
