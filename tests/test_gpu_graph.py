"""A decode step (cache write + decode) captured in a CUDA graph and replayed:
the library makes no host synchronisation and allocates nothing per call, so
the captured step gives the oracle's result on every replay, and a replay
after the inputs change in place sees the new inputs."""
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import mla_latent_kv_15_gb300 as mla
    from gpu_case import GpuCase, compare, bf16_tensor


def _capture(g, case):
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        mla.cache_write(g.new_kv_c, g.new_k_pe, g.slots, g.cache, case.kv_scale)
        mla.decode(g.q_abs, g.q_pe, g.cache, g.block_table, g.seq_lens, g.out, g.workspace, scale=case.scale,
                   query_start_loc=g.qsl, lse=g.lse, kv_scale=case.kv_scale)
    return graph


@pytest.mark.parametrize("cache_dtype,num_heads", [("bf16", 128), ("bf16", 16), ("fp8", 128)])
def test_step_in_a_cuda_graph(cache_dtype, num_heads):
    case = synth.make_decode_case(num_heads=num_heads, batch=5, ctx=(500, 2000), page_size=64,
                                  cache_dtype=cache_dtype, seed=47, poison=False)
    g = GpuCase(case, write_new=False)
    g.write_new()
    g.decode()                               # one eager step first (one-time launch setup)
    graph = _capture(g, case)
    cache_host = oracle.prepare_cache(case)
    for _ in range(2):
        g.out.fill_(float("nan"))
        g.lse.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        compare(case, g, cache_host=cache_host)
        assert mla.decode_status(g.workspace) == 0


def test_graph_replay_sees_new_inputs():
    """The captured step reads its inputs at replay time: a new query copied
    into the same buffer changes the result to the new query's."""
    case = synth.make_decode_case(num_heads=128, batch=4, ctx=(300, 1500), page_size=64, seed=48, poison=False)
    g = GpuCase(case, write_new=False)
    g.write_new()
    g.decode()
    graph = _capture(g, case)
    other = synth.make_decode_case(num_heads=128, batch=4, ctx=(300, 1500), page_size=64, seed=49, poison=False)
    case.q_abs = other.q_abs                 # same shapes; the cache, lengths and tables stay
    case.q_pe = other.q_pe
    g.q_abs.copy_(bf16_tensor(other.q_abs))
    g.q_pe.copy_(bf16_tensor(other.q_pe))
    graph.replay()
    torch.cuda.synchronize()
    compare(case, g)
