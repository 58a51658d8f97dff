"""The multi-process path of bench.py on CPU (gloo, two ranks): the decode of
one batch does not shard, so N GPUs run N replicas; the job's time is the
slowest rank's and its rate counts the units of every rank."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    # rank r's step, kernel and e2e times
    mine = [1.0 + rank, 0.5 + 0.25 * rank, 2.0 - rank]
    got = bench.max_over_ranks(mine, dist)
    rate = bench.job_throughput(64, world, got[0])
    # the reference arm: only rank 0 produces a line
    args = type("A", (), {"op": "decode", "workload": "tiny_n16_ctx256", "steps": 1, "warmup": 0,
                          "ref_requests": 1})()
    ref = bench.run_reference(args)
    out.put((rank, got, rate, ref is not None))
    dist.barrier()
    dist.destroy_process_group()


def test_replicas_take_the_slowest_rank_and_count_every_rank():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = {}
    for _ in range(world):
        rank, got, rate, printed = q.get(timeout=120)
        res[rank] = (got, rate, printed)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank in range(world):
        got, rate, printed = res[rank]
        assert got == [2.0, 0.75, 2.0]                       # element-wise max over the two ranks
        assert rate == pytest.approx(2 * 64 / 2.0e-3)         # both ranks' tokens / the slowest time
        assert printed == (rank == 0)
