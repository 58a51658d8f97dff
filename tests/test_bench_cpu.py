"""bench.py's host-only paths on CPU: every reference arm (the fp64 oracle
timed on the host) prints one well-formed JSON line on rank 0 and nothing on
the other ranks."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.parametrize("op", ["v_up_proj", "q_absorb"])
def test_projection_reference_arm_line(op):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--op", op,
                        "--steps", "1", "--warmup", "0"], capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["op"] == op
    assert d["value"] > 0 and d["unit"] == "tokens/s" and d["higher_is_better"] is True
    for key in ("cpu_baseline", "e2e", "config", "ms_per_step", "steps", "warmup"):
        assert key in d
    assert d["config"]["num_heads"] == 128 and d["config"]["num_tokens"] == 64


@pytest.mark.parametrize("op", ["decode", "gather"])
def test_reference_arm_line_small_workload(op):
    """The decode and gather reference arms (oracle on the host cores) on the
    small workload: one JSON line with the contract's keys; the reference
    line carries its own cpu_baseline and an e2e with no copies."""
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--op", op,
                        "--workload", "tiny_n16_ctx256", "--steps", "2", "--warmup", "1"],
                       capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["steps"] == 2 and d["warmup"] == 1 and d["n_gpus"] == 1
    assert d["value"] > 0 and d["higher_is_better"] is True and d["vs_baseline"] is None
    assert d["config"]["workload"].startswith("tiny_n16_ctx256")
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["e2e"]["value"] == d["value"] and d["e2e"]["unit"] == d["unit"]


def test_reference_arm_other_ranks_exit_quietly():
    """Under a multi-rank launch only rank 0 runs the reference arm; the
    other ranks print nothing and exit 0."""
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "tiny_n16_ctx256", "--steps", "2", "--warmup", "1"],
                       capture_output=True, text=True, timeout=300, cwd=ROOT, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""


def test_algorithmic_bytes_and_flops_by_hand():
    """The roofline's numerator: every visible latent row read once, queries
    read, outputs and LSE written; 2 * (576 + 512) FLOP per visible (key,
    query row), with the multi-token causal window (token t of an Sq-token
    request sees seq_len - Sq + 1 + t keys)."""
    sys.path.insert(0, ROOT)
    import bench
    import synth
    N = 4
    case = synth.make_decode_case(num_heads=N, batch=3, ctx=(1, 1), sq=[1, 1, 2], seq_lens=[5, 0, 3],
                                  page_size=16, seed=3, poison=False)
    a = bench.algorithmic(case)
    T = 4
    assert a["kv"] == (5 + 0 + 3) * 576 * 2
    assert a["q"] == T * N * 576 * 2
    assert a["out"] == T * N * (512 * 2 + 4)
    assert a["decode_bytes"] == a["kv"] + a["q"] + a["out"]
    visible = 5 + 0 + (2 + 3)
    assert a["flops"] == 2 * (576 + 512) * N * visible
    fp8 = synth.make_decode_case(num_heads=N, batch=3, ctx=(1, 1), sq=[1, 1, 2], seq_lens=[5, 0, 3],
                                 page_size=16, seed=3, poison=False, cache_dtype="fp8")
    assert bench.algorithmic(fp8)["kv"] == 8 * 576
