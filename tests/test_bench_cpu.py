"""bench.py's host-only paths on CPU: the projection ops' reference arm (the
fp64 oracle timed on the host) prints one well-formed JSON line."""
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
