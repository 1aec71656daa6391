"""bench.py's JSON line on a GPU: one short run of the quarter-length 1.4B layer (with the
end-to-end, decode, backward and SSD objects, a short oracle sample and no per-config
objects) prints one line with the contract's keys and self-consistent values."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.gpu
def test_bench_json_line():
    cmd = [sys.executable, "bench.py", "--workload", "m1p4b_L1024", "--steps", "5", "--warmup", "3", "--no-configs",
           "--cpu-seconds", "1", "--e2e-steps", "3", "--decode-steps", "64", "--bwd-steps", "2", "--ssd-steps", "2"]
    out = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    line = json.loads(out.stdout.strip().splitlines()[-1])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
              "vs_baseline", "dtype", "data", "config", "roofline", "cpu_baseline", "e2e", "gpu_launches", "clocks"):
        assert k in line, k
    assert line["n_gpus"] == 1 and line["steps"] == 5 and line["warmup"] == 3 and line["value"] > 0
    r = line["roofline"]
    for k in ("bound", "achieved", "peak", "unit", "frac", "traffic"):
        assert k in r, k
    assert 0 < r["frac"] < 1.5 and abs(r["achieved"] / r["peak"] - r["frac"]) < 1e-6
    assert line["gpu_launches"] == line["steps"]  # one launch per forward step
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] > 0
    e = line["e2e"]
    assert e["value"] > 0 and e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] > 0
    c = line["clocks"]
    assert c["sm_mhz"] is None or c["sm_mhz"] > 0
    for k in ("decode", "backward", "ssd"):
        assert k in line and line[k], k
