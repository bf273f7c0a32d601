"""bench.py's real GPU path on the tiny workload: one JSON line with every key the bench contract asks for, values
that agree with each other, and the kernels of this library doing the work (a positive launch count)."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_bench_line_on_the_tiny_workload():
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--workload", "tiny", "--steps", "4", "--warmup", "3",
           "--legs", "io,floor,e2e,noio,cpu,spread", "--cpu-budget", "1"]
    out = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    line = json.loads(out.stdout.strip().splitlines()[-1])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
                "vs_baseline", "dtype", "data", "config", "roofline", "cpu_baseline", "e2e", "clocks",
                "gpu_launches"):
        assert key in line, key
    assert line["n_gpus"] == 1 and line["steps"] == 4 and line["warmup"] == 3
    assert line["value"] > 0 and line["gpu_launches"] > 0
    # value = selections per step over the timed time (tiny: 1 request x 1 layer per step)
    assert abs(line["value"] - 1.0 / (line["ms_per_step"] / 1e3)) <= 1e-6 * line["value"]
    assert "tiny" in line["config"]["workload"]
    roof = line["roofline"]
    assert roof["peak"] > 0 and abs(roof["frac"] - max(roof["frac"], roof["hbm_frac"])) < 1e-12
    e2e = line["e2e"]
    assert e2e["value"] > 0 and e2e["h2d_bytes_per_step"] > 0 and e2e["out_slots_match_device_path"]
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["noio"]["value"] > 0
    assert len(line["headline"]["repeats"]["values"]) == 3
