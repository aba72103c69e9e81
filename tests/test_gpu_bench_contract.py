"""The benchmark's JSON line on a GB300, as its consumers read it.

`python bench.py` with only short step counts: one line whose headline is the
long-context split-K workload, with the roofline, the end-to-end number and its
copy sizes, the clocks, the launch count, and a `per_config` entry (with its own
roofline and oracle baseline) for every workload of the benchmark.
"""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_default_bench_line():
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--steps", "4", "--warmup", "3",
           "--cpu-seconds", "0.5"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
              "roofline", "cpu_baseline", "e2e", "gpu_launches", "clocks", "per_config",
              "append_us", "attention_us"):
        assert k in d, k
    assert d["config"]["workload"] == "long_splitk"
    assert d["steps"] == 4 and d["warmup"] == 3 and d["n_gpus"] == 1 and d["value"] > 0
    rf = d["roofline"]
    assert rf["bound"] == "hbm" and rf["unit"] == "GB/s" and rf["peak"] > 0
    assert abs(rf["frac"] - rf["achieved"] / rf["peak"]) < 1e-3
    e2e = d["e2e"]
    assert e2e["value"] > 0 and e2e["h2d_bytes_per_step"] > 0 and e2e["d2h_bytes_per_step"] > 0
    assert d["gpu_launches"] == 3 * d["steps"]
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert set(d["per_config"]) == {"tiny", "llama3_8b_decode", "llama3_70b_mix",
                                    "long_splitk", "spec_verify"}
    for name, e in d["per_config"].items():
        assert e["us_per_step"] > 0 and e["kernel_us"] > 0, name
        assert e["roofline"]["bound"] == "hbm", name
        assert e["cpu_baseline"]["value"] > 0, name
        assert e.get("device_error_word", 0) == 0, name
