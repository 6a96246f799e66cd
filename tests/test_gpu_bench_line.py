"""bench.py's own arm on the GPU prints one JSON line with the keys the
harness reads: the metric, the roofline object of the dominant kernel, the
end-to-end figure through the host-buffer pipeline with its copy bytes, the
launch count, the sampled clocks and the per-kernel breakdown.  A small
workload (the toy and the decode shape), a few steps, in a subprocess."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(*args):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT,
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    return json.loads(lines[0])


@pytest.mark.parametrize("workload", ["toy", "decode"])
def test_bench_line_keys(workload):
    d = _run("--workload", workload, "--steps", "3", "--warmup", "3", "--no-cpu-baseline")
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
              "roofline", "e2e", "gpu_launches", "clocks", "kernels"):
        assert k in d, k
    assert d["n_gpus"] == 1 and d["steps"] == 3 and d["warmup"] == 3
    assert d["unit"] == "tokens/s" and d["value"] > 0 and d["higher_is_better"] is True
    assert d["data"] == "synthetic" and d["scaling"] == "weak"
    assert isinstance(d["config"]["workload"], str)
    rf = d["roofline"]
    assert rf["bound"] == "hbm" and rf["unit"] == "GB/s" and rf["peak"] > 0
    assert abs(rf["frac"] - rf["achieved"] / rf["peak"]) < 1e-3
    assert "traffic" in rf  # null away from the captured prefill size
    e = d["e2e"]
    assert e["unit"] == "tokens/s" and e["value"] > 0
    assert e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] > 0
    # route, layout, dispatch, combine per step: four calls, six kernels at most
    assert 4 * d["steps"] <= d["gpu_launches"] <= 6 * d["steps"]
    c = d["clocks"]
    assert "sm_mhz" in c and "sm_max_mhz" in c and isinstance(c["reasons"], list)
    for k in ("route", "layout", "dispatch", "combine"):
        assert d["kernels"][k]["ms"] > 0 and d["kernels"][k]["bound"] in ("alu", "latency", "hbm")
