"""The benchmark's own arm, run as the driver runs it (a fresh process), on a
truncated workload: its one JSON line carries the contract's keys with
sensible values in every mode (fused, split at the flag, CUDA graph, half
accumulator, clipping)."""
import json
import os
import subprocess
import sys

import pytest

import bench

pytestmark = pytest.mark.gpu


def run(args):
    out = subprocess.run([sys.executable, os.path.join(bench.ROOT, "bench.py")] + args,
                         capture_output=True, text=True, timeout=900, cwd=bench.ROOT)
    assert out.returncode == 0, out.stderr[-3000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, out.stdout[-2000:]
    return json.loads(lines[0])


@pytest.mark.parametrize("mode", [[], ["--split"], ["--graph"], ["--acc", "half"],
                                  ["--clip", "1.0"]])
def test_bench_line(mode):
    d = run(["--workload", "llama7b-n1", "--elements", str(1 << 24), "--steps", "3",
             "--warmup", "3", "--e2e-steps", "1", "--skip-cpu", "--skip-probe"] + mode)
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
              "roofline", "clocks", "gpu_launches", "e2e"):
        assert k in d, k
    assert d["metric"] == bench.METRIC and d["unit"] == "params/s" and d["n_gpus"] == 1
    assert d["steps"] == 3 and d["warmup"] == 3 and d["scaling"] == "weak"
    assert d["value"] == pytest.approx((1 << 24) / (d["ms_per_step"] * 1e-3), rel=1e-6)
    assert d["config"]["workload"].startswith("llama7b-n1")
    r = d["roofline"]
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and r["peak"] > 0
    assert r["frac"] == pytest.approx(r["achieved"] / r["peak"], rel=1e-3)
    assert r["traffic"] is None            # truncated workload: no recorded traffic applies
    assert d["gpu_launches"] >= 3 * 9      # at least the step's kernels, every step
    e = d["e2e"]
    assert e["value"] > 0 and e["h2d_bytes_per_step"] == 8 * (1 << 24) * 2
    assert e["d2h_bytes_per_step"] > 0
    assert "sm_mhz" in d["clocks"] and "reasons" in d["clocks"]
