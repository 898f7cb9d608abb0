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


@pytest.mark.parametrize("mode", [["--skip-table"], ["--api", "sync"], ["--split"], ["--graph"],
                                  ["--acc", "half"], ["--acc", "half", "--api", "sync"],
                                  ["--acc", "half", "--api", "async"],
                                  ["--clip", "1.0", "--skip-table"],
                                  ["--clip", "1.0", "--api", "sync"], ["--clip", "1.0", "--graph"],
                                  ["--api", "async_oop", "--skip-table"]])
def test_bench_line(mode):
    d = run(["--workload", "llama7b-n1", "--elements", str(1 << 24), "--steps", "3",
             "--warmup", "3", "--e2e-steps", "1", "--skip-cpu", "--skip-probe"] + mode)
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
              "roofline", "clocks", "gpu_launches", "e2e"):
        assert k in d, k
    assert d["metric"] == bench.METRIC and d["unit"] == "params/s" and d["n_gpus"] == 1
    assert d["steps"] == 3 and d["warmup"] == 3 and d["scaling"] == "strong"
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
    if "half" in mode:   # every half-accumulator form names its own entry points
        assert "halfacc" in d["config"]["api"]
        assert d["config"]["accumulator"] == "half"


def test_small_shard_runs_the_fused_step():
    """The 2^20-parameter workload's shard fits one co-resident grid: every
    step of the default API is one fused launch, and it dominates the roofline."""
    d = run(["--workload", "flat-1m-n2", "--steps", "20", "--warmup", "3", "--e2e-steps", "2",
             "--skip-cpu", "--skip-probe", "--skip-table"])
    assert d["roofline"]["kernel"] == "fused"
    assert d["gpu_launches"] == 20
    assert d["value"] > 0 and d["e2e"]["value"] > 0


def test_graph_of_a_short_step_replays_several_steps():
    """A step far shorter than the host's replay call is captured several to a
    graph: exactly K steps are timed, the warm-up is whole replays, and the
    device state counts every step."""
    d = run(["--workload", "flat-1m-n2", "--graph", "--steps", "100", "--warmup", "3",
             "--e2e-steps", "2", "--skip-cpu", "--skip-probe", "--skip-table"])
    c = d["config"]
    per = c["steps_per_replay"]
    assert per > 1 and 100 % per == 0 and c["warmup_steps_run"] == per
    assert d["steps"] == 100 and d["gpu_launches"] == 100      # one fused kernel per step
    assert c["device_state_after_timed_steps"]["iterations"] == 1 + per + 100


def test_default_api_keeps_the_step_state_on_the_device_and_measures_the_table():
    """The default API (zs_shard_step_async, no host round trip) runs every
    step: the device state read back after the run counts the warm-up and
    timed steps; the e2e leg reads each step's state back; the other target
    workloads are measured in the same run, each with its own clock record."""
    el = 1 << 22
    d = run(["--elements", str(el), "--steps", "4", "--warmup", "3", "--e2e-steps", "2",
             "--skip-cpu", "--skip-probe"])
    c = d["config"]
    assert "zs_shard_step_async" in c["api"]
    assert c["device_state_after_timed_steps"]["iterations"] == 3 + 4
    assert d["e2e"]["d2h_bytes_per_step"] == 64 and d["e2e"]["last_result"]["iterations"] == 3
    assert set(c["workloads"]) == set(bench.TABLE_WORKLOADS)
    for name, w in c["workloads"].items():
        wl = bench.synth.WORKLOADS[name]
        assert w["shard_len"] == el and w["n_ranks_simulated"] == wl.n
        for api in ("async", "async_oop", "sync"):
            a = w[api]
            # owned parameters: the 2^20 workload's shard holds fewer than el
            assert a["value"] == pytest.approx(w["owned_params"] / (a["ms_per_step"] * 1e-3),
                                               rel=1e-3)
            assert a["step_frac_of_peak"] > 0 and "sm_mhz" in a["clocks"]
            assert a["gpu_launches"] >= 100 * 2 and a["steps"] == 100
        assert w["async"]["device_state"]["iterations"] == 3 + 2 * 100   # two timed passes
        assert "update_oop" in w["async_oop"]["kernels"]
        # the same out-of-place step replayed from a CUDA graph: its GPU rate
        g = w["graph_oop"]
        assert g["value"] > 0 and g["step_frac_of_peak"] > 0 and g["gpu_launches"] >= 100 * 2
        # the uncaptured first call, whole replays of warm-up, two timed passes
        assert g["warmup_steps"] >= 3 and g["warmup_steps"] % g.get("steps_per_replay", 1) == 0
        assert g["device_state"]["iterations"] == 1 + g["warmup_steps"] + 2 * 100
