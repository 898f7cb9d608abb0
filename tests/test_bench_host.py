"""Host-side logic of the benchmark: the algorithmic byte model against the
workload table, and the rule that recorded ncu traffic is only reported for
the workload and kernel sources it was captured with.  No GPU."""
import json
import os

import pytest

import bench
import synth


def test_algorithmic_bytes_per_step():
    # 2·N·G (every gradient once) + 8·(G-1) (fp32 accumulator carried) + 26 (master/m/v r/w, half)
    want = {"flat-1m-n2": 30, "gpt2-small-n8": 114, "decoder-1.3b-n16": 98,
            "llama7b-zero3-n64": 154, "llama7b-n1": 98}
    for name, b in want.items():
        wl = synth.WORKLOADS[name]
        assert bench.alg_bytes_per_elem_step(wl.n, wl.g) == b
    # the half accumulator carries 2-byte values
    assert bench.alg_bytes_per_elem_step(1, 8, acc_bytes=2) == 2 * 8 + 4 * 7 + 26


def test_kernel_bytes_add_up_to_the_step():
    # materialise path (N >= 4): first + (G-2) later accumulates + last accumulate + update
    for n, g in ((8, 4), (16, 2), (64, 1)):
        ks = [bench.kernel_alg_bytes("reduce", n, first=(k == 0)) for k in range(g)]
        ks.append(bench.kernel_alg_bytes("apply", n))
        # materialising the last micro-step writes acc (4) and the update reads it back (4)
        assert sum(ks) == bench.alg_bytes_per_elem_step(n, g) + 8
    # re-read path (N < 4): the flag pass re-reads the last slices
    n, g = 1, 8
    ks = [bench.kernel_alg_bytes("reduce", n, first=(k == 0)) for k in range(g - 1)]
    ks += [bench.kernel_alg_bytes("check", n), bench.kernel_alg_bytes("apply_recompute", n,
                                                                        with_acc=True)]
    assert sum(ks) == bench.alg_bytes_per_elem_step(n, g) + 2 * n


def test_recorded_traffic_requires_matching_sources(tmp_path, monkeypatch):
    rec = json.load(open(os.path.join(bench.ROOT, "profiles", "traffic.json")))
    assert set(rec["bytes_per_elem"]) >= {"reduce", "check", "apply_recompute", "reduce_first"}
    # reads measured by ncu never exceed the algorithmic bytes (no re-reads)
    for k, alg in rec["algorithmic_bytes_per_elem"].items():
        assert rec["bytes_per_elem"][k] <= alg + 0.01
    assert bench.recorded_traffic("gpt2-small-n8", "reduce", 1e6) is None
    # a copy of the repo whose record was taken on its own sources
    fake = tmp_path / "repo"
    (fake / "profiles").mkdir(parents=True)
    for rel in rec["sources_code_sha256"]:
        p = fake / rel
        p.parent.mkdir(parents=True, exist_ok=True)
        p.write_text(open(os.path.join(bench.ROOT, rel)).read())
    rec = dict(rec, sources_code_sha256={rel: bench.code_digest(str(fake / rel))
                                         for rel in rec["sources_code_sha256"]})
    (fake / "profiles" / "traffic.json").write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "ROOT", str(fake))
    per = rec["bytes_per_elem"]["reduce"]
    assert bench.recorded_traffic(rec["workload"], "reduce", 1e6) == per * 1e6
    # comments and blank lines do not change the code the counters describe
    for rel in rec["sources_code_sha256"]:
        src = (fake / rel).read_text()
        (fake / rel).write_text("// a comment\n\n" + src.replace("\n", "  \n") + "/* more */\n")
    assert bench.recorded_traffic(rec["workload"], "reduce", 1e6) == per * 1e6
    # a change of the code voids the record
    for rel in rec["sources_code_sha256"]:
        (fake / rel).write_text((fake / rel).read_text() + "int changed;\n")
    assert bench.recorded_traffic(rec["workload"], "reduce", 1e6) is None


def test_launch_plans():
    kinds = lambda plan: [k for k, _ in plan]
    # Llama-7B, one rank, 8 micro-steps: the re-read form
    p = bench.step_launch_plan(1, 8, "fp16")
    assert kinds(p) == ["reduce_first"] + ["reduce"] * 6 + ["check", "apply_recompute"]
    assert sum(b for _, b in p) == bench.alg_bytes_per_elem_step(1, 8) + 2
    # the split step launches the same kernels; with clipping the fused form folds the
    # norm into the flag pass (which then reads acc), the split form adds a norm pass
    assert bench.step_launch_plan(1, 8, "fp16", split=True) == p
    fused = dict(bench.step_launch_plan(1, 8, "fp16", clip=1.0))
    split = dict(bench.step_launch_plan(1, 8, "fp16", clip=1.0, split=True))
    assert fused["check"] == 6 and split["check"] == 2 and split["sumsq"] == 6
    # 64 ranks, one micro-step: materialise, then update from acc
    p = bench.step_launch_plan(64, 1, "fp16")
    assert kinds(p) == ["reduce_first", "apply"]
    assert kinds(bench.step_launch_plan(64, 1, "fp16", clip=1.0, split=True)) == \
        ["reduce_first", "sumsq", "apply"]
    # bf16 re-read flag pass reads acc as well
    assert dict(bench.step_launch_plan(2, 3, "bf16"))["check"] == 2 * 2 + 4
    # half accumulator
    p = bench.step_launch_plan(1, 8, "fp16", acc_kind="half")
    assert sum(b for _, b in p) == bench.alg_bytes_per_elem_step(1, 8, acc_bytes=2) + 4


def _bench_line(args, env=None):
    import subprocess
    import sys
    out = subprocess.run([sys.executable, os.path.join(bench.ROOT, "bench.py")] + args,
                         capture_output=True, text=True, timeout=600,
                         env=dict(os.environ, **(env or {})), cwd=bench.ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    return json.loads(lines[-1]) if lines else None


def test_reference_arm_line():
    """--impl reference times the oracle on the host cores and prints the
    contract's line, with an e2e object that moves no bytes."""
    d = _bench_line(["--impl", "reference", "--steps", "1", "--warmup", "1"])
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC
    assert d["value"] > 0 and d["unit"] == "params/s" and d["higher_is_better"] is True
    assert d["config"]["workload"] == bench.DEFAULT_WORKLOAD
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["sample"] and cb["value"] == d["value"]
    e = d["e2e"]
    assert e["value"] == d["value"] and e["h2d_bytes_per_step"] == 0 and e["d2h_bytes_per_step"] == 0


def test_reference_arm_other_ranks_print_nothing():
    d = _bench_line(["--impl", "reference", "--steps", "1", "--warmup", "1"],
                    env={"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"})
    assert d is None


def test_out_of_place_plan_moves_exactly_the_algorithmic_bytes():
    """The out-of-place step writes the state once and reads every gradient
    once: its launches move 2·N·G + 8·(G-1) + 26 bytes per element, nothing more."""
    for name in ("flat-1m-n2", "gpt2-small-n8", "decoder-1.3b-n16", "llama7b-zero3-n64",
                 "llama7b-n1"):
        wl = synth.WORKLOADS[name]
        plan = bench.step_launch_plan(wl.n, wl.g, wl.dtype, oop=True)
        assert [k for k, _ in plan][-1] == "update_oop"
        assert sum(b for _, b in plan) == bench.alg_bytes_per_elem_step(wl.n, wl.g)


def test_half_accumulator_oop_plan_moves_exactly_the_algorithmic_bytes():
    for name in ("gpt2-small-n8", "decoder-1.3b-n16", "llama7b-n1"):
        wl = synth.WORKLOADS[name]
        plan = bench.step_launch_plan(wl.n, wl.g, wl.dtype, acc_kind="half", oop=True)
        assert [k for k, _ in plan][-1] == "update_oop"
        assert sum(b for _, b in plan) == bench.alg_bytes_per_elem_step(wl.n, wl.g, acc_bytes=2)


def test_fused_plan_moves_exactly_the_algorithmic_bytes():
    """The fused step (shards that fit one co-resident grid): the carried
    micro-steps, then one kernel; nothing is read twice or written twice."""
    for name in ("flat-1m-n2", "gpt2-small-n8", "decoder-1.3b-n16"):
        wl = synth.WORKLOADS[name]
        plan = bench.step_launch_plan(wl.n, wl.g, wl.dtype, fused=True)
        assert [k for k, _ in plan] == ["reduce_first"] * (wl.g > 1) + ["reduce"] * max(
            0, wl.g - 2) + ["fused"]
        assert sum(b for _, b in plan) == bench.alg_bytes_per_elem_step(wl.n, wl.g)
        half = bench.step_launch_plan(wl.n, wl.g, wl.dtype, acc_kind="half", fused=True)
        assert [k for k, _ in half] == [k for k, _ in plan]
        assert sum(b for _, b in half) == bench.alg_bytes_per_elem_step(wl.n, wl.g, acc_bytes=2)


def test_bench_line_names_the_entry_points_each_api_calls():
    """The half-accumulator forms name the halfacc entry points (and only they
    do); clipping names the clipped forms; the split step is the same either way."""
    for api in ("async", "async_oop", "sync"):
        assert "halfacc" in bench.api_desc(api, "half", 0.0, api == "sync")
    assert bench.api_desc("sync", "half", 0.0, True).startswith(
        "zs_grad_accum_halfacc + zs_shard_step_halfacc_oop")
    assert bench.api_desc("sync", "half", 0.0, False).endswith("zs_shard_step_halfacc")
    for api in bench.API_DESC:
        assert "halfacc" not in bench.api_desc(api, "fp32", 0.0, False)
        assert bench.api_desc(api, "fp32", 0.0, False) == bench.API_DESC[api]
    assert bench.api_desc("sync", "fp32", 1.0, False) == "zs_grad_accum + zs_shard_step_clipped"
    assert "zs_shard_step_async_clipped" in bench.api_desc("async", "fp32", 1.0, False)
    assert "zs_shard_step_async_clipped" in bench.api_desc("graph", "fp32", 1.0, False)
    for api in ("async_oop", "graph_oop"):     # no clipped out-of-place entry point
        with pytest.raises(ValueError):
            bench.api_desc(api, "fp32", 1.0, False)
    assert bench.api_desc("split", "fp32", 1.0, False) == bench.API_DESC["split"]


def test_graph_replays_several_steps_only_where_a_step_is_short():
    """Steps of ~2 us (the 2^20-parameter workload) go 50 to a replay; steps of
    hundreds of microseconds or more go one to a replay; the count always
    divides the timed steps."""
    small = 524288 * 30
    assert bench.graph_steps_per_replay(small, 2000) == 50
    assert bench.graph_steps_per_replay(small, 3) == 3
    assert bench.graph_steps_per_replay(small, 98) == 49
    for sb in (15555008 * 114, 82232704 * 98, 6738415616 * 98):
        assert bench.graph_steps_per_replay(sb, 20) == 1
    for steps in (1, 7, 100, 2000):
        for sb in (1e3, small, 4e8, 1e12):
            r = bench.graph_steps_per_replay(sb, steps)
            assert 1 <= r <= 50 and steps % r == 0
