"""The benchmark's multi-GPU path, launched as a multi-GPU run is (torchrun,
one process per rank), with two ranks sharing the one GPU over a gloo process
group: every exchange of the path (the overflow flag's MAX, the clipping
norm's SUM, the timing and totals) runs, no kernel waits on another rank, and
the one JSON line reports the whole job."""
import json
import os
import socket
import subprocess
import sys

import pytest

import bench

pytestmark = pytest.mark.gpu


def free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def torchrun(args, n=2):
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={n}",
           "--master-addr=127.0.0.1", f"--master-port={free_port()}",
           os.path.join(bench.ROOT, "bench.py"), "--gpus", str(n), "--dist-backend", "gloo"] + args
    out = subprocess.run(cmd, capture_output=True, text=True, timeout=900, cwd=bench.ROOT)
    assert out.returncode == 0, out.stderr[-3000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, out.stdout[-2000:]      # rank 0 alone prints
    return json.loads(lines[0])


@pytest.mark.parametrize("workload,elements,extra", [("llama7b-n1", 1 << 22, []),
                                                     ("gpt2-small-n8", 1 << 20, []),
                                                     ("llama7b-n1", 1 << 22, ["--clip", "1.0"])])
def test_two_ranks_on_one_gpu(workload, elements, extra):
    d = torchrun(["--workload", workload, "--elements", str(elements), "--steps", "3",
                  "--warmup", "3", "--e2e-steps", "1", "--skip-cpu", "--skip-probe"] + extra)
    assert d["n_gpus"] == 2 and d["scaling"] == "weak"
    assert d["config"]["parallelism"].startswith("replicas + overflow-flag all-reduce")
    if extra:
        assert d["config"]["parallelism"].endswith("norm all-reduce")
    assert "split at the flag" in d["config"]["api"]
    # whole job: both ranks' elements over the slowest rank's step
    assert d["value"] == pytest.approx(2 * elements / (d["ms_per_step"] * 1e-3), rel=1e-6)
    wl = bench.synth.WORKLOADS[workload]
    assert d["gpu_launches"] >= 2 * 3 * (wl.g + 1)
    e = d["e2e"]
    assert e["h2d_bytes_per_step"] == 2 * wl.g * wl.n * elements * 2 and e["value"] > 0
    assert d["cpu_baseline"] is None                 # rank 0 at N = 1 only
