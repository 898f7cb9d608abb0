"""The C ABI from plain C: tests/c_abi_main.c links libzeroshard.so and the
CUDA runtime only (no Python, no torch), runs one step with cudaMalloc'ed
buffers (in place through the fused step or the multi-kernel path, out of
place with the caller swapping to the written set, or the two-phase
out-of-place update over two ranges), and its output is compared with the
oracle."""
import os
import subprocess

import numpy as np
import pytest

import oracle

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def build_c_caller(tmp_path):
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    pkg = os.path.join(ROOT, "zero_mixed_precision_shard_gb300")
    exe = str(tmp_path / "c_abi_main")
    subprocess.check_call([
        "gcc", "-O2", "-std=c11", "-o", exe, os.path.join(ROOT, "tests", "c_abi_main.c"),
        "-I", os.path.join(ROOT, "include"), "-I", os.path.join(cuda, "include"),
        "-L", pkg, "-lzeroshard", "-L", os.path.join(cuda, "lib64"), "-lcudart",
        f"-Wl,-rpath,{pkg}", f"-Wl,-rpath,{os.path.join(cuda, 'lib64')}"])
    return exe


@pytest.mark.parametrize("form", ["in_place", "oop", "multi", "twophase"])
def test_plain_c_caller_matches_oracle(tmp_path, form):
    exe = build_c_caller(tmp_path)
    rng = np.random.default_rng(77)
    count, n, g, scale = 50_003, 3, 2, 1024.0
    hp = (1e-4, 0.9, 0.999, 1e-8, 0.01)
    grads = (rng.standard_normal((g, n, count)) * 1e-3 * scale).astype(np.float16).view(np.uint16)
    master0 = (rng.standard_normal(count) * 0.02).astype(np.float32)
    inp = tmp_path / "in.bin"
    with open(inp, "wb") as fh:
        fh.write(np.array([count, n, g], np.int64).tobytes())
        fh.write(np.array([scale, *hp], np.float32).tobytes())
        fh.write(np.ascontiguousarray(grads).tobytes())
        fh.write(master0.tobytes())
    out = tmp_path / "out.bin"
    subprocess.check_call([exe, str(inp), str(out)] + ([] if form == "in_place" else [form]))
    raw = open(out, "rb").read()
    ovf = np.frombuffer(raw[:4], np.int32)[0]
    new_scale = np.frombuffer(raw[4:8], np.float32)[0]
    off = 8
    got = {}
    for k in ("master", "m", "v"):
        got[k] = np.frombuffer(raw[off:off + 4 * count], np.float32)
        off += 4 * count
    got["half"] = np.frombuffer(raw[off:off + 2 * count], np.uint16)

    st = oracle.ShardState.from_master(master0, oracle.FP16)
    sc = oracle.make_scaler(scale, 1.0, 1000, 1, True)
    ovf_o, t, _ = oracle.shard_step([[np.ascontiguousarray(grads[k, r]) for r in range(n)]
                                     for k in range(g)], oracle.FP16, st,
                                    oracle.make_hparams(*hp), 0, sc)
    assert ovf == ovf_o == 0 and new_scale == sc.scale and t == 1
    for k in ("master", "m", "v"):
        want = getattr(st, k).astype(np.float64)
        assert np.all(np.abs(got[k] - want) <= 1e-6 * np.abs(want) + 1e-9), k
    h = got["half"].astype(np.int32)
    w = st.half.astype(np.int32)
    assert np.abs(np.where(h & 0x8000, -(h & 0x7FFF), h) - np.where(w & 0x8000, -(w & 0x7FFF), w)).max() <= 1
