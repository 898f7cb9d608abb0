"""Seeded synthetic inputs shared by the oracle harness and the CUDA harness.

Host side: libzssynth_host.so (gcc) returns fp32 values at arbitrary flat
indices; they are converted to fp16 with numpy and to bf16 with torch (both
round to nearest even).  Device side: libzssynth_dev.so fills HBM buffers with
the same values, converted by CUDA's RNE intrinsics.  Nothing here performs a
step of the optimizer.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

from .configs import ALIGN_ELEMS, WORKLOADS, Injection, Workload  # noqa: F401

_HERE = os.path.dirname(os.path.abspath(__file__))
HOST_SO = os.path.join(_HERE, "libzssynth_host.so")
DEV_SO = os.path.join(_HERE, "libzssynth_dev.so")
MAX_SEG = 4

FP16_POS_INF = 0x7C00
FP16_NAN = 0x7E00
BF16_POS_INF = 0x7F80
BF16_NAN = 0x7FC0


class GradRecipe(ctypes.Structure):
    _fields_ = [
        ("seed", ctypes.c_uint64),
        ("stream", ctypes.c_uint64),
        ("c_normal", ctypes.c_float),
        ("c_tail", ctypes.c_float),
        ("tail_threshold", ctypes.c_uint32),
        ("n_seg", ctypes.c_int32),
        ("seg_begin", ctypes.c_int64 * MAX_SEG),
        ("seg_end", ctypes.c_int64 * MAX_SEG),
        ("seg_c", ctypes.c_float * MAX_SEG),
        ("pad_", ctypes.c_int32),
    ]


def _stale(out: str, srcs) -> bool:
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    return any(os.path.getmtime(s) > t for s in srcs)


def build_host(force: bool = False) -> str:
    srcs = [os.path.join(_HERE, "synth_host.c"), os.path.join(_HERE, "zs_synth.h")]
    if force or _stale(HOST_SO, srcs):
        tmp = HOST_SO + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared",
                               "-o", tmp, srcs[0], "-lm"])
        os.replace(tmp, HOST_SO)
    return HOST_SO


def dev_build_cmd(out: str = DEV_SO):
    return ["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-lineinfo",
            "-Xcompiler", "-fPIC", "-shared", "-o", out, os.path.join(_HERE, "synth_dev.cu")]


_host = None
_dev = None


def host_lib():
    global _host
    if _host is None:
        lib = ctypes.CDLL(build_host())
        i64p = ctypes.POINTER(ctypes.c_int64)
        f32p = ctypes.POINTER(ctypes.c_float)
        lib.zs_synth_host_grad_values.argtypes = [
            i64p, ctypes.c_int64, ctypes.c_int64, ctypes.c_uint32, ctypes.c_uint32,
            ctypes.c_uint32, ctypes.POINTER(GradRecipe), f32p]
        lib.zs_synth_host_master_values.argtypes = [
            i64p, ctypes.c_int64, ctypes.c_int64, ctypes.c_uint64, ctypes.c_uint64,
            ctypes.c_float, f32p]
        u64p = ctypes.POINTER(ctypes.c_uint64)
        lib.zs_synth_host_philox.argtypes = [u64p, u64p, u64p]
        _host = lib
    return _host


def dev_lib():
    global _dev
    if _dev is None:
        if not os.path.exists(DEV_SO):
            raise RuntimeError(f"{DEV_SO} is not built: run __graft_entry__.build()")
        lib = ctypes.CDLL(DEV_SO)
        lib.zs_synth_dev_fill_grads.argtypes = [
            ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
            ctypes.c_uint32, ctypes.c_uint32, ctypes.c_uint32, ctypes.POINTER(GradRecipe),
            ctypes.c_void_p]
        lib.zs_synth_dev_fill_grads.restype = ctypes.c_int
        lib.zs_synth_dev_fill_master.argtypes = [
            ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_uint64,
            ctypes.c_uint64, ctypes.c_float, ctypes.c_void_p]
        lib.zs_synth_dev_fill_master.restype = ctypes.c_int
        _dev = lib
    return _dev


def philox(ctr, key):
    lib = host_lib()
    c = (ctypes.c_uint64 * 4)(*[int(x) for x in ctr])
    k = (ctypes.c_uint64 * 2)(*[int(x) for x in key])
    o = (ctypes.c_uint64 * 4)()
    lib.zs_synth_host_philox(c, k, o)
    return [int(x) for x in o]


def grad_recipe(wl: Workload, scale: float) -> GradRecipe:
    r = GradRecipe()
    r.seed = wl.seed
    r.stream = wl.stream
    r.c_normal = float(np.float32(wl.sigma * scale / 131072.0))
    r.c_tail = float(np.float32(wl.sigma * scale))
    r.tail_threshold = int(round(wl.tail_fraction * 2.0 ** 32)) if wl.tail_fraction > 0 else 0
    segs = []
    if wl.low_sigma_tensors:
        ranges = {name: (b, e) for name, b, e in wl.tensor_ranges()}
        for name, sig in wl.low_sigma_tensors:
            b, e = ranges[name]
            segs.append((b, e, float(np.float32(sig * scale / 131072.0))))
    if len(segs) > MAX_SEG:
        raise ValueError("too many special-sigma segments")
    r.n_seg = len(segs)
    for k, (b, e, c) in enumerate(segs):
        r.seg_begin[k] = b
        r.seg_end[k] = e
        r.seg_c[k] = c
    return r


def master_c(wl: Workload) -> float:
    return float(np.float32(wl.master_sigma / 131072.0))


def to_half_bits(vals: np.ndarray, dtype: str) -> np.ndarray:
    vals = np.ascontiguousarray(vals, dtype=np.float32)
    if dtype == "fp16":
        return vals.astype(np.float16).view(np.uint16)
    import torch
    return torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def injection_bits(kind: str, dtype: str) -> int:
    if dtype == "fp16":
        return FP16_POS_INF if kind == "inf" else FP16_NAN
    return BF16_POS_INF if kind == "inf" else BF16_NAN


def host_grad_bits(wl: Workload, idx, step: int, micro: int, rank: int, scale: float,
                   inject: bool = True) -> np.ndarray:
    """Half bit patterns of rank `rank`'s gradient at flat indices `idx`."""
    idx = np.ascontiguousarray(idx, dtype=np.int64)
    out = np.empty(idx.shape[0], dtype=np.float32)
    rec = grad_recipe(wl, scale)
    host_lib().zs_synth_host_grad_values(
        idx.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), idx.shape[0], wl.psi, step, micro,
        rank, ctypes.byref(rec), out.ctypes.data_as(ctypes.POINTER(ctypes.c_float)))
    bits = to_half_bits(out, wl.dtype)
    if inject:
        for j in wl.injections_at(step):
            if j.micro == micro and j.rank == rank:
                hit = np.nonzero(idx == j.index)[0]
                bits[hit] = injection_bits(j.kind, wl.dtype)
    return bits


def host_master(wl: Workload, idx) -> np.ndarray:
    idx = np.ascontiguousarray(idx, dtype=np.int64)
    out = np.empty(idx.shape[0], dtype=np.float32)
    host_lib().zs_synth_host_master_values(
        idx.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), idx.shape[0], wl.psi, wl.seed,
        wl.stream, master_c(wl), out.ctypes.data_as(ctypes.POINTER(ctypes.c_float)))
    return out


def dev_fill_grads(ptr: int, count: int, global_begin: int, wl: Workload, step: int, micro: int,
                   rank: int, scale: float, stream: int = 0, inject: bool = True,
                   inject_writer=None):
    """Fill `count` half elements at device address `ptr` with rank `rank`'s
    gradient over flat indices [global_begin, global_begin + count).
    `inject_writer(offset, bits)` writes one 16-bit pattern into the buffer
    (the caller supplies it, e.g. a torch indexed assignment)."""
    rec = grad_recipe(wl, scale)
    rc = dev_lib().zs_synth_dev_fill_grads(ptr, wl.dtype_code, count, global_begin, wl.psi, step,
                                           micro, rank, ctypes.byref(rec), stream)
    if rc != 0:
        raise RuntimeError(f"zs_synth_dev_fill_grads failed: {rc}")
    if inject:
        for j in wl.injections_at(step):
            if j.micro == micro and j.rank == rank and global_begin <= j.index < global_begin + count:
                inject_writer(j.index - global_begin, injection_bits(j.kind, wl.dtype))


def dev_fill_master(ptr: int, count: int, global_begin: int, wl: Workload, stream: int = 0):
    rc = dev_lib().zs_synth_dev_fill_master(ptr, count, global_begin, wl.psi, wl.seed, wl.stream,
                                            master_c(wl), stream)
    if rc != 0:
        raise RuntimeError(f"zs_synth_dev_fill_master failed: {rc}")
