"""In-tree nvcc build of libzeroshard.so (importable without loading the library)."""
from __future__ import annotations

import os
import subprocess

_HERE = os.path.dirname(os.path.abspath(__file__))
_ROOT = os.path.dirname(_HERE)
# ZEROSHARD_LIB points the binding at another build of the same library.
LIB_PATH = os.environ.get("ZEROSHARD_LIB", os.path.join(_HERE, "libzeroshard.so"))
HEADER = os.path.join(_ROOT, "include", "zeroshard.h")
SOURCES = [os.path.join(_HERE, "csrc", "zeroshard.cu"), os.path.join(_HERE, "csrc", "zs_kernels.cuh"),
           HEADER]


def build_cmd(out: str = LIB_PATH):
    return ["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-lineinfo",
            "-std=c++17", "-I", os.path.join(_ROOT, "include"), "-Xcompiler", "-fPIC", "-shared",
            "-o", out, SOURCES[0]]


def stale() -> bool:
    return not os.path.exists(LIB_PATH) or any(
        os.path.getmtime(s) > os.path.getmtime(LIB_PATH) for s in SOURCES)


def build(force: bool = False) -> str:
    """Compile libzeroshard.so in-tree with nvcc for sm_103a."""
    if force or stale():
        tmp = LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(build_cmd(tmp))
        os.replace(tmp, LIB_PATH)
    return LIB_PATH
