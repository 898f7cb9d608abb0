"""The C-ABI library: builds, loads without a GPU, exports every symbol the
header declares, and its host-only calls (partition, shard ranges, memory
accounting, scaler init, argument checks) agree with the oracle.  No kernel
is launched here."""
import ctypes
import os
import re
import subprocess

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def zs():
    import zero_mixed_precision_shard_gb300 as pkg
    pkg_lib = pkg.build()
    assert os.path.exists(pkg_lib)
    return pkg


def declared_functions():
    text = open(os.path.join(ROOT, "include", "zeroshard.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"\b(zs_[a-z_0-9]+)\s*\(", text)
    return sorted(set(names))


def test_header_declares_the_path():
    names = declared_functions()
    for must in ("zs_init_partition", "zs_grad_accum", "zs_shard_step", "zs_reduce_check",
                 "zs_apply", "zs_scaler_update", "zs_copy_peak", "zs_ctx_create"):
        assert must in names


def test_every_declared_symbol_is_exported(zs):
    names = declared_functions()
    lib = ctypes.CDLL(zs.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n
    out = subprocess.run(["nm", "-D", "--defined-only", zs.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\sT\s(zs_\w+)", out))
    assert set(names) <= exported


def test_library_has_no_torch_dependency(zs):
    out = subprocess.run(["ldd", zs.LIB_PATH], capture_output=True, text=True).stdout
    assert "torch" not in out and "libc10" not in out


@pytest.mark.parametrize("psi,n,align", [(0, 1, 64), (1, 1, 64), (1000, 3, 64), (12345, 7, 8),
                                         (1 << 20, 2, 64), (124_439_808, 8, 64),
                                         (1_315_723_264, 16, 64), (6_738_415_616, 64, 64),
                                         (6_738_415_616, 1, 64), (99, 256, 1)])
def test_partition_matches_oracle(zs, psi, n, align):
    p = zs.zs_init_partition(psi, n, align)
    assert (p.psi_pad, p.shard_len) == oracle.partition(psi, n, align)
    for r in sorted({0, n // 2, n - 1}):
        assert zs.zs_shard_range(p, r) == oracle.shard_range(psi, p.shard_len, n, r)
    for stage in range(4):
        assert zs.zs_model_state_bytes(p, stage) == oracle.state_bytes(psi, p.shard_len, stage)


def test_host_argument_errors(zs):
    for bad in ((-1, 2, 64), (10, 0, 64), (10, 257, 64), (10, 2, 0)):
        with pytest.raises(zs.ZsError):
            zs.zs_init_partition(*bad)
    p = zs.zs_init_partition(100, 4)
    with pytest.raises(zs.ZsError):
        zs.zs_shard_range(p, 4)
    with pytest.raises(zs.ZsError):
        zs.zs_model_state_bytes(p, 4)
    with pytest.raises(zs.ZsError):
        zs.zs_scaler_init(0.0)
    s = zs.zs_scaler_init(65536.0, 1.0, 1000, 2, True)
    assert (s.scale, s.hyst_left, s.clean_count, s.dynamic) == (65536.0, 2, 0, 1)


def test_null_context_is_rejected(zs):
    lib = zs.lib
    assert lib.zs_grad_accum(None, None, 1, 0, 8, None, 1, None) == zs.ZS_ERR_ARG
    assert lib.zs_ctx_destroy(None) == zs.ZS_ERR_ARG
    assert lib.zs_last_error(None) == b"null context"
