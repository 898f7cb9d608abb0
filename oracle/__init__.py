"""CPU oracle for the ZeRO shard step (ctypes wrapper over zs_oracle.c).

TEST INFRASTRUCTURE ONLY: imported by the tests, the smoke check and the
benchmark's CPU-baseline leg, never by the library.  The C source states the
pages and readings it follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SO = os.path.join(_HERE, "libzsoracle.so")
FP16, BF16 = 0, 1

_i64p = ctypes.POINTER(ctypes.c_int64)
_u64p = ctypes.POINTER(ctypes.c_uint64)
_f32p = ctypes.POINTER(ctypes.c_float)
_f64p = ctypes.POINTER(ctypes.c_double)
_u16p = ctypes.POINTER(ctypes.c_uint16)


class HParams(ctypes.Structure):
    _fields_ = [("lr", ctypes.c_double), ("beta1", ctypes.c_double), ("beta2", ctypes.c_double),
                ("eps", ctypes.c_double), ("weight_decay", ctypes.c_double)]


class Scaler(ctypes.Structure):
    _fields_ = [("scale", ctypes.c_double), ("min_scale", ctypes.c_double),
                ("window", ctypes.c_int32), ("clean_count", ctypes.c_int32),
                ("hysteresis", ctypes.c_int32), ("hyst_left", ctypes.c_int32),
                ("dynamic", ctypes.c_int32), ("consecutive", ctypes.c_int32)]


def make_hparams(lr, beta1, beta2, eps, weight_decay) -> HParams:
    """Hyper-parameters as the fp32 values the library receives."""
    f = lambda x: float(np.float32(x))  # noqa: E731
    return HParams(f(lr), f(beta1), f(beta2), f(eps), f(weight_decay))


def make_scaler(scale, min_scale=1.0, window=1000, hysteresis=1, dynamic=True,
                consecutive=False) -> Scaler:
    return Scaler(float(scale), float(min_scale), int(window), 0, int(hysteresis),
                  int(hysteresis), 1 if dynamic else 0, 1 if consecutive else 0)


def _stale(out, srcs):
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    return any(os.path.getmtime(s) > t for s in srcs)


def build(force: bool = False) -> str:
    srcs = [os.path.join(_HERE, "zs_oracle.c"), os.path.join(_HERE, "zs_oracle.h")]
    if force or _stale(SO, srcs):
        tmp = SO + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O1", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared",
                               "-o", tmp, srcs[0], "-lm"])
        os.replace(tmp, SO)
    return SO


_lib = None


def lib():
    global _lib
    if _lib is not None:
        return _lib
    L = ctypes.CDLL(build())
    L.zso_partition.argtypes = [ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, _i64p, _i64p]
    L.zso_shard_range.argtypes = [ctypes.c_int64, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32,
                                  _i64p, _i64p, _i64p]
    L.zso_state_bytes.argtypes = [ctypes.c_int64, ctypes.c_int64, ctypes.c_int32, _u64p]
    L.zso_half_to_double.argtypes = [ctypes.c_uint16, ctypes.c_int32]
    L.zso_half_to_double.restype = ctypes.c_double
    L.zso_f32_to_half.argtypes = [ctypes.c_float, ctypes.c_int32]
    L.zso_f32_to_half.restype = ctypes.c_uint16
    L.zso_half_to_double_array.argtypes = [_u16p, ctypes.c_int64, ctypes.c_int32, _f64p]
    L.zso_f32_to_half_array.argtypes = [_f32p, ctypes.c_int64, ctypes.c_int32, _u16p]
    PP = ctypes.POINTER(_u16p)
    L.zso_reduce_accumulate.argtypes = [PP, ctypes.c_int32, ctypes.c_int32, ctypes.c_int64, _f32p,
                                        ctypes.c_int32]
    L.zso_any_nonfinite.argtypes = [PP, ctypes.c_int32, ctypes.c_int32, ctypes.c_int64]
    L.zso_any_nonfinite.restype = ctypes.c_int32
    L.zso_any_nonfinite_f32.argtypes = [_f32p, ctypes.c_int64]
    L.zso_any_nonfinite_f32.restype = ctypes.c_int32
    L.zso_adamw_apply.argtypes = [_f32p, ctypes.c_int64, ctypes.c_double, _f32p, _f32p, _f32p,
                                  _u16p, ctypes.c_int32, ctypes.POINTER(HParams), ctypes.c_int64]
    L.zso_scaler_update.argtypes = [ctypes.POINTER(Scaler), ctypes.c_int32]
    L.zso_reduce_accumulate_half.argtypes = [PP, ctypes.c_int32, ctypes.c_int32, ctypes.c_int64,
                                             _u16p, ctypes.c_int32]
    L.zso_shard_step_halfacc.argtypes = [PP, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                         ctypes.c_int64, _u16p, _f32p, _f32p, _f32p, _u16p,
                                         ctypes.POINTER(HParams), _i64p, ctypes.POINTER(Scaler),
                                         ctypes.c_int32]
    L.zso_shard_step_halfacc.restype = ctypes.c_int32
    L.zso_lr_at.argtypes = [ctypes.c_int32, ctypes.c_double, ctypes.c_double, ctypes.c_int64,
                            ctypes.c_int64, ctypes.c_int64]
    L.zso_lr_at.restype = ctypes.c_double
    L.zso_grad_sumsq.argtypes = [_f32p, ctypes.c_int64, ctypes.c_double]
    L.zso_grad_sumsq.restype = ctypes.c_double
    L.zso_clip_coef.argtypes = [ctypes.c_double, ctypes.c_double]
    L.zso_clip_coef.restype = ctypes.c_double
    L.zso_adamw_apply_clipped.argtypes = [_f32p, ctypes.c_int64, ctypes.c_double, ctypes.c_double,
                                          _f32p, _f32p, _f32p, _u16p, ctypes.c_int32,
                                          ctypes.POINTER(HParams), ctypes.c_int64]
    L.zso_shard_step.argtypes = [PP, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                 ctypes.c_int64, _f32p, _f32p, _f32p, _f32p, _u16p,
                                 ctypes.POINTER(HParams), _i64p, ctypes.POINTER(Scaler),
                                 ctypes.c_int32]
    L.zso_shard_step.restype = ctypes.c_int32
    L.zso_shard_step_clipped.argtypes = L.zso_shard_step.argtypes + [ctypes.c_double, _f64p]
    L.zso_shard_step_clipped.restype = ctypes.c_int32
    _lib = L
    return L


def _p(a, t):
    return a.ctypes.data_as(t)


def _check_u16(a):
    assert a.dtype == np.uint16 and a.flags.c_contiguous
    return a


def _check_f32(a):
    assert a.dtype == np.float32 and a.flags.c_contiguous
    return a


def _ptr_array(slices):
    arr = (_u16p * len(slices))()
    for i, s in enumerate(slices):
        arr[i] = _p(_check_u16(s), _u16p)
    return arr


def partition(psi: int, n: int, align: int = 64):
    a, b = ctypes.c_int64(), ctypes.c_int64()
    if lib().zso_partition(psi, n, align, ctypes.byref(a), ctypes.byref(b)) != 0:
        raise ValueError("bad partition arguments")
    return a.value, b.value


def shard_range(psi: int, shard_len: int, n: int, rank: int):
    b, ve, pe = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()
    if lib().zso_shard_range(psi, shard_len, n, rank, ctypes.byref(b), ctypes.byref(ve),
                             ctypes.byref(pe)) != 0:
        raise ValueError("bad shard range arguments")
    return b.value, ve.value, pe.value


def state_bytes(psi: int, shard_len: int, stage: int) -> int:
    out = ctypes.c_uint64()
    if lib().zso_state_bytes(psi, shard_len, stage, ctypes.byref(out)) != 0:
        raise ValueError("bad stage")
    return out.value


def half_to_double(bits: np.ndarray, dtype: int) -> np.ndarray:
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    out = np.empty(bits.shape, dtype=np.float64)
    lib().zso_half_to_double_array(_p(bits, _u16p), bits.size, dtype, _p(out, _f64p))
    return out


def f32_to_half(x: np.ndarray, dtype: int) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint16)
    lib().zso_f32_to_half_array(_p(x, _f32p), x.size, dtype, _p(out, _u16p))
    return out


def reduce_accumulate(slices, dtype: int, acc: np.ndarray, first: bool):
    _check_f32(acc)
    for s in slices:
        assert s.shape[0] >= acc.shape[0]
    lib().zso_reduce_accumulate(_ptr_array(slices), len(slices), dtype, acc.shape[0],
                                _p(acc, _f32p), 1 if first else 0)


def any_nonfinite(slices, dtype: int, count: int) -> int:
    return int(lib().zso_any_nonfinite(_ptr_array(slices), len(slices), dtype, count))


def any_nonfinite_f32(x: np.ndarray) -> int:
    _check_f32(x)
    return int(lib().zso_any_nonfinite_f32(_p(x, _f32p), x.shape[0]))


def adamw_apply(acc, grad_div, master, m, v, half_out, dtype, hp: HParams, t: int):
    for a in (acc, master, m, v):
        _check_f32(a)
    _check_u16(half_out)
    lib().zso_adamw_apply(_p(acc, _f32p), acc.shape[0], float(grad_div), _p(master, _f32p),
                          _p(m, _f32p), _p(v, _f32p), _p(half_out, _u16p), dtype,
                          ctypes.byref(hp), t)


LR_CONSTANT, LR_WARMUP, LR_WARMUP_DECAY = 0, 1, 2


def lr_at(kind: int, min_lr: float, max_lr: float, warmup_steps: int, total_steps: int,
          t: int) -> float:
    return float(lib().zso_lr_at(kind, float(min_lr), float(max_lr), int(warmup_steps),
                                 int(total_steps), int(t)))


def grad_sumsq(acc: np.ndarray, grad_div: float) -> float:
    _check_f32(acc)
    return float(lib().zso_grad_sumsq(_p(acc, _f32p), acc.shape[0], float(grad_div)))


def clip_coef(sumsq_total: float, max_norm: float) -> float:
    return float(lib().zso_clip_coef(float(sumsq_total), float(max_norm)))


def adamw_apply_clipped(acc, grad_div, coef, master, m, v, half_out, dtype, hp: HParams, t: int):
    for a in (acc, master, m, v):
        _check_f32(a)
    _check_u16(half_out)
    lib().zso_adamw_apply_clipped(_p(acc, _f32p), acc.shape[0], float(grad_div), float(coef),
                                  _p(master, _f32p), _p(m, _f32p), _p(v, _f32p),
                                  _p(half_out, _u16p), dtype, ctypes.byref(hp), t)


def scaler_update(sc: Scaler, overflow: int):
    lib().zso_scaler_update(ctypes.byref(sc), int(overflow))


@dataclass
class ShardState:
    """fp32 master / m / v and the half copy of one shard (or of any range)."""
    master: np.ndarray
    m: np.ndarray
    v: np.ndarray
    half: np.ndarray

    @classmethod
    def from_master(cls, master: np.ndarray, dtype: int):
        master = np.array(master, dtype=np.float32)
        return cls(master, np.zeros_like(master), np.zeros_like(master),
                   f32_to_half(master, dtype))

    def copy(self):
        return ShardState(self.master.copy(), self.m.copy(), self.v.copy(), self.half.copy())


def shard_step(grads, dtype: int, state: ShardState, hp: HParams, t: int, sc: Scaler,
               extra_overflow: int = 0, max_norm: float = 0.0, return_norm: bool = False):
    """One step of one owned-shard view.  grads[k][r] = rank r's slice in
    micro-step k.  Returns (overflow, new t, acc) (and the gradient norm when
    return_norm)."""
    g = len(grads)
    n = len(grads[0])
    count = state.master.shape[0]
    flat = [s for micro in grads for s in micro]
    acc = np.zeros(count, dtype=np.float32)
    tt = ctypes.c_int64(t)
    norm = ctypes.c_double(0.0)
    ovf = lib().zso_shard_step_clipped(_ptr_array(flat), g, n, dtype, count, _p(acc, _f32p),
                                       _p(state.master, _f32p), _p(state.m, _f32p),
                                       _p(state.v, _f32p), _p(state.half, _u16p),
                                       ctypes.byref(hp), ctypes.byref(tt), ctypes.byref(sc),
                                       int(extra_overflow), float(max_norm), ctypes.byref(norm))
    if return_norm:
        return int(ovf), tt.value, acc, norm.value
    return int(ovf), tt.value, acc


def reduce_accumulate_half(slices, dtype: int, acc_half: np.ndarray, first: bool):
    _check_u16(acc_half)
    lib().zso_reduce_accumulate_half(_ptr_array(slices), len(slices), dtype, acc_half.shape[0],
                                     _p(acc_half, _u16p), 1 if first else 0)


def shard_step_halfacc(grads, dtype: int, state: ShardState, hp: HParams, t: int, sc: Scaler,
                       extra_overflow: int = 0):
    """shard_step with the half-precision accumulator.  Returns (overflow, t, acc_half)."""
    g = len(grads)
    n = len(grads[0])
    count = state.master.shape[0]
    flat = [s for micro in grads for s in micro]
    acc = np.zeros(count, dtype=np.uint16)
    tt = ctypes.c_int64(t)
    ovf = lib().zso_shard_step_halfacc(_ptr_array(flat), g, n, dtype, count, _p(acc, _u16p),
                                       _p(state.master, _f32p), _p(state.m, _f32p),
                                       _p(state.v, _f32p), _p(state.half, _u16p),
                                       ctypes.byref(hp), ctypes.byref(tt), ctypes.byref(sc),
                                       int(extra_overflow))
    return int(ovf), tt.value, acc


def multi_shard_step(grads_per_shard, dtype: int, states, hp: HParams, t: int, sc: Scaler,
                     max_norm: float = 0.0):
    """One step of all N ranks' shards with a global overflow flag (every
    rank skips together): reduce each shard, OR the flags, then update every
    shard with the same step count and scale, then update the scale once.
    grads_per_shard[q][k][r] = rank r's slice of shard q in micro-step k."""
    flag = 0
    accs = []
    for q, grads in enumerate(grads_per_shard):
        count = states[q].master.shape[0]
        acc = np.zeros(count, dtype=np.float32)
        for k, micro in enumerate(grads):
            reduce_accumulate(micro, dtype, acc, first=(k == 0))
            flag |= any_nonfinite(micro, dtype, count)
        flag |= any_nonfinite_f32(acc)
        accs.append(acc)
    if not flag:
        t += 1
        n = len(grads_per_shard[0][0])
        g = len(grads_per_shard[0])
        div = float(n) * g * sc.scale
        coef = 1.0
        if max_norm > 0:
            coef = clip_coef(sum(grad_sumsq(a, div) for a in accs), max_norm)
        for q, st in enumerate(states):
            adamw_apply_clipped(accs[q], div, coef, st.master, st.m, st.v, st.half, dtype, hp, t)
    scaler_update(sc, flag)
    return flag, t, accs
