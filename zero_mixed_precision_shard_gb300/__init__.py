"""Python binding of libzeroshard (the C ABI in include/zeroshard.h).

Argument marshalling only: every call goes to the CUDA library, whose
kernels do all of the work.  Tensors are torch CUDA tensors (or raw device
addresses as ints); streams are torch streams, raw handles, or None for the
current torch stream.  Importing this module fails loudly if the library has
not been built (see build()); there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

from ._build import HEADER, LIB_PATH, SOURCES, build, build_cmd  # noqa: F401,E402

ZS_OK, ZS_ERR_ARG, ZS_ERR_ALIGN, ZS_ERR_DTYPE, ZS_ERR_CUDA, ZS_ERR_TIMEOUT = 0, -1, -2, -3, -4, -5
ZS_ERR_LIMIT = -6
ZS_NOALLOC_MAX_COUNT = 16384 * 16384
ZS_FP16, ZS_BF16 = 0, 1
ZS_MAX_RANKS = 256
ZS_DEFAULT_ALIGN = 64
(ZS_KERNEL_REDUCE, ZS_KERNEL_CHECK, ZS_KERNEL_APPLY, ZS_KERNEL_APPLY_RECOMPUTE, ZS_KERNEL_SCALER,
 ZS_KERNEL_COPY, ZS_KERNEL_SUMSQ, ZS_KERNEL_REDUCE_FIRST, ZS_KERNEL_UPDATE_OOP,
 ZS_KERNEL_FUSED) = range(10)
KERNEL_NAMES = ["reduce", "check", "apply", "apply_recompute", "scaler", "copy", "sumsq",
                "reduce_first", "update_oop", "fused"]
ZS_FUSED_OFF, ZS_FUSED_ON, ZS_FUSED_TEST_TIMEOUT = 0, 1, 2
_STATUS = {0: "ZS_OK", -1: "ZS_ERR_ARG", -2: "ZS_ERR_ALIGN", -3: "ZS_ERR_DTYPE", -4: "ZS_ERR_CUDA",
           -5: "ZS_ERR_TIMEOUT", -6: "ZS_ERR_LIMIT"}


class ZsError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{_STATUS.get(status, status)}: {msg}")
        self.status = status


class zs_partition(ctypes.Structure):
    _fields_ = [("psi", ctypes.c_int64), ("psi_pad", ctypes.c_int64),
                ("shard_len", ctypes.c_int64), ("n", ctypes.c_int32), ("align", ctypes.c_int32)]


class zs_adam_hparams(ctypes.Structure):
    _fields_ = [("lr", ctypes.c_float), ("beta1", ctypes.c_float), ("beta2", ctypes.c_float),
                ("eps", ctypes.c_float), ("weight_decay", ctypes.c_float)]


class zs_scaler(ctypes.Structure):
    _fields_ = [("scale", ctypes.c_float), ("min_scale", ctypes.c_float),
                ("window", ctypes.c_int32), ("clean_count", ctypes.c_int32),
                ("hysteresis", ctypes.c_int32), ("hyst_left", ctypes.c_int32),
                ("dynamic", ctypes.c_int32), ("consecutive_hysteresis", ctypes.c_int32)]


class zs_lr_schedule(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("pad_", ctypes.c_int32),
                ("warmup_steps", ctypes.c_int64), ("total_steps", ctypes.c_int64),
                ("min_lr", ctypes.c_float), ("max_lr", ctypes.c_float)]


class zs_device_state(ctypes.Structure):
    _fields_ = [("scaler", zs_scaler), ("overflow", ctypes.c_int32), ("buf", ctypes.c_int32),
                ("step", ctypes.c_int64),
                ("iterations", ctypes.c_int64), ("lr", ctypes.c_float),
                ("grad_div", ctypes.c_float)]


ZS_LR_CONSTANT, ZS_LR_WARMUP, ZS_LR_WARMUP_DECAY = 0, 1, 2


class zs_engine_config(ctypes.Structure):
    _fields_ = [("n", ctypes.c_int32), ("dt", ctypes.c_int32), ("count", ctypes.c_int64),
                ("accum_steps", ctypes.c_int32), ("acc", ctypes.c_void_p),
                ("master", ctypes.c_void_p), ("m", ctypes.c_void_p), ("v", ctypes.c_void_p),
                ("half_out", ctypes.c_void_p), ("hp", zs_adam_hparams),
                ("schedule", zs_lr_schedule), ("has_schedule", ctypes.c_int32),
                ("scaler", zs_scaler), ("max_grad_norm", ctypes.c_float)]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is missing: build it with zero_mixed_precision_shard_gb300.build() "
            "or __graft_entry__.build(); there is no CPU fallback")
    L = ctypes.CDLL(LIB_PATH)
    vp, i32, i64, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float
    i64p, i32p, u64p = (ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(ctypes.c_int32),
                        ctypes.POINTER(ctypes.c_uint64))
    pp = ctypes.POINTER(ctypes.c_void_p)
    sig = {
        "zs_init_partition": [i64, i32, i32, ctypes.POINTER(zs_partition)],
        "zs_shard_range": [ctypes.POINTER(zs_partition), i32, i64p, i64p, i64p],
        "zs_model_state_bytes": [ctypes.POINTER(zs_partition), i32, u64p],
        "zs_scaler_init": [ctypes.POINTER(zs_scaler), f32, f32, i32, i32, i32],
        "zs_ctx_create": [ctypes.POINTER(vp)],
        "zs_ctx_destroy": [vp],
        "zs_ctx_overflow_flag": [vp, ctypes.POINTER(vp)],
        "zs_grad_accum": [vp, pp, i32, i32, i64, vp, i32, vp],
        "zs_reduce_check": [vp, pp, i32, i32, i64, vp, i32, vp, vp],
        "zs_check_last": [vp, pp, i32, i32, i64, vp, vp, vp],
        "zs_apply": [vp, vp, pp, i32, i32, vp, i64, f32, vp, vp, vp, vp,
                     ctypes.POINTER(zs_adam_hparams), i64, vp],
        "zs_scaler_update": [vp, vp, ctypes.POINTER(zs_scaler), i32p, vp],
        "zs_shard_step": [vp, pp, i32, i32, i64, vp, i32, vp, vp, vp, vp,
                          ctypes.POINTER(zs_adam_hparams), i64, ctypes.POINTER(zs_scaler), i32p,
                          ctypes.POINTER(ctypes.c_float), vp],
        "zs_copy_peak": [vp, vp, vp, i64, i32, vp],
        "zs_engine_create": [vp, ctypes.POINTER(zs_engine_config), ctypes.POINTER(vp)],
        "zs_engine_destroy": [vp],
        "zs_engine_backward": [vp, pp, vp],
        "zs_engine_step": [vp, i32p, i32p, ctypes.POINTER(ctypes.c_float),
                           ctypes.POINTER(ctypes.c_float), vp],
        "zs_engine_state": [vp, i64p, i64p, i64p, ctypes.POINTER(zs_scaler)],
        "zs_grad_accum_halfacc": [vp, pp, i32, i32, i64, vp, i32, vp],
        "zs_shard_step_halfacc": [vp, pp, i32, i32, i64, vp, i32, vp, vp, vp, vp,
                                  ctypes.POINTER(zs_adam_hparams), i64, ctypes.POINTER(zs_scaler),
                                  i32p, ctypes.POINTER(ctypes.c_float), vp],
        "zs_shard_step_async": [vp, pp, i32, i32, i64, vp, i32, vp, vp, vp, vp,
                                ctypes.POINTER(zs_adam_hparams), ctypes.POINTER(zs_lr_schedule),
                                vp, vp],
        "zs_shard_step_async_clipped": [vp, pp, i32, i32, i64, vp, i32, vp, vp, vp, vp,
                                        ctypes.POINTER(zs_adam_hparams),
                                        ctypes.POINTER(zs_lr_schedule), f32, vp, vp, vp],
        "zs_shard_step_oop": [vp, pp, i32, i32, i64, vp, i32, vp, vp, vp, vp, vp, vp, vp,
                              ctypes.POINTER(zs_adam_hparams), i64, ctypes.POINTER(zs_scaler),
                              i32p, ctypes.POINTER(ctypes.c_float), vp],
        "zs_shard_step_async_oop": [vp, pp, i32, i32, i64, vp, i32, pp, pp, pp, pp,
                                    ctypes.POINTER(zs_adam_hparams),
                                    ctypes.POINTER(zs_lr_schedule), vp, vp],
        "zs_grad_sumsq": [vp, pp, i32, i32, vp, i64, f32, vp, vp],
        "zs_grad_sumsq_noalloc": [pp, i32, i32, vp, i64, f32, vp, vp],
        "zs_apply_clipped": [vp, vp, vp, f32, pp, i32, i32, vp, i64, f32, vp, vp, vp, vp,
                             ctypes.POINTER(zs_adam_hparams), i64, vp],
        "zs_shard_step_clipped": [vp, pp, i32, i32, i64, vp, i32, vp, vp, vp, vp,
                                  ctypes.POINTER(zs_adam_hparams), i64, ctypes.POINTER(zs_scaler),
                                  f32, i32p, ctypes.POINTER(ctypes.c_float),
                                  ctypes.POINTER(ctypes.c_float), vp],
        "zs_update_oop": [vp, pp, i32, i32, i64, vp, f32, vp, vp, vp, vp, vp, vp, vp,
                          ctypes.POINTER(zs_adam_hparams), i64, vp, vp],
        "zs_shard_step_halfacc_oop": [vp, pp, i32, i32, i64, vp, i32, vp, vp, vp, vp, vp, vp,
                                      vp, ctypes.POINTER(zs_adam_hparams), i64,
                                      ctypes.POINTER(zs_scaler), i32p,
                                      ctypes.POINTER(ctypes.c_float), vp],
        "zs_shard_step_halfacc_async": [vp, pp, i32, i32, i64, vp, i32, vp, vp, vp, vp,
                                        ctypes.POINTER(zs_adam_hparams),
                                        ctypes.POINTER(zs_lr_schedule), vp, vp],
        "zs_shard_step_halfacc_async_oop": [vp, pp, i32, i32, i64, vp, i32, pp, pp, pp, pp,
                                            ctypes.POINTER(zs_adam_hparams),
                                            ctypes.POINTER(zs_lr_schedule), vp, vp],
        "zs_ctx_set_timing": [vp, i32],
        "zs_ctx_set_fused": [vp, i32, i64],
        "zs_ctx_fused_capacity": [vp, i64p],
        "zs_ctx_timing": [vp, i32, ctypes.POINTER(ctypes.c_double), i64p, i64p],
        "zs_ctx_timing_reset": [vp],
        "zs_ctx_launch_count": [vp, i64p],
    }
    for name, args in sig.items():
        fn = getattr(L, name)
        fn.argtypes = args
        fn.restype = ctypes.c_int
    L.zs_last_error.argtypes = [vp]
    L.zs_last_error.restype = ctypes.c_char_p
    return L


lib = _load()


def _addr(x) -> int | None:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _current_stream() -> int:
    """The calling thread's current torch stream on the current device, as a
    cudaStream_t (a Stream object costs a few microseconds to build; a short
    step is launched in about as long)."""
    import torch
    raw = getattr(torch._C, "_cuda_getCurrentRawStream", None)
    if raw is not None:
        return raw(torch._C._cuda_getDevice())
    return torch.cuda.current_stream().cuda_stream


def _stream(s) -> int | None:
    if s is None:
        return _current_stream()
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _ptrs(tensors):
    if isinstance(tensors, ctypes.Array):  # prebuilt by the caller (see pointer_array)
        return tensors
    arr = (ctypes.c_void_p * len(tensors))()
    for i, t in enumerate(tensors):
        arr[i] = _addr(t)
    return arr


def pointer_array(tensors):
    """A reusable host array of device pointers for the `grads` arguments."""
    return _ptrs(list(tensors))


def _dtype(dt) -> int:
    if isinstance(dt, int):
        return dt
    s = str(dt)
    if s in ("fp16", "torch.float16"):
        return ZS_FP16
    if s in ("bf16", "torch.bfloat16"):
        return ZS_BF16
    raise ValueError(f"unsupported gradient dtype {dt}")


class Ctx:
    """A zs_ctx on the current CUDA device."""

    def __init__(self):
        h = ctypes.c_void_p()
        rc = lib.zs_ctx_create(ctypes.byref(h))
        if rc != ZS_OK:
            raise ZsError(rc, "zs_ctx_create failed")
        self.handle = h

    def check(self, rc: int):
        if rc != ZS_OK:
            raise ZsError(rc, lib.zs_last_error(self.handle).decode())

    def close(self):
        if self.handle:
            lib.zs_ctx_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @property
    def overflow_flag_ptr(self) -> int:
        p = ctypes.c_void_p()
        self.check(lib.zs_ctx_overflow_flag(self.handle, ctypes.byref(p)))
        return p.value

    def set_timing(self, enable: bool):
        self.check(lib.zs_ctx_set_timing(self.handle, 1 if enable else 0))

    def set_fused(self, mode: int, wait_ns: int = 0):
        """ZS_FUSED_OFF / ZS_FUSED_ON / ZS_FUSED_TEST_TIMEOUT; wait_ns <= 0: the default."""
        self.check(lib.zs_ctx_set_fused(self.handle, mode, wait_ns))

    @property
    def fused_capacity(self) -> int:
        """The largest count the fused step takes on this device."""
        n = ctypes.c_int64()
        self.check(lib.zs_ctx_fused_capacity(self.handle, ctypes.byref(n)))
        return n.value

    def timing(self, kind: int):
        ms, n, el = ctypes.c_double(), ctypes.c_int64(), ctypes.c_int64()
        self.check(lib.zs_ctx_timing(self.handle, kind, ctypes.byref(ms), ctypes.byref(n),
                                     ctypes.byref(el)))
        return ms.value, n.value, el.value

    def timing_reset(self):
        self.check(lib.zs_ctx_timing_reset(self.handle))

    @property
    def launch_count(self) -> int:
        n = ctypes.c_int64()
        self.check(lib.zs_ctx_launch_count(self.handle, ctypes.byref(n)))
        return n.value


@dataclass
class Partition:
    psi: int
    psi_pad: int
    shard_len: int
    n: int
    align: int

    def _c(self):
        return zs_partition(self.psi, self.psi_pad, self.shard_len, self.n, self.align)


def zs_init_partition(psi: int, n: int, align_elems: int = ZS_DEFAULT_ALIGN) -> Partition:
    p = zs_partition()
    rc = lib.zs_init_partition(psi, n, align_elems, ctypes.byref(p))
    if rc != ZS_OK:
        raise ZsError(rc, f"zs_init_partition({psi}, {n}, {align_elems})")
    return Partition(p.psi, p.psi_pad, p.shard_len, p.n, p.align)


def zs_shard_range(p: Partition, rank: int):
    b, ve, pe = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()
    cp = p._c()
    rc = lib.zs_shard_range(ctypes.byref(cp), rank, ctypes.byref(b), ctypes.byref(ve),
                            ctypes.byref(pe))
    if rc != ZS_OK:
        raise ZsError(rc, f"zs_shard_range(rank={rank})")
    return b.value, ve.value, pe.value


def zs_model_state_bytes(p: Partition, stage: int) -> int:
    out = ctypes.c_uint64()
    cp = p._c()
    rc = lib.zs_model_state_bytes(ctypes.byref(cp), stage, ctypes.byref(out))
    if rc != ZS_OK:
        raise ZsError(rc, f"zs_model_state_bytes(stage={stage})")
    return out.value


def zs_scaler_init(scale: float, min_scale: float = 1.0, window: int = 1000,
                   hysteresis: int = 2, dynamic: bool = True,
                   consecutive_hysteresis: bool = False) -> zs_scaler:
    s = zs_scaler()
    rc = lib.zs_scaler_init(ctypes.byref(s), scale, min_scale, window, hysteresis,
                            1 if dynamic else 0)
    if rc != ZS_OK:
        raise ZsError(rc, "zs_scaler_init")
    s.consecutive_hysteresis = 1 if consecutive_hysteresis else 0
    return s


def make_hparams(lr, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.0) -> zs_adam_hparams:
    return zs_adam_hparams(lr, beta1, beta2, eps, weight_decay)


def zs_grad_accum(ctx: Ctx, grads, dt, count: int, acc, first: bool, stream=None):
    ctx.check(lib.zs_grad_accum(ctx.handle, _ptrs(grads), len(grads), _dtype(dt), count,
                                _addr(acc), 1 if first else 0, _stream(stream)))


def zs_reduce_check(ctx: Ctx, grads, dt, count: int, acc, first: bool, d_flag, stream=None):
    ctx.check(lib.zs_reduce_check(ctx.handle, _ptrs(grads), len(grads), _dtype(dt), count,
                                  _addr(acc), 1 if first else 0, _addr(d_flag), _stream(stream)))


def zs_check_last(ctx: Ctx, grads, dt, count: int, acc, d_flag, stream=None):
    ctx.check(lib.zs_check_last(ctx.handle, _ptrs(grads), len(grads), _dtype(dt), count,
                                _addr(acc), _addr(d_flag), _stream(stream)))


def zs_apply(ctx: Ctx, d_flag, grads, dt, acc, count: int, grad_div: float, master, m, v,
             half_out, hp: zs_adam_hparams, step: int, stream=None):
    g = _ptrs(grads) if grads is not None else None
    n = len(grads) if grads is not None else 0
    ctx.check(lib.zs_apply(ctx.handle, _addr(d_flag), g, n, _dtype(dt), _addr(acc), count,
                           grad_div, _addr(master), _addr(m), _addr(v), _addr(half_out),
                           ctypes.byref(hp), step, _stream(stream)))


def zs_scaler_update(ctx: Ctx, d_flag, scaler: zs_scaler, stream=None) -> int:
    ovf = ctypes.c_int32()
    ctx.check(lib.zs_scaler_update(ctx.handle, _addr(d_flag), ctypes.byref(scaler),
                                   ctypes.byref(ovf), _stream(stream)))
    return ovf.value


def zs_shard_step(ctx: Ctx, grads, dt, count: int, acc, accum_steps: int, master, m, v,
                  half_out, hp: zs_adam_hparams, step: int, scaler: zs_scaler, stream=None):
    """Returns (overflow, new_scale); *scaler is updated in place."""
    ovf = ctypes.c_int32()
    ns = ctypes.c_float()
    ctx.check(lib.zs_shard_step(ctx.handle, _ptrs(grads), len(grads), _dtype(dt), count,
                                _addr(acc), accum_steps, _addr(master), _addr(m), _addr(v),
                                _addr(half_out), ctypes.byref(hp), step, ctypes.byref(scaler),
                                ctypes.byref(ovf), ctypes.byref(ns), _stream(stream)))
    return ovf.value, ns.value


def zs_grad_sumsq(ctx: Ctx, grads, dt, acc, count: int, grad_div: float, d_sumsq, stream=None):
    g = _ptrs(grads) if grads is not None else None
    n = len(grads) if grads is not None else 0
    ctx.check(lib.zs_grad_sumsq(ctx.handle, g, n, _dtype(dt), _addr(acc), count, grad_div,
                                _addr(d_sumsq), _stream(stream)))


def zs_grad_sumsq_noalloc(grads, dt, acc, count: int, grad_div: float, d_sumsq, stream=None):
    """Allocation-free zs_grad_sumsq (no context; count <= ZS_NOALLOC_MAX_COUNT)."""
    g = _ptrs(grads) if grads is not None else None
    n = len(grads) if grads is not None else 0
    rc = lib.zs_grad_sumsq_noalloc(g, n, _dtype(dt), _addr(acc), count, grad_div,
                                   _addr(d_sumsq), _stream(stream))
    if rc != ZS_OK:
        raise ZsError(rc, "zs_grad_sumsq_noalloc failed")


def zs_apply_clipped(ctx: Ctx, d_flag, d_sumsq, max_norm: float, grads, dt, acc, count: int,
                     grad_div: float, master, m, v, half_out, hp: zs_adam_hparams, step: int,
                     stream=None):
    g = _ptrs(grads) if grads is not None else None
    n = len(grads) if grads is not None else 0
    ctx.check(lib.zs_apply_clipped(ctx.handle, _addr(d_flag), _addr(d_sumsq), max_norm, g, n,
                                   _dtype(dt), _addr(acc), count, grad_div, _addr(master),
                                   _addr(m), _addr(v), _addr(half_out), ctypes.byref(hp), step,
                                   _stream(stream)))


def zs_shard_step_clipped(ctx: Ctx, grads, dt, count: int, acc, accum_steps: int, master, m, v,
                          half_out, hp: zs_adam_hparams, step: int, scaler: zs_scaler,
                          max_norm: float, stream=None):
    """Returns (overflow, new_scale, grad_norm); *scaler is updated in place."""
    ovf = ctypes.c_int32()
    ns = ctypes.c_float()
    gn = ctypes.c_float()
    ctx.check(lib.zs_shard_step_clipped(ctx.handle, _ptrs(grads), len(grads), _dtype(dt), count,
                                        _addr(acc), accum_steps, _addr(master), _addr(m),
                                        _addr(v), _addr(half_out), ctypes.byref(hp), step,
                                        ctypes.byref(scaler), max_norm, ctypes.byref(ovf),
                                        ctypes.byref(ns), ctypes.byref(gn), _stream(stream)))
    return ovf.value, ns.value, gn.value


class DeviceState:
    """A zs_device_state in device memory (a 64-byte torch buffer)."""

    def __init__(self, scaler: zs_scaler, step: int = 0, device=None):
        import torch
        assert ctypes.sizeof(zs_device_state) == 64
        st = zs_device_state()
        st.scaler = scaler
        st.step = step
        host = torch.frombuffer(bytearray(bytes(st)), dtype=torch.uint8)
        self.buf = host.to(device or torch.device("cuda", torch.cuda.current_device()))

    def data_ptr(self) -> int:
        return self.buf.data_ptr()

    def read(self) -> zs_device_state:
        return zs_device_state.from_buffer_copy(self.buf.cpu().numpy().tobytes())


def make_schedule(kind: int, min_lr: float, max_lr: float, warmup_steps: int = 0,
                  total_steps: int = 0) -> zs_lr_schedule:
    return zs_lr_schedule(kind, 0, warmup_steps, total_steps, min_lr, max_lr)


def zs_shard_step_async(ctx: Ctx, grads, dt, count: int, acc, accum_steps: int, master, m, v,
                        half_out, hp: zs_adam_hparams, sched, d_state, stream=None):
    ctx.check(lib.zs_shard_step_async(ctx.handle, _ptrs(grads), len(grads), _dtype(dt), count,
                                      _addr(acc), accum_steps, _addr(master), _addr(m), _addr(v),
                                      _addr(half_out), ctypes.byref(hp),
                                      ctypes.byref(sched) if sched is not None else None,
                                      _addr(d_state), _stream(stream)))


def zs_shard_step_async_clipped(ctx: Ctx, grads, dt, count: int, acc, accum_steps: int, master,
                                m, v, half_out, hp: zs_adam_hparams, sched, max_norm: float,
                                d_state, d_grad_norm=None, stream=None):
    ctx.check(lib.zs_shard_step_async_clipped(
        ctx.handle, _ptrs(grads), len(grads), _dtype(dt), count, _addr(acc), accum_steps,
        _addr(master), _addr(m), _addr(v), _addr(half_out), ctypes.byref(hp),
        ctypes.byref(sched) if sched is not None else None, max_norm, _addr(d_state),
        _addr(d_grad_norm), _stream(stream)))


def zs_shard_step_oop(ctx: Ctx, grads, dt, count: int, acc, accum_steps: int, master_in, m_in,
                      v_in, master_out, m_out, v_out, half_out, hp: zs_adam_hparams, step: int,
                      scaler: zs_scaler, stream=None):
    """Returns (overflow, new_scale); on overflow == 0 the *_out buffers hold the
    new state.  *scaler is updated in place."""
    ovf = ctypes.c_int32()
    ns = ctypes.c_float()
    ctx.check(lib.zs_shard_step_oop(ctx.handle, _ptrs(grads), len(grads), _dtype(dt), count,
                                    _addr(acc), accum_steps, _addr(master_in), _addr(m_in),
                                    _addr(v_in), _addr(master_out), _addr(m_out), _addr(v_out),
                                    _addr(half_out), ctypes.byref(hp), step, ctypes.byref(scaler),
                                    ctypes.byref(ovf), ctypes.byref(ns), _stream(stream)))
    return ovf.value, ns.value


def zs_update_oop(ctx: Ctx, grads, dt, count: int, acc, grad_div: float, master_in, m_in, v_in,
                  master_out, m_out, v_out, half_out, hp: zs_adam_hparams, step: int, d_flag,
                  stream=None):
    """The two-phase out-of-place update of one range: ORs its flag into d_flag
    and writes the *_out buffers whatever the flag (the commit is the caller's,
    after zs_scaler_update)."""
    ctx.check(lib.zs_update_oop(ctx.handle, _ptrs(grads), len(grads), _dtype(dt), count,
                                _addr(acc), grad_div, _addr(master_in), _addr(m_in), _addr(v_in),
                                _addr(master_out), _addr(m_out), _addr(v_out), _addr(half_out),
                                ctypes.byref(hp), step, _addr(d_flag), _stream(stream)))


def zs_shard_step_async_oop(ctx: Ctx, grads, dt, count: int, acc, accum_steps: int, master,
                            m, v, half, hp: zs_adam_hparams, sched, d_state, stream=None):
    """master, m, v, half: pairs of buffers; d_state.buf names the current one."""
    ctx.check(lib.zs_shard_step_async_oop(
        ctx.handle, _ptrs(grads), len(grads), _dtype(dt), count, _addr(acc), accum_steps,
        _ptrs(master), _ptrs(m), _ptrs(v), _ptrs(half), ctypes.byref(hp),
        ctypes.byref(sched) if sched is not None else None, _addr(d_state), _stream(stream)))


def zs_grad_accum_halfacc(ctx: Ctx, grads, dt, count: int, acc_half, first: bool, stream=None):
    ctx.check(lib.zs_grad_accum_halfacc(ctx.handle, _ptrs(grads), len(grads), _dtype(dt), count,
                                        _addr(acc_half), 1 if first else 0, _stream(stream)))


def zs_shard_step_halfacc(ctx: Ctx, grads, dt, count: int, acc_half, accum_steps: int, master,
                          m, v, half_out, hp: zs_adam_hparams, step: int, scaler: zs_scaler,
                          stream=None):
    """Returns (overflow, new_scale); *scaler is updated in place."""
    ovf = ctypes.c_int32()
    ns = ctypes.c_float()
    ctx.check(lib.zs_shard_step_halfacc(ctx.handle, _ptrs(grads), len(grads), _dtype(dt), count,
                                        _addr(acc_half), accum_steps, _addr(master), _addr(m),
                                        _addr(v), _addr(half_out), ctypes.byref(hp), step,
                                        ctypes.byref(scaler), ctypes.byref(ovf),
                                        ctypes.byref(ns), _stream(stream)))
    return ovf.value, ns.value


def zs_shard_step_halfacc_oop(ctx: Ctx, grads, dt, count: int, acc_half, accum_steps: int,
                              master_in, m_in, v_in, master_out, m_out, v_out, half_out,
                              hp: zs_adam_hparams, step: int, scaler: zs_scaler, stream=None):
    """Returns (overflow, new_scale); on overflow == 0 the *_out buffers hold the
    new state.  *scaler is updated in place."""
    ovf = ctypes.c_int32()
    ns = ctypes.c_float()
    ctx.check(lib.zs_shard_step_halfacc_oop(
        ctx.handle, _ptrs(grads), len(grads), _dtype(dt), count, _addr(acc_half), accum_steps,
        _addr(master_in), _addr(m_in), _addr(v_in), _addr(master_out), _addr(m_out),
        _addr(v_out), _addr(half_out), ctypes.byref(hp), step, ctypes.byref(scaler),
        ctypes.byref(ovf), ctypes.byref(ns), _stream(stream)))
    return ovf.value, ns.value


def zs_shard_step_halfacc_async(ctx: Ctx, grads, dt, count: int, acc_half, accum_steps: int,
                                master, m, v, half_out, hp: zs_adam_hparams, sched, d_state,
                                stream=None):
    ctx.check(lib.zs_shard_step_halfacc_async(
        ctx.handle, _ptrs(grads), len(grads), _dtype(dt), count, _addr(acc_half), accum_steps,
        _addr(master), _addr(m), _addr(v), _addr(half_out), ctypes.byref(hp),
        ctypes.byref(sched) if sched is not None else None, _addr(d_state), _stream(stream)))


def zs_shard_step_halfacc_async_oop(ctx: Ctx, grads, dt, count: int, acc_half,
                                    accum_steps: int, master, m, v, half, hp: zs_adam_hparams,
                                    sched, d_state, stream=None):
    """master, m, v, half: pairs of buffers; d_state.buf names the current one."""
    ctx.check(lib.zs_shard_step_halfacc_async_oop(
        ctx.handle, _ptrs(grads), len(grads), _dtype(dt), count, _addr(acc_half), accum_steps,
        _ptrs(master), _ptrs(m), _ptrs(v), _ptrs(half), ctypes.byref(hp),
        ctypes.byref(sched) if sched is not None else None, _addr(d_state), _stream(stream)))


class Engine:
    """zs_engine: backward() per micro-batch, step() after each (§5.1's loop)."""

    def __init__(self, ctx: Ctx, n, dt, count, accum_steps, acc, master, m, v, half_out,
                 hp: zs_adam_hparams, scaler: zs_scaler, schedule=None, max_grad_norm=0.0):
        cfg = zs_engine_config()
        cfg.n, cfg.dt, cfg.count, cfg.accum_steps = n, _dtype(dt), count, accum_steps
        cfg.acc, cfg.master, cfg.m, cfg.v = _addr(acc), _addr(master), _addr(m), _addr(v)
        cfg.half_out = _addr(half_out)
        cfg.hp = hp
        if schedule is not None:
            cfg.schedule = schedule
            cfg.has_schedule = 1
        cfg.scaler = scaler
        cfg.max_grad_norm = max_grad_norm
        self.ctx = ctx
        self.handle = ctypes.c_void_p()
        ctx.check(lib.zs_engine_create(ctx.handle, ctypes.byref(cfg), ctypes.byref(self.handle)))

    def backward(self, grads, stream=None):
        self.ctx.check(lib.zs_engine_backward(self.handle, _ptrs(grads), _stream(stream)))

    def step(self, stream=None):
        """Returns None between boundaries, else (overflow, new_scale, grad_norm)."""
        st, ovf = ctypes.c_int32(), ctypes.c_int32()
        sc, gn = ctypes.c_float(), ctypes.c_float()
        self.ctx.check(lib.zs_engine_step(self.handle, ctypes.byref(st), ctypes.byref(ovf),
                                          ctypes.byref(sc), ctypes.byref(gn), _stream(stream)))
        return (ovf.value, sc.value, gn.value) if st.value else None

    def state(self):
        g, a, mi = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()
        sc = zs_scaler()
        lib.zs_engine_state(self.handle, ctypes.byref(g), ctypes.byref(a), ctypes.byref(mi),
                            ctypes.byref(sc))
        return {"global_steps": g.value, "applied_steps": a.value, "micro_steps": mi.value,
                "scaler": sc}

    def close(self):
        if self.handle:
            lib.zs_engine_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def zs_copy_peak(ctx: Ctx, src, dst, nbytes: int, read_only: bool = False, stream=None):
    ctx.check(lib.zs_copy_peak(ctx.handle, _addr(src), _addr(dst), nbytes,
                               1 if read_only else 0, _stream(stream)))
