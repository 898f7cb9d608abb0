"""Benchmark of the ZeRO shard step on GB300.

One GPU: one step = one optimizer step of the owned shard: G-1 calls of
zs_grad_accum (micro-steps 1..G-1, each summing the N simulated ranks'
gradient slices onto the fp32 accumulator) and the step's last call (last
micro-step, overflow resolution, AdamW + half cast, loss-scale update).  By
default that call is zs_shard_step_async, which keeps the scale and step count
on the device (no host round trip per step); --api sync uses zs_shard_step.
Inputs are synthetic and seeded (synth/), resident in HBM before the timed
region.  After the headline workload the other target workloads are measured
in the same run (config.workloads).

Default workload: the Llama-7B-shaped full model on one GPU (N = 1 simulated
rank, G = 8 micro-steps, fp16 gradients, AdamW), 6,738,415,616 parameters,
~229 GB resident.  Output: one JSON line (metric: shard-step params/s, with the
achieved HBM GB/s of the dominant kernel against the measured peak).

N GPUs (torchrun, one rank per GPU): the ZeRO-2 step with its real exchanges
(dp.Zero2Step): the workload's parameters partitioned over the N ranks, each
rank's own full gradients exchanged bucket by bucket, the flag agreed, the
half copy all-gathered.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the CPU oracle on a bounded sample
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import synth  # noqa: E402

DEFAULT_WORKLOAD = "llama7b-n1"
METRIC = "ZeRO shard-step params/s and achieved HBM GB/s vs measured GB300 peak"


# ---------------------------------------------------------------- byte model

def alg_bytes_per_elem_step(n: int, g: int, acc_bytes: int = 4) -> int:
    """Algorithmic bytes per owned element per step: read every gradient once
    (2·N·G), carry the accumulator between micro-steps (2·acc_bytes·(G-1):
    8 for fp32, 4 for the half accumulator), read and write master/m/v (24)
    and write the half copy (2)."""
    return 2 * n * g + 2 * acc_bytes * (g - 1) + 26


def kernel_alg_bytes(kind: str, n: int, first: bool = False, with_acc: bool = False,
                     acc_bytes: int = 4) -> int:
    """Algorithmic bytes per element of one launch of each kernel kind."""
    if kind == "reduce":
        return 2 * n + (acc_bytes if first else 2 * acc_bytes)
    if kind == "check":
        return 2 * n + (4 if with_acc else 0)
    if kind == "apply":
        return acc_bytes + 12 + 14
    if kind == "apply_recompute":
        return (4 if with_acc else 0) + 2 * n + 26
    if kind == "sumsq":   # a separate norm pass: acc and/or the re-read slices
        return (4 if with_acc else 0) + (2 * n if first else 0)
    if kind == "update_oop":   # last micro-step + flag + update, state written out of place
        return (acc_bytes if with_acc else 0) + 2 * n + 26
    if kind == "fused":   # last micro-step + flag + grid barrier + update, one kernel
        return (acc_bytes if with_acc else 0) + 2 * n + 26
    raise ValueError(kind)


def step_launch_plan(n: int, g: int, dtype: str, acc_kind: str = "fp32", has_acc: bool = True,
                     clip: float = 0.0, split: bool = False, oop: bool = False,
                     fused: bool = False):
    """(kind, alg bytes per element) of every kernel one step launches, in the
    order the step launches them (split: the step split at the overflow flag
    as every rank of a multi-GPU run does, the clipping norm in its own pass;
    oop: the out-of-place step, whose last pass is the update; fused: the
    shard fits the fused step, whose last call is one kernel in every form)."""
    if fused:
        ab = 2 if acc_kind == "half" else 4
        plan = [("reduce_first" if k == 0 else "reduce",
                 kernel_alg_bytes("reduce", n, first=(k == 0), acc_bytes=ab))
                for k in range(g - 1)]
        plan.append(("fused", kernel_alg_bytes("fused", n, with_acc=g > 1, acc_bytes=ab)))
        return plan
    if oop:
        ab = 2 if acc_kind == "half" else 4
        plan = [("reduce_first" if k == 0 else "reduce",
                 kernel_alg_bytes("reduce", n, first=(k == 0), acc_bytes=ab))
                for k in range(g - 1)]
        plan.append(("update_oop", kernel_alg_bytes("update_oop", n, with_acc=g > 1,
                                                    acc_bytes=ab)))
        return plan
    if acc_kind == "half":
        plan = [("reduce_first" if k == 0 else "reduce",
                 kernel_alg_bytes("reduce", n, first=(k == 0), acc_bytes=2)) for k in range(g)]
        plan.append(("apply", kernel_alg_bytes("apply", n, acc_bytes=2)))
        return plan
    plan = [("reduce_first" if k == 0 else "reduce",
             kernel_alg_bytes("reduce", n, first=(k == 0))) for k in range(g - 1)]
    recompute = n < 4 or not has_acc
    clip_fused = clip > 0 and not split
    if recompute:
        # the flag pass reads acc too for bf16, or to fold in the clipping norm
        with_acc = g > 1 and (dtype == "bf16" or clip_fused)
        plan.append(("check", kernel_alg_bytes("check", n, with_acc=with_acc)))
        if clip > 0 and split:
            plan.append(("sumsq", kernel_alg_bytes("sumsq", n, first=True, with_acc=g > 1)))
        plan.append(("apply_recompute", kernel_alg_bytes("apply_recompute", n, with_acc=g > 1)))
    else:
        plan.append(("reduce_first" if g == 1 else "reduce",
                     kernel_alg_bytes("reduce", n, first=(g == 1))))
        if clip > 0 and split:
            plan.append(("sumsq", kernel_alg_bytes("sumsq", n, with_acc=True)))
        plan.append(("apply", kernel_alg_bytes("apply", n)))
    return plan


# ---------------------------------------------------------------- device workload

class DeviceWorkload:
    """HBM-resident buffers of one owned shard of a workload: the gradient
    slices (half) of N ranks for each of `grad_buffers` micro-steps (None: all
    G; micro-step k reads buffer k mod grad_buffers, as a training loop refills
    one buffer while another is reduced), the fp32 accumulator, fp32 master /
    m / v and the half copy."""

    def __init__(self, wl: synth.Workload, shard: int = 0, device=None, count: int | None = None,
                 acc: str = "fp32", clip: float = 0.0, grad_buffers: int | None = None):
        import torch
        import zero_mixed_precision_shard_gb300 as zs
        self.zs = zs
        self.wl = wl
        self.dev = device or torch.device("cuda", torch.cuda.current_device())
        self.part = zs.zs_init_partition(wl.psi, wl.n, synth.ALIGN_ELEMS)
        self.shard = shard
        self.begin, self.valid_end, _ = zs.zs_shard_range(self.part, shard)
        self.E = self.part.shard_len if count is None else count
        E, n, g = self.E, wl.n, wl.g
        self.nbuf = g if grad_buffers is None else max(1, min(g, grad_buffers))
        self.grads = torch.empty((self.nbuf, n, E), dtype=torch.int16, device=self.dev)
        self.acc_kind = acc
        self.clip = clip
        self.hacc_oop = False   # set by the caller once every buffer is allocated
        if acc == "half":
            self.acc = torch.empty(E, dtype=torch.int16, device=self.dev)
        else:
            need_acc = g > 1 or n >= 4
            self.acc = torch.empty(E, dtype=torch.float32, device=self.dev) if need_acc else None
        self.master = torch.empty(E, dtype=torch.float32, device=self.dev)
        self.m = torch.zeros(E, dtype=torch.float32, device=self.dev)
        self.v = torch.zeros(E, dtype=torch.float32, device=self.dev)
        self.half = torch.zeros(E, dtype=torch.int16, device=self.dev)
        synth.dev_fill_master(self.master.data_ptr(), E, self.begin, wl,
                              torch.cuda.current_stream().cuda_stream)
        self.hp = zs.make_hparams(wl.lr, wl.beta1, wl.beta2, wl.eps, wl.weight_decay)
        self.scaler = zs.zs_scaler_init(wl.scale0, wl.min_scale, wl.window, wl.hysteresis,
                                        wl.dynamic)
        self.t = 0  # applied Adam updates

    @property
    def dt(self):
        return self.wl.dtype_code

    def slices(self, k: int):
        """Host array of the N slice pointers micro-step k reads."""
        if not hasattr(self, "_ptr_arrays"):
            self._ptr_arrays = [self.zs.pointer_array(self.grads[j, r] for r in range(self.wl.n))
                                for j in range(self.nbuf)]
        return self._ptr_arrays[k % self.nbuf]

    def slice_tensors(self, k: int):
        return [self.grads[k % self.nbuf, r] for r in range(self.wl.n)]

    def fill_micro(self, step: int, k: int, scale: float, inject: bool = True):
        """Write micro-step k's gradients of `step` into the buffer it reads."""
        import torch
        s = torch.cuda.current_stream().cuda_stream
        for r in range(self.wl.n):
            buf = self.grads[k % self.nbuf, r]

            def writer(off, bits, buf=buf):
                buf[off] = int(np.array(bits, np.uint16).view(np.int16))

            synth.dev_fill_grads(buf.data_ptr(), self.E, self.begin, self.wl, step, k + 1, r,
                                 scale, s, inject=inject, inject_writer=writer)

    def fill_grads(self, step: int, scale: float, inject: bool = True):
        """Every buffer: micro-step b's values in buffer b (all G micro-steps when
        each has its own buffer)."""
        for k in range(self.nbuf):
            self.fill_micro(step, k, scale, inject)

    def accum(self, ctx, k: int):
        """Micro-step k (< G-1) of a step through the C ABI."""
        zs = self.zs
        if self.acc_kind == "half":
            zs.zs_grad_accum_halfacc(ctx, self.slices(k), self.dt, self.E, self.acc, k == 0)
        else:
            zs.zs_grad_accum(ctx, self.slices(k), self.dt, self.E, self.acc, k == 0)

    def finish(self, ctx) -> int:
        """The last micro-step and the update (the step's one synchronising
        call); returns the overflow flag."""
        zs, wl = self.zs, self.wl
        last = self.slices(wl.g - 1)
        if self.acc_kind == "half" and self.hacc_oop:
            # out of place where the second state set fits: the last micro-step,
            # its rounding to the half format, the flag and the update in one pass
            if not hasattr(self, "_hset"):
                import torch
                self._hset = (torch.empty_like(self.master), torch.empty_like(self.m),
                              torch.empty_like(self.v), torch.empty_like(self.half))
            dst = self._hset
            ovf, _ = zs.zs_shard_step_halfacc_oop(ctx, last, self.dt, self.E,
                                                  self.acc if wl.g > 1 else None, wl.g,
                                                  self.master, self.m, self.v, *dst, self.hp,
                                                  self.t + 1, self.scaler)
            if not ovf:
                self._hset = (self.master, self.m, self.v, self.half)
                self.master, self.m, self.v, self.half = dst
        elif self.acc_kind == "half":
            ovf, _ = zs.zs_shard_step_halfacc(ctx, last, self.dt, self.E, self.acc, wl.g,
                                              self.master, self.m, self.v, self.half, self.hp,
                                              self.t + 1, self.scaler)
        elif self.clip > 0:
            ovf, _, self.grad_norm = zs.zs_shard_step_clipped(
                ctx, last, self.dt, self.E, self.acc, wl.g, self.master, self.m, self.v,
                self.half, self.hp, self.t + 1, self.scaler, self.clip)
        else:
            ovf, _ = zs.zs_shard_step(ctx, last, self.dt, self.E, self.acc, wl.g, self.master,
                                      self.m, self.v, self.half, self.hp, self.t + 1,
                                      self.scaler)
        if not ovf:
            self.t += 1
        return ovf

    def step(self, ctx) -> int:
        """One optimizer step through the C ABI; returns the overflow flag."""
        for k in range(self.wl.g - 1):
            self.accum(ctx, k)
        return self.finish(ctx)

    def step_async_calls(self, ctx, state):
        """The calls of one step on the device-resident path (capturable)."""
        for k in range(self.wl.g - 1):
            self.accum(ctx, k)
        self.finish_async(ctx, state)

    def finish_async(self, ctx, state):
        """The last call of a step on the device-resident path: the scale, Adam's
        step count and the step's outcome stay in `state` on the device (with
        clipping, the norm in a device word too)."""
        zs, wl = self.zs, self.wl
        if self.acc_kind == "half":
            zs.zs_shard_step_halfacc_async(ctx, self.slices(wl.g - 1), self.dt, self.E, self.acc,
                                           wl.g, self.master, self.m, self.v, self.half, self.hp,
                                           None, state)
        elif self.clip > 0:
            if not hasattr(self, "d_norm"):
                import torch
                self.d_norm = torch.zeros(1, dtype=torch.float64, device=self.dev)
            zs.zs_shard_step_async_clipped(ctx, self.slices(wl.g - 1), self.dt, self.E, self.acc,
                                           wl.g, self.master, self.m, self.v, self.half, self.hp,
                                           None, self.clip, state, self.d_norm)
        else:
            zs.zs_shard_step_async(ctx, self.slices(wl.g - 1), self.dt, self.E, self.acc, wl.g,
                                   self.master, self.m, self.v, self.half, self.hp, None, state)

    def launch_plan(self, split: bool = False, oop: bool = False, fused: bool = False):
        """(kind, alg bytes per element) of every kernel one step launches."""
        return step_launch_plan(self.wl.n, self.wl.g, self.wl.dtype, self.acc_kind,
                                self.acc is not None, self.clip, split, oop, fused)

    def takes_fused(self, ctx, api: str) -> bool:
        """Whether `api`'s last call runs as the fused single-kernel step here:
        every form (clipped or not, either accumulator), when the shard fits one
        co-resident grid (and the context has the fused step on)."""
        return (api in ("async", "async_oop", "graph", "sync")
                and self.E <= ctx.fused_capacity
                and os.environ.get("ZEROSHARD_FUSED", "1") != "0")

    def step_oop_calls(self, ctx, state):
        """One step of the device-resident out-of-place form."""
        for k in range(self.wl.g - 1):
            self.accum(ctx, k)
        self.finish_oop(ctx, state)

    def finish_oop(self, ctx, state):
        """The last call of an out-of-place step (the second state set is
        allocated on first use; state.buf names the current set)."""
        import torch
        zs, wl = self.zs, self.wl
        if not hasattr(self, "_pairs"):
            E = self.E
            self.master2 = torch.empty(E, dtype=torch.float32, device=self.dev)
            self.m2 = torch.empty(E, dtype=torch.float32, device=self.dev)
            self.v2 = torch.empty(E, dtype=torch.float32, device=self.dev)
            self.half2 = torch.empty(E, dtype=torch.int16, device=self.dev)
            self._pairs = [zs.pointer_array(x) for x in ((self.master, self.master2),
                                                         (self.m, self.m2), (self.v, self.v2),
                                                         (self.half, self.half2))]
        step = (zs.zs_shard_step_halfacc_async_oop if self.acc_kind == "half"
                else zs.zs_shard_step_async_oop)
        step(ctx, self.slices(wl.g - 1), self.dt, self.E, self.acc, wl.g, *self._pairs, self.hp,
             None, state)


# ---------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples during the timed region (SM clock, throttle reasons)."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.gpu_id = None
        try:
            import torch
            pr = torch.cuda.get_device_properties(device_index)
            self.gpu_id = f"{pr.pci_domain_id:08X}:{pr.pci_bus_id:02X}:{pr.pci_device_id:02X}.0"
        except Exception:
            pass
        self.rows = []
        self._stop = threading.Event()
        self._t = None

    def _run(self):
        while not self._stop.is_set():
            try:
                cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader"]
                if self.gpu_id:
                    cmd.insert(1, f"--id={self.gpu_id}")
                out = subprocess.run(cmd, capture_output=True, text=True, timeout=5).stdout
                if not out.strip() and self.gpu_id:
                    self.gpu_id = None
                    continue
                for line in out.strip().splitlines():
                    row = [x.strip() for x in line.split(",")]
                    if len(row) == 9:
                        self.rows.append(row)
            except Exception:
                return
            self._stop.wait(0.2)

    def __enter__(self):
        self._t = threading.Thread(target=self._run, daemon=True)
        self._t.start()
        return self

    def __exit__(self, *a):
        self._stop.set()
        if self._t:
            self._t.join(timeout=10)

    def summary(self):
        if not self.rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}

        def num(x):
            try:
                return float(x.split()[0])
            except Exception:
                return None
        sm = [num(r[1]) for r in self.rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in self.rows if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in self.rows:
            for name, val in zip(names, r[5:9]):
                if val.strip().lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": sorted(reasons),
                "samples": len(self.rows)}


# ---------------------------------------------------------------- helpers

def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def code_digest(path: str) -> str:
    """sha256 of a C/CUDA source with its comments, trailing blanks and blank
    lines removed: recorded counters stay tied to the code, not to its comments
    (the kernel sources hold no string literal with a comment marker)."""
    import hashlib
    import re
    with open(path, encoding="utf-8") as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    lines = [ln.rstrip() for ln in text.splitlines()]
    return hashlib.sha256("\n".join(ln for ln in lines if ln).encode()).hexdigest()


def recorded_traffic(workload: str, kind: str, elements_per_launch: float):
    """DRAM bytes per launch of `kind` from the ncu summary in profiles/traffic.json,
    scaled by elements; None unless that capture was taken of this workload
    with the kernel sources' code as it is now."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as f:
            rec = json.load(f)
        for rel, digest in rec["sources_code_sha256"].items():
            if code_digest(os.path.join(ROOT, rel)) != digest:
                return None
        if rec.get("workload") != workload:
            return None
        per = rec["bytes_per_elem"].get(kind)
        return None if per is None else per * elements_per_launch
    except (OSError, KeyError, ValueError):
        return None


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def copy_probe(zs, ctx, nbytes: int = 4 << 30, reps: int = 5):
    """Our own copy and read-only kernels over a buffer far larger than L2."""
    import torch
    src = torch.empty(nbytes // 4, dtype=torch.int32, device="cuda")
    dst = torch.empty_like(src)
    src.fill_(1)
    out = {}
    for name, ro in (("copy", False), ("read", True)):
        best = 0.0
        for _ in range(reps + 1):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            a.record()
            zs.zs_copy_peak(ctx, src, dst, nbytes, ro)
            b.record()
            b.synchronize()
            moved = nbytes * (1 if ro else 2)
            best = max(best, moved / (a.elapsed_time(b) * 1e-3) / 1e9)
        out[name] = round(best, 1)
    del src, dst
    torch.cuda.empty_cache()
    return out


def _oracle_worker(args):
    """One process: the oracle as it stands on its own contiguous slice of the
    owned shard; times whole steps after every worker is ready."""
    name, offset, count, budget_s, max_steps, barrier, warmup = args
    import oracle
    wl = synth.WORKLOADS[name]
    idx = np.arange(offset, offset + count, dtype=np.int64)
    grads = [[synth.host_grad_bits(wl, idx, 1, k + 1, r, wl.scale0, inject=False)
              for r in range(wl.n)] for k in range(wl.g)]
    st = oracle.ShardState.from_master(synth.host_master(wl, idx), wl.dtype_code)
    hp = oracle.make_hparams(wl.lr, wl.beta1, wl.beta2, wl.eps, wl.weight_decay)
    sc = oracle.make_scaler(wl.scale0, wl.min_scale, wl.window, wl.hysteresis, wl.dynamic)
    t = 0
    for _ in range(warmup):
        _, t, _ = oracle.shard_step(grads, wl.dtype_code, st, hp, t, sc)
    barrier.wait()
    steps, elapsed = 0, 0.0
    while steps < max_steps and elapsed < budget_s:
        t0 = time.perf_counter()
        _, t, _ = oracle.shard_step(grads, wl.dtype_code, st, hp, t, sc)
        elapsed += time.perf_counter() - t0
        steps += 1
    return count * steps, elapsed


def cpu_baseline(wl: synth.Workload, budget_s: float = 10.0, max_steps: int = 50):
    """The oracle, as it stands (single-threaded C, fp64), run as one process
    per host core on disjoint contiguous slices of the owned shard (the step
    is elementwise), each repeating whole steps (G micro-steps x N ranks) for
    about budget_s seconds; input generation is outside the timed calls.
    Processes are spawned, never forked."""
    import multiprocessing as mp
    cores = os.cpu_count() or 1
    per = min(1 << 22, max(1 << 16, (1 << 28) // (wl.n * wl.g * cores)))
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        barrier = mgr.Barrier(cores)
        with ctx.Pool(cores) as pool:
            res = pool.map(_oracle_worker, [(wl.name, i * per, per, budget_s, max_steps, barrier,
                                             0) for i in range(cores)])
    elems = sum(r[0] for r in res)
    slowest = max(r[1] for r in res)
    single = res[0][0] / res[0][1]
    return {"value": elems / slowest, "unit": "params/s", "cores": cores, "kind": "oracle",
            "single_core_value": single,
            "sample": f"{cores} processes x {per} contiguous elements of the owned shard "
                      f"({wl.g} micro-steps x {wl.n} ranks), whole steps for ~{budget_s:.0f} s "
                      f"each; slowest process {slowest:.1f} s"}


# ---------------------------------------------------------------- arms

def run_reference(args):
    """The oracle as it stands, on every host core (one spawned process per
    core, disjoint slices of the owned shard): W warm-up steps, then K timed
    steps; the slowest process's time counts."""
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    import multiprocessing as mp
    wl = synth.WORKLOADS[args.workload]
    cores = os.cpu_count() or 1
    per = min(1 << 20, max(1 << 14, (1 << 25) // (wl.n * wl.g * cores)))
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        barrier = mgr.Barrier(cores)
        with ctx.Pool(cores) as pool:
            res = pool.map(_oracle_worker, [(wl.name, i * per, per, float("inf"), args.steps,
                                             barrier, args.warmup) for i in range(cores)])
    elems = sum(r[0] for r in res)
    slowest = max(r[1] for r in res)
    value = elems / slowest
    sample = (f"{cores} processes x {per} contiguous elements of the owned shard "
              f"({wl.g} micro-steps x {wl.n} ranks) per step")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "params/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": slowest / args.steps * 1e3, "higher_is_better": True, "scaling": "strong",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": wl.name, "n_ranks_simulated": wl.n, "accum_steps": wl.g,
                   "grad_dtype": wl.dtype, "sample_elements_per_step": per * cores},
        "cpu_baseline": {"value": value, "unit": "params/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "params/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


API_DESC = {
    "async": "zs_grad_accum + zs_shard_step_async (scale, step count and outcome stay on the "
             "device; no host round trip; the state is read back after the timed steps)",
    "async_oop": "zs_grad_accum + zs_shard_step_async_oop (device-resident, state written out "
                 "of place: the last micro-step, the flag and the update in one pass)",
    "sync": "zs_grad_accum + zs_shard_step (one host round trip per step)",
    "graph": "CUDA graph of zs_grad_accum + zs_shard_step_async",
    "graph_oop": "zs_grad_accum + zs_shard_step_async_oop captured once in a CUDA graph and "
                 "replayed (no host launch work per step: the step's GPU rate)",
    "split": "zs_reduce_check / zs_check_last + zs_apply + zs_scaler_update (split at the flag)",
}
HALF_API_DESC = {
    "async": "zs_grad_accum_halfacc + zs_shard_step_halfacc_async (half-precision carried "
             "sums; scale, step count and outcome stay on the device)",
    "async_oop": "zs_grad_accum_halfacc + zs_shard_step_halfacc_async_oop (half-precision "
                 "carried sums, device-resident, state written out of place)",
}


def api_desc(api: str, acc: str, clip: float, hacc_oop: bool) -> str:
    """The entry points one step of `api` calls, as the bench line names them."""
    if acc == "half":
        if api != "sync":
            return HALF_API_DESC[api]
        return ("zs_grad_accum_halfacc + zs_shard_step_halfacc"
                + ("_oop (the second state set fits)" if hacc_oop else ""))
    if clip and api == "sync":
        return "zs_grad_accum + zs_shard_step_clipped"
    if clip and api in ("async_oop", "graph_oop"):
        raise ValueError("the out-of-place step has no clipped form")
    if clip:
        return API_DESC[api].replace("zs_shard_step_async", "zs_shard_step_async_clipped")
    return API_DESC[api]


# the other target workloads, measured in the same run after the headline one
TABLE_WORKLOADS = ("decoder-1.3b-n16", "llama7b-zero3-n64", "gpt2-small-n8", "flat-1m-n2")


def resolve_api(args, world: int) -> str:
    if world > 1 or args.split:
        return "split"
    if args.graph:
        return "graph"
    if args.api == "auto":   # decided once the workload's buffers are allocated
        return "async" if args.clip else "auto"
    return args.api


def oop_fits(E: int, margin: int = 4 << 30) -> bool:
    """Whether the out-of-place step's second master/m/v/half set (14 bytes per
    owned element) fits in the device memory still free."""
    import torch
    torch.cuda.synchronize()
    return torch.cuda.mem_get_info()[0] > 14 * E + margin


def graph_steps_per_replay(step_bytes: float, steps: int, peak_gbs: float = 6781.0) -> int:
    """Steps captured in one CUDA graph: 1 while a step keeps the GPU busy far
    longer than the host takes to replay a graph (~12 us per replay from
    Python), else enough for ~0.5 ms of work per replay, at most 50, and a
    divisor of `steps` so that exactly `steps` steps are timed."""
    est_us = step_bytes / (peak_gbs * 1e3)
    if est_us >= 200.0:
        return 1
    want = min(50, max(1, int(500.0 / max(est_us, 1e-3))), steps)
    return next(r for r in range(want, 0, -1) if steps % r == 0)


def make_step(zs, ctx, W: DeviceWorkload, api: str, clip: float = 0.0, per_replay: int = 1):
    """One step of `api` on W's buffers; returns (step function, device state or
    None).  The graph forms capture `per_replay` consecutive steps, so their
    step function runs that many."""
    import torch
    wl, E = W.wl, W.E
    if api in ("async", "async_oop"):
        state = zs.DeviceState(W.scaler)
        calls = W.step_oop_calls if api == "async_oop" else W.step_async_calls

        def one_step():
            calls(ctx, state)
        return one_step, state
    if api in ("graph", "graph_oop"):
        state = zs.DeviceState(W.scaler)
        calls = W.step_oop_calls if api == "graph_oop" else W.step_async_calls
        calls(ctx, state)       # uncaptured first call caches launch shapes (and buffers)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for _ in range(per_replay):
                calls(ctx, state)
        return graph.replay, state
    if api == "sync":
        return (lambda: W.step(ctx)), None
    # split at the flag, as every rank of a multi-GPU run takes the step: the one
    # real exchange is the overflow flag, all-reduced on the device before any
    # state is written, so every rank skips together (with clipping, also the
    # shards' sums of squares, so every rank clips alike)
    from zero_mixed_precision_shard_gb300.dp import dp_shard_step, dp_shard_step_clipped
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    d_sumsq = torch.zeros(1, dtype=torch.float64, device="cuda")
    # the same re-read form (N < 4) or materialised form as zs_shard_step chooses
    recompute = wl.n < 4 or W.acc is None
    last = W.slices(wl.g - 1) if recompute else None
    acc_in = W.acc if (wl.g > 1 or not recompute) else None

    def reduce_last(f):
        f.zero_()
        for k in range(wl.g - 1):
            zs.zs_reduce_check(ctx, W.slices(k), W.dt, E, W.acc, k == 0, f)
        if recompute:
            zs.zs_check_last(ctx, W.slices(wl.g - 1), W.dt, E, acc_in, f)
        else:
            zs.zs_reduce_check(ctx, W.slices(wl.g - 1), W.dt, E, W.acc, wl.g == 1, f)

    def div():
        return float(wl.n * wl.g * W.scaler.scale)

    def apply(f):
        zs.zs_apply(ctx, f, last, W.dt, acc_in, E, div(), W.master, W.m, W.v, W.half, W.hp,
                    W.t + 1)

    def sumsq(d):
        zs.zs_grad_sumsq(ctx, last, W.dt, acc_in, E, div(), d)

    def apply_clipped(f, d):
        zs.zs_apply_clipped(ctx, f, d, clip, last, W.dt, acc_in, E, div(), W.master, W.m, W.v,
                            W.half, W.hp, W.t + 1)

    def scaler_update(f):
        ovf = zs.zs_scaler_update(ctx, f, W.scaler)
        if not ovf:
            W.t += 1
        return ovf

    def one_step():
        if clip:
            return dp_shard_step_clipped(reduce_last, sumsq, apply_clipped, scaler_update, flag,
                                         d_sumsq)
        return dp_shard_step(reduce_last, apply, scaler_update, flag)
    return one_step, None


def kernel_table(zs, ctx, plan):
    """Per-kernel event times of the timed region, with algorithmic GB/s."""
    kinds = {}
    for kind_id, name in enumerate(zs.KERNEL_NAMES):
        tot, nl, el = ctx.timing(kind_id)
        if nl:
            kinds[name] = {"ms": tot, "launches": nl, "elements": el}
    alg_bytes = {}
    for name, b in plan:
        alg_bytes.setdefault(name, []).append(b)
    for name, d in kinds.items():
        per_launch = alg_bytes.get(name, [0])
        avg_b = sum(per_launch) / len(per_launch) if per_launch else 0
        d["alg_bytes_per_elem"] = avg_b
        d["gbs"] = avg_b * (d["elements"] / d["launches"]) / (d["ms"] / d["launches"] * 1e-3) / 1e9
    return kinds


def timed_steps(ctx, one_step, steps: int, warmup: int, dev: int, world: int,
                kernel_timing: bool = True, per_call: int = 1):
    """W untimed steps, then K steps between CUDA events on the launching
    stream, bracketed by a barrier and device synchronisation, with per-kernel
    event timing (unless kernel_timing is False) and nvidia-smi clock samples
    during the timed region.  one_step runs `per_call` steps (a graph of
    several steps): W is rounded up to whole calls, K must be whole calls."""
    import torch
    import torch.distributed as dist
    if steps % per_call:
        raise ValueError(f"{steps} steps are not whole calls of {per_call}")
    for _ in range(-(-warmup // per_call)):
        one_step()
    torch.cuda.synchronize()
    ctx.timing_reset()
    ctx.set_timing(kernel_timing)
    l0 = ctx.launch_count
    with ClockSampler(dev) as clocks:
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ev0.record()
        for _ in range(steps // per_call):
            one_step()
        ev1.record()
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
    ctx.set_timing(False)
    return ev0.elapsed_time(ev1), ctx.launch_count - l0, clocks.summary()


def measure_table_workload(zs, ctx, name: str, args, peak: float, dev: int):
    """One more target workload in the same run: its own buffers, warm-up,
    timed steps and clock record, through the default API and the
    synchronising one (truncated like the headline workload under --elements)."""
    import torch
    wl = synth.WORKLOADS[name]
    W = DeviceWorkload(wl, shard=0, count=args.elements, grad_buffers=2)
    W.fill_grads(1, wl.scale0, inject=False)
    torch.cuda.synchronize()
    valid = min(W.valid_end - W.begin, W.E)
    step_bytes = alg_bytes_per_elem_step(wl.n, wl.g) * W.E
    out = {"workload": name + (f" (first {W.E} elements)" if args.elements else ""),
           "params": wl.psi, "owned_params": valid, "shard_len": W.E, "n_ranks_simulated": wl.n,
           "accum_steps": wl.g, "grad_dtype": wl.dtype, "alg_bytes_per_step": step_bytes}
    # these steps take 0.3-2.5 ms: at least 100 of them, so that one stall of the
    # host (which the synchronising API waits on every step) cannot dominate
    steps = max(args.steps, 100)
    for api in ("async", "async_oop", "sync", "graph_oop"):
        # a graph of several steps where one step is shorter than the host's
        # replay call (the step's GPU rate, not the host's)
        per = graph_steps_per_replay(step_bytes, steps) if api == "graph_oop" else 1
        one_step, state = make_step(zs, ctx, W, api, per_replay=per)
        # the step rate without per-kernel events (an event pair around each of
        # a short step's launches costs it a few percent), then the same steps
        # again with them for the per-kernel rates (none inside a graph replay)
        ms, launches, clocks = timed_steps(ctx, one_step, steps, args.warmup, dev, 1,
                                           kernel_timing=False, per_call=per)
        timed_steps(ctx, one_step, steps, 0, dev, 1, per_call=per)
        per_step = ms / steps
        gbs = step_bytes / (per_step * 1e-3) / 1e9
        oop = api in ("async_oop", "graph_oop")
        plan = W.launch_plan(oop=oop, fused=W.takes_fused(ctx, "async_oop" if oop else api))
        if api == "graph_oop":   # replays bypass the context's launch counter
            launches = steps * (len(plan) + (0 if W.takes_fused(ctx, "async_oop") else 2))
        kinds = kernel_table(zs, ctx, plan)
        out[api] = {"api": API_DESC[api], "value": valid / (per_step * 1e-3), "unit": "params/s",
                    "steps": steps, "ms_per_step": round(per_step, 6), "step_gbs": round(gbs, 1),
                    "step_frac_of_peak": round(gbs / peak, 4), "gpu_launches": launches,
                    "warmup_steps": -(-args.warmup // per) * per, "clocks": clocks,
                    "kernels": {k: {"gbs": round(d["gbs"], 1), "frac_of_peak":
                                    round(d["gbs"] / peak, 4), "launches": d["launches"]}
                                for k, d in kinds.items()}}
        if per > 1:
            out[api]["steps_per_replay"] = per
        if state is not None:
            d = state.read()
            out[api]["device_state"] = {"iterations": d.iterations, "step": d.step,
                                        "scale": d.scaler.scale}
    del W
    torch.cuda.empty_cache()
    return out


class Zero2Workload:
    """One real rank of a ZeRO-2 job over the workload's flat parameter buffer
    (its first `count` parameters with --elements): the buffer is partitioned
    over the job's ranks, this rank holds its own full flat fp16/bf16 gradient
    of every micro-step (synthetic, seeded by its rank), its shard's fp32
    accumulator, master, m and v, its shard's half copy and the full half
    parameter buffer that the all-gather rebuilds."""

    def __init__(self, zs, ctx, wl: synth.Workload, world: int, rank: int, count=None,
                 clip: float = 0.0):
        import torch
        from zero_mixed_precision_shard_gb300.dp import Zero2Step, ZsShardOps
        self.wl, self.world, self.rank = wl, world, rank
        psi = wl.psi if count is None else count
        self.part = zs.zs_init_partition(psi, world, synth.ALIGN_ELEMS)
        self.psi = psi
        P, E = self.part.psi_pad, self.part.shard_len
        self.E = E
        b, ve, _ = zs.zs_shard_range(self.part, rank)
        self.valid = ve - b
        dev = torch.device("cuda", torch.cuda.current_device())
        s = torch.cuda.current_stream().cuda_stream
        self.grads = torch.empty((wl.g, P), dtype=torch.int16, device=dev)
        for k in range(wl.g):
            synth.dev_fill_grads(self.grads[k].data_ptr(), P, 0, wl, 1, k + 1, rank, wl.scale0,
                                 s, inject=False)
            self.grads[k, psi:].zero_()
        self.acc = torch.empty(E, dtype=torch.float32, device=dev)
        self.master = torch.empty(E, dtype=torch.float32, device=dev)
        synth.dev_fill_master(self.master.data_ptr(), E, b, wl, s)
        if ve - b < E:
            self.master[max(ve - b, 0):].zero_()
        self.m = torch.zeros(E, dtype=torch.float32, device=dev)
        self.v = torch.zeros(E, dtype=torch.float32, device=dev)
        self.half_shard = torch.zeros(E, dtype=torch.int16, device=dev)
        self.half_full = torch.zeros(P, dtype=torch.int16, device=dev)
        self.scaler = zs.zs_scaler_init(wl.scale0, wl.min_scale, wl.window, wl.hysteresis,
                                        wl.dynamic)
        hp = zs.make_hparams(wl.lr, wl.beta1, wl.beta2, wl.eps, wl.weight_decay)
        # unclipped steps apply the last micro-step out of place, bucket by bucket,
        # where the second master/m/v/half set (14 B per shard element) fits
        second = None
        self.oop = clip <= 0 and oop_fits(E)
        if self.oop:
            p2 = torch.zeros(E, dtype=torch.float32, device=dev)
            second = (p2, torch.zeros_like(p2), torch.zeros_like(p2),
                      torch.zeros(E, dtype=torch.int16, device=dev))
        self.ops = ZsShardOps(zs, ctx, wl.dtype_code, E, world, wl.g, self.acc, self.master,
                              self.m, self.v, self.half_shard, hp, self.scaler, clip,
                              second=second)
        bucket = wl.bucket_elems
        # two receive slots: the next bucket's exchange overlaps this one's sum
        self.recv = torch.empty(2 * world * min(E, bucket // 64 * 64), dtype=torch.int16,
                                device=dev)
        self.flag = torch.zeros(1, dtype=torch.int32, device=dev)
        self.step_obj = Zero2Step(self.ops, P, E, rank, bucket, self.recv, self.flag,
                                  torch.zeros(1, dtype=torch.float64, device=dev))
        self.clip = clip

    def step(self):
        return self.step_obj.step([self.grads[k] for k in range(self.wl.g)], self.half_full,
                                  clip=self.clip > 0)

    def launch_plan(self):
        """(kind, alg bytes per element of the shard) of every kernel a step launches:
        per micro-step the accumulate of the received slices (split by bucket),
        the update from the accumulator (and the norm pass when clipping); out of
        place, the last micro-step's buckets are summed and applied in one pass."""
        n, g = self.world, self.wl.g
        if self.oop:
            return step_launch_plan(n, g, self.wl.dtype, oop=True)
        plan = [("reduce_first" if k == 0 else "reduce",
                 kernel_alg_bytes("reduce", n, first=(k == 0))) for k in range(g)]
        if self.clip > 0:
            plan.append(("sumsq", kernel_alg_bytes("sumsq", n, with_acc=True)))
        plan.append(("apply", kernel_alg_bytes("apply", n)))
        return plan


def run_zero2(args, zs, ctx, wl, world: int, rank: int, dev: int, probe):
    """N > 1: the ZeRO-2 step with its real exchanges on every rank."""
    import torch
    import torch.distributed as dist
    Z = Zero2Workload(zs, ctx, wl, world, rank, args.elements, args.clip)
    torch.cuda.synchronize()
    ms, launches, clock_summary = timed_steps(ctx, Z.step, args.steps, args.warmup, dev, world)
    kinds = kernel_table(zs, ctx, Z.launch_plan())
    t = torch.tensor([ms], dtype=torch.float64, device="cuda")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    ms = float(t.item())
    n_l = torch.tensor([launches], dtype=torch.int64, device="cuda")
    dist.all_reduce(n_l)
    launches = int(n_l.item())
    per_step_ms = ms / args.steps
    value = Z.psi / (per_step_ms * 1e-3)        # every rank's owned params over the slowest step
    xb = Z.step_obj.exchanged_bytes(wl.g)
    # + the materialised last micro-step unless it is applied out of place
    shard_bytes = (alg_bytes_per_elem_step(world, wl.g) + (0 if Z.oop else 8)) * Z.E
    peak, peak_kind = measured_peaks()
    dom = max(kinds, key=lambda k: kinds[k]["ms"]) if kinds else None
    roofline = None
    if dom is not None:
        per_launch_elems = kinds[dom]["elements"] / kinds[dom]["launches"]
        roofline = {"bound": "hbm", "kernel": dom, "achieved": round(kinds[dom]["gbs"], 1),
                    "peak": peak, "unit": "GB/s", "frac": round(kinds[dom]["gbs"] / peak, 4),
                    "traffic": None, "traffic_unit": "bytes per launch",
                    "alg_bytes_per_launch": kinds[dom]["alg_bytes_per_elem"] * per_launch_elems,
                    "peak_source": f"MEASURED_PEAKS.json hbm_gbs ({peak_kind})"}
    e2e = None
    if not args.skip_e2e:
        dist.barrier()
        e2e = run_e2e_zero2(Z, args.e2e_steps)
        t = torch.tensor([e2e["ms_per_step"]], dtype=torch.float64, device="cuda")
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        e2e["ms_per_step"] = float(t.item())
        e2e["value"] = Z.psi / (e2e["ms_per_step"] * 1e-3)
        e2e["h2d_bytes_per_step"] *= world
        e2e["d2h_bytes_per_step"] *= world
    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "params/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": per_step_ms,
            "higher_is_better": True, "scaling": "strong", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic",
            "config": {
                "workload": wl.name + (f" (first {Z.psi} parameters)" if args.elements else ""),
                "params": Z.psi, "shard_len": Z.E, "accum_steps": wl.g, "grad_dtype": wl.dtype,
                "optimizer": "AdamW" if wl.weight_decay else "Adam",
                "parallelism": f"ZeRO-2 dp{world}: per micro-step an all-to-all of each "
                               f"{wl.bucket_elems}-element gradient bucket's shard slices "
                               "(rank q receives every rank's slice of shard q), fp32 "
                               "rank-ordered sum in the reduce kernel; flag MAX"
                               + (" + norm SUM" if args.clip else "")
                               + " all-reduce; update; all-gather of the half copy",
                "dist_backend": args.dist_backend,
                "clip_max_norm": args.clip or None,
                "api": "dp.Zero2Step over zs_reduce_check, "
                       + ("zs_update_oop (the last micro-step per bucket, out of place)"
                          if Z.oop else "zs_apply"
                          + ("_clipped + zs_grad_sumsq" if args.clip else ""))
                       + ", zs_scaler_update",
                "exchange_bytes_per_rank_per_step": xb,
                "shard_alg_bytes_per_step": shard_bytes,
                "l2": "inputs larger than L2 (129 MB): no flush needed",
                "inputs": "every rank's full gradients generated once on the device (step-1 "
                          "values of its rank, no injections) and reused by every timed step",
                "copy_probe_gbs": probe,
                "kernels": {k: {kk: (round(vv, 4) if isinstance(vv, float) else vv)
                                for kk, vv in d.items()} for k, d in kinds.items()},
            },
            "roofline": roofline,
            "clocks": clock_summary,
            "gpu_launches": launches,
            "e2e": e2e,
            "cpu_baseline": None,
        }
        print(json.dumps(line), flush=True)
    ctx.close()
    dist.destroy_process_group()
    return 0


def run_e2e_zero2(Z: Zero2Workload, steps: int):
    """The ZeRO-2 step with every micro-step's full flat gradient copied in
    from pinned host memory first, and the step's result (the overflow flag
    the loss-scale update returns) read by the host."""
    import torch
    host = torch.empty(Z.grads.shape[1], dtype=Z.grads.dtype, pin_memory=True)
    host.copy_(Z.grads[0])   # device -> pinned host directly (no pageable copy)
    copy_stream = torch.cuda.Stream()
    compute = torch.cuda.current_stream()

    def step():
        ev = []
        for k in range(Z.wl.g):
            with torch.cuda.stream(copy_stream):
                copy_stream.wait_stream(compute)
                Z.grads[k].copy_(host, non_blocking=True)
                e = torch.cuda.Event()
                e.record(copy_stream)
                ev.append(e)
        for e in ev:
            compute.wait_event(e)
        return Z.step()

    step()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(steps):
        step()
    b.record()
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / steps
    h2d = Z.wl.g * Z.grads.shape[1] * 2
    return {"value": Z.psi / (ms * 1e-3), "unit": "params/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": 8, "ms_per_step": ms, "steps": steps}


def run_ours(args):
    import torch
    import torch.distributed as dist

    import zero_mixed_precision_shard_gb300 as zs

    world, rank, local = dist_env()
    # one rank per GPU; --dist-backend gloo lets several ranks share one GPU (the
    # exchanges then go through host memory, and no kernel waits on another rank)
    dev = local % torch.cuda.device_count()
    torch.cuda.set_device(dev)
    if world > 1:
        if args.dist_backend == "nccl":
            dist.init_process_group("nccl", device_id=torch.device("cuda", dev))
        else:
            dist.init_process_group("gloo")
    wl = synth.WORKLOADS[args.workload]
    ctx = zs.Ctx()
    probe = copy_probe(zs, ctx) if not args.skip_probe else {}
    if world > 1:
        if args.acc != "fp32" or args.graph or args.split:
            raise SystemExit("N > 1 runs the ZeRO-2 step with the fp32 accumulator")
        return run_zero2(args, zs, ctx, wl, world, rank, dev, probe)
    api = resolve_api(args, world)
    if api == "split" and args.acc != "fp32":
        raise SystemExit("--acc half runs the fused step on one GPU")
    if args.split and args.graph:
        raise SystemExit("--split and --graph are separate modes")
    if api == "graph" and args.acc != "fp32":
        raise SystemExit("--graph runs the fp32-accumulator path on one GPU")
    if api == "async_oop" and args.clip:
        raise SystemExit("--api async_oop runs the unclipped step")

    # two gradient buffers alternate across the micro-steps (the split form reads
    # every micro-step's slices in one call, so it keeps one buffer each)
    W = DeviceWorkload(wl, shard=0, count=args.elements, acc=args.acc, clip=args.clip,
                       grad_buffers=None if api == "split" else 2)
    W.fill_grads(1, wl.scale0, inject=False)
    torch.cuda.synchronize()
    if api == "auto":
        api = "async_oop" if oop_fits(W.E) else "async"
    # the synchronising half-accumulator step out of place where its second
    # state set fits (the device-resident forms name their own form in `api`)
    hacc_oop = W.hacc_oop = args.acc == "half" and api == "sync" and oop_fits(W.E)
    E = W.E
    valid = min(W.valid_end - W.begin, E)
    # a graph of several steps where one step is shorter than the host's replay
    per = (graph_steps_per_replay(alg_bytes_per_elem_step(wl.n, wl.g) * E, args.steps)
           if api == "graph" else 1)
    one_step, state = make_step(zs, ctx, W, api, args.clip, per_replay=per)
    ms, launches, clock_summary = timed_steps(ctx, one_step, args.steps, args.warmup, dev, world,
                                              per_call=per)
    fused = W.takes_fused(ctx, api)
    plan = W.launch_plan(split=api == "split", oop=api == "async_oop" or hacc_oop, fused=fused)
    if api == "graph":  # replays bypass the context's counter: the kernels of a captured step
        # (the streaming ones, the prologue and the flag reset; with clipping the
        # norm's finalize and the coefficient, and the fold of many partials;
        # the fused step is one kernel)
        extra = 0 if fused else 2 + (2 + (1 if W.E // (8 * 256) > 4096 else 0) if args.clip
                                     else 0)
        launches = args.steps * (len(plan) + extra)
    dstate = None
    if state is not None:
        d = state.read()
        dstate = {"iterations": d.iterations, "step": d.step, "scale": d.scaler.scale,
                  "overflow": d.overflow}
    if world > 1:   # every rank's launches
        n_l = torch.tensor([launches], dtype=torch.int64, device="cuda")
        dist.all_reduce(n_l)
        launches = int(n_l.item())
        t = torch.tensor([ms], dtype=torch.float64, device="cuda")
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
    per_step_ms = ms / args.steps
    owned_total = valid
    if world > 1:
        v = torch.tensor([valid], dtype=torch.float64, device="cuda")
        dist.all_reduce(v)
        owned_total = int(v.item())
    value = owned_total / (per_step_ms * 1e-3)

    # per-kernel times and the dominant kernel's roofline
    kinds = kernel_table(zs, ctx, plan)
    step_bytes = alg_bytes_per_elem_step(wl.n, wl.g, 2 if args.acc == "half" else 4) * E
    if not kinds:  # graph replay: no per-kernel events inside the graph
        kinds = {"step": {"ms": ms, "launches": args.steps, "elements": E * args.steps,
                          "alg_bytes_per_elem": step_bytes / E}}
        kinds["step"]["gbs"] = step_bytes / (per_step_ms * 1e-3) / 1e9
    dom = max(kinds, key=lambda k: kinds[k]["ms"])
    peak, peak_kind = measured_peaks()
    per_launch_elems = kinds[dom]["elements"] / kinds[dom]["launches"]
    traffic = recorded_traffic(wl.name, dom, per_launch_elems) if not args.elements else None
    roofline = {"bound": "hbm", "kernel": dom, "achieved": round(kinds[dom]["gbs"], 1),
                "peak": peak, "unit": "GB/s", "frac": round(kinds[dom]["gbs"] / peak, 4),
                "traffic": traffic, "traffic_unit": "bytes per launch",
                "alg_bytes_per_launch": kinds[dom]["alg_bytes_per_elem"] * per_launch_elems,
                "peak_source": f"MEASURED_PEAKS.json hbm_gbs ({peak_kind})"}

    # end to end: gradients copied from pinned host memory every micro-step
    e2e = None
    if not args.skip_e2e:
        if world > 1:
            dist.barrier()
        e2e = run_e2e(zs, ctx, W, args.e2e_steps, api,
                      step_fn=one_step if api == "split" else None)
        if world > 1:  # whole job: every rank's params over the slowest rank's step
            t = torch.tensor([e2e["ms_per_step"]], dtype=torch.float64, device="cuda")
            dist.all_reduce(t, op=dist.ReduceOp.MAX)
            e2e["ms_per_step"] = float(t.item())
            e2e["value"] = owned_total / (e2e["ms_per_step"] * 1e-3)
            e2e["h2d_bytes_per_step"] *= world
            e2e["d2h_bytes_per_step"] *= world
            e2e["h2d_gbs"] = round(e2e["h2d_bytes_per_step"] / (e2e["ms_per_step"] * 1e-3) / 1e9,
                                   1)

    # the other target workloads, each with its own clock record (one GPU only)
    table = None
    inputs_desc = ("gradients generated once on the device (step-1 values, no injections) and "
                   "reused by every timed step; "
                   + (f"{W.nbuf} gradient buffers alternate across the {wl.g} micro-steps, each "
                      "micro-step reading its N slices from HBM" if W.nbuf < wl.g
                      else "one gradient buffer per micro-step"))
    if (world == 1 and not args.skip_table and args.workload == DEFAULT_WORKLOAD
            and args.api == "auto" and api in ("async", "async_oop") and not args.clip):
        del W, one_step, state
        torch.cuda.empty_cache()
        table = {name: measure_table_workload(zs, ctx, name, args, peak, dev)
                 for name in TABLE_WORKLOADS}

    cpu = None
    if rank == 0 and world == 1 and not args.skip_cpu:
        cpu = cpu_baseline(wl)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "params/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": per_step_ms,
            # the same model at every N: N > 1 partitions it over the ranks (ZeRO-2)
            "higher_is_better": True, "scaling": "strong", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic",
            "config": {
                "workload": wl.name + (f" (first {E} elements)" if args.elements else ""),
                "params": wl.psi, "owned_params": valid,
                "shard_len": E, "n_ranks_simulated": wl.n, "accum_steps": wl.g,
                "grad_dtype": wl.dtype, "optimizer": "AdamW" if wl.weight_decay else "Adam",
                "parallelism": ("replicas + overflow-flag all-reduce"
                                + (" + norm all-reduce" if args.clip else "")) if world > 1
                               else "1 GPU",
                "accumulator": args.acc,
                "clip_max_norm": args.clip or None,
                "api": api_desc(api, args.acc, args.clip, hacc_oop),
                # graph replays of several steps each (warm-up rounded up to whole replays)
                **({"steps_per_replay": per, "warmup_steps_run": -(-args.warmup // per) * per}
                   if per > 1 else {}),
                "l2": "inputs larger than L2 (129 MB): no flush needed",
                "inputs": inputs_desc,
                "alg_bytes_per_step": step_bytes,
                "step_gbs": round(step_bytes / (per_step_ms * 1e-3) / 1e9, 1),
                "step_frac_of_peak": round(step_bytes / (per_step_ms * 1e-3) / 1e9 / peak, 4),
                "copy_probe_gbs": probe,
                "device_state_after_timed_steps": dstate,
                "kernels": {k: {kk: (round(vv, 4) if isinstance(vv, float) else vv)
                                for kk, vv in d.items()} for k, d in kinds.items()},
                "workloads": table,
            },
            "achieved_gbs": round(step_bytes / (per_step_ms * 1e-3) / 1e9, 1),
            "achieved_frac_of_peak": round(step_bytes / (per_step_ms * 1e-3) / 1e9 / peak, 4),
            "roofline": roofline,
            "clocks": clock_summary,
            "gpu_launches": launches,
            "e2e": e2e,
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)
    ctx.close()
    if world > 1:
        dist.destroy_process_group()
    return 0


def run_e2e(zs, ctx, W: DeviceWorkload, steps: int, api: str = "sync", step_fn=None):
    """Same step, but every micro-step's N gradient slices are first copied
    from pinned host memory (the values a backward pass would hand over), and
    each step's result is read back: on the device-resident path an
    asynchronous copy of the step state (flag, scale, step count) into pinned
    host memory, on the synchronising path the flag and scale the step call
    returns.  Copies run on a side stream, one micro-step ahead of the
    compute.  step_fn (the step split at the flag, as each rank of a
    multi-GPU run takes it) instead waits for all G copies, then runs."""
    import torch
    wl = W.wl
    nb = W.nbuf
    host = torch.empty((wl.n, W.E), dtype=torch.int16, pin_memory=True)
    host.copy_(W.grads[0])   # device -> pinned host directly (no pageable copy)
    copy_stream = torch.cuda.Stream()
    compute = torch.cuda.current_stream()
    done = [torch.cuda.Event() for _ in range(nb)]   # buffer b filled
    free = [torch.cuda.Event() for _ in range(nb)]   # buffer b consumed
    state = zs.DeviceState(W.scaler) if api in ("async", "async_oop", "graph") else None
    result = torch.empty(64, dtype=torch.uint8, pin_memory=True)

    def copy_in(k):
        b = k % nb
        with torch.cuda.stream(copy_stream):
            copy_stream.wait_event(free[b])
            W.grads[b].copy_(host, non_blocking=True)
            done[b].record(copy_stream)
        return b

    def step():
        if step_fn is not None:   # every micro-step has its own buffer here
            for k in range(wl.g):
                copy_in(k)
            for b in range(nb):
                compute.wait_event(done[b])
            step_fn()
            for b in range(nb):
                free[b].record(compute)
            return
        # micro-step k's copy waits only for the micro-step that last read its
        # buffer, so it runs while the compute stream reduces micro-step k-1
        for k in range(wl.g):
            b = copy_in(k)
            compute.wait_event(done[b])
            if k < wl.g - 1:
                W.accum(ctx, k)
            elif state is not None:
                (W.finish_oop if api == "async_oop" else W.finish_async)(ctx, state)
                result.copy_(state.buf, non_blocking=True)
            else:
                W.finish(ctx)
            free[b].record(compute)

    for e in free:
        e.record(compute)
    step()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(steps):
        step()
    b.record()
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / steps
    valid = min(W.valid_end - W.begin, W.E)
    h2d = wl.g * wl.n * W.E * 2
    d2h = result.numel() if state is not None else 8
    out = {"value": valid / (ms * 1e-3), "unit": "params/s", "h2d_bytes_per_step": h2d,
           "d2h_bytes_per_step": d2h, "ms_per_step": ms, "steps": steps,
           "h2d_gbs": round(h2d / (ms * 1e-3) / 1e9, 1),
           "wall_s": round(time.perf_counter() - t0, 2)}
    if state is not None:
        d = zs.zs_device_state.from_buffer_copy(result.numpy().tobytes())
        out["last_result"] = {"iterations": d.iterations, "overflow": d.overflow,
                              "scale": d.scaler.scale}
        assert d.iterations == steps + 1, "the step results read back are not the last step's"
    return out


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="zeroshard", choices=["zeroshard", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(synth.WORKLOADS))
    ap.add_argument("--e2e-steps", type=int, default=3)
    ap.add_argument("--skip-e2e", action="store_true")
    ap.add_argument("--skip-cpu", action="store_true")
    ap.add_argument("--skip-probe", action="store_true")
    ap.add_argument("--acc", default="fp32", choices=["fp32", "half"],
                    help="accumulator format (half: zs_*_halfacc entry points)")
    ap.add_argument("--clip", type=float, default=0.0,
                    help="global-norm gradient clipping at this max norm (zs_shard_step_clipped)")
    ap.add_argument("--api", default="auto", choices=["auto", "async", "async_oop", "sync"],
                    help="auto (default): async_oop where its second state set fits in HBM, "
                         "else async; async: zs_shard_step_async with the scale and step count "
                         "on the device, no host round trip per step; async_oop: the same with "
                         "the state written out of place (one pass for the last micro-step and "
                         "the update); sync: zs_shard_step, which returns the flag and scale to "
                         "the host every step")
    ap.add_argument("--skip-table", action="store_true",
                    help="skip the other target workloads measured after the headline one")
    ap.add_argument("--graph", action="store_true",
                    help="replay each step from a CUDA graph (device-resident scaler)")
    ap.add_argument("--split", action="store_true",
                    help="run the step split at the overflow flag, as a caller that exchanges "
                         "the flag between ranks does (zs_reduce_check / zs_check_last, "
                         "zs_apply, zs_scaler_update), instead of the fused call")
    ap.add_argument("--dist-backend", default="nccl", choices=["nccl", "gloo"],
                    help="process group of a multi-GPU (ZeRO-2) run (gloo: ranks may share a "
                         "GPU, the exchanges staged through host memory, for testing the "
                         "multi-rank path on one)")
    ap.add_argument("--elements", type=int, default=None,
                    help="truncate the owned shard to its first ELEMENTS elements (profiling)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
