"""Data-parallel orchestration of the shard step across real ranks.

With one process per GPU, each rank owns one contiguous shard of the flat
parameter buffer (ZeRO-1/2: DeepSpeed Complete Guide, §2.1 and §2.2) and
must skip or apply the step together with every other rank: an overflow seen
by any rank skips the step everywhere and lowers every rank's loss scale
identically (§4.2).

Two levels live here.

dp_shard_step / dp_shard_step_clipped: the step of one shard whose rank
slices are already on this GPU, split at the overflow flag; the exchange they
add is a MAX all-reduce of the int32 flag (and, with clipping, a SUM of the
shards' squared norms) between the reduce/check phase and the update.

Zero2Step: the whole ZeRO-2 step of a rank that holds its own full flat
gradient per micro-step.  Per micro-step the flat gradient travels in
contiguous buckets of at most reduce_bucket_size elements (§2.2 and its
config block); the part of a bucket that falls in shard q goes to rank q, so
rank q receives every rank's slice of its own shard, in rank order, and sums
them in fp32 onto its accumulator with the library's reduce kernel.  This
all-to-all of half slices moves the bytes a ring reduce-scatter moves, while
the sum stays the sequential rank-ordered fp32 sum of the single-GPU path (a
reduce-scatter in the wire format would add in half precision, in an order
the library does not fix).  After the micro-steps: the flag's MAX, the norm's
SUM when clipping, the update of the owned shard, the loss-scale update, and
on an applied step the all-gather that rebuilds every rank's full half
parameter buffer (§2.1).  The collectives are torch.distributed calls (NCCL on
GPUs); every byte of arithmetic runs in the library's kernels.
"""
from __future__ import annotations

from dataclasses import dataclass


def _dist():
    import torch.distributed as dist
    return dist


def _world(group=None) -> int:
    dist = _dist()
    if dist.is_available() and dist.is_initialized():
        return dist.get_world_size(group)
    return 1


def dp_shard_step(reduce_last, apply, scaler_update, flag, group=None) -> int:
    """Run one step of this rank's shard.

    reduce_last(flag): OR this rank's overflow of the step into `flag` (a
        one-element int32 tensor; it arrives holding 0 or the OR of earlier
        micro-steps).
    apply(flag): the update, which writes nothing if flag != 0.
    scaler_update(flag) -> int: the loss-scale update; returns the overflow.
    Every rank must call this once per step, in the same order."""
    dist = _dist()
    reduce_last(flag)
    if _world(group) > 1:
        dist.all_reduce(flag, op=dist.ReduceOp.MAX, group=group)
    apply(flag)
    return scaler_update(flag)


def dp_shard_step_clipped(reduce_last, sumsq, apply_clipped, scaler_update, flag, d_sumsq,
                          group=None) -> int:
    """dp_shard_step with global-norm clipping (§4.1 gradient_clipping, §5.1).
    The norm is over the whole model, so each rank's sum of squares of its
    shard's mean gradient is added across ranks (a SUM all-reduce of one
    float64) beside the MAX all-reduce of the flag, and every rank clips with
    the same coefficient.

    sumsq(d_sumsq): write this rank's sum of squares into `d_sumsq` (a
        one-element float64 tensor), e.g. zs_grad_sumsq.
    apply_clipped(flag, d_sumsq): the update from the global sum (e.g.
        zs_apply_clipped), which writes nothing if flag != 0."""
    dist = _dist()
    reduce_last(flag)
    sumsq(d_sumsq)
    if _world(group) > 1:
        dist.all_reduce(flag, op=dist.ReduceOp.MAX, group=group)
        dist.all_reduce(d_sumsq, op=dist.ReduceOp.SUM, group=group)
    apply_clipped(flag, d_sumsq)
    return scaler_update(flag)


# ---------------------------------------------------------------- ZeRO-2

@dataclass(frozen=True)
class Bucket:
    """One bucket of the flat gradient, [x0, x1), as this rank exchanges it:
    send[q] elements of it go to rank q (its overlap with shard q), and this
    rank receives `length` elements from every rank, landing at `offset` of
    its own shard (length 0 when the bucket misses the shard)."""
    x0: int
    x1: int
    send: tuple
    offset: int
    length: int


def bucket_plan(psi_pad: int, shard_len: int, world: int, rank: int, bucket_elems: int):
    """Cut the flat padded buffer [0, psi_pad) into contiguous buckets of at
    most bucket_elems elements (§2.2 reduce_bucket_size) and describe each
    bucket's exchange for `rank`.  Buckets are cut at multiples of 64
    elements (bucket_elems is rounded down to one; shards are multiples of
    64 already), so every received slice and accumulator range stays 16-byte
    aligned.  Pure host arithmetic."""
    bucket_elems = bucket_elems // 64 * 64
    if bucket_elems < 64 or world < 1 or psi_pad != shard_len * world or shard_len % 64:
        raise ValueError("bad bucket plan arguments")
    lo, hi = rank * shard_len, (rank + 1) * shard_len
    plan = []
    for x0 in range(0, psi_pad, bucket_elems):
        x1 = min(x0 + bucket_elems, psi_pad)
        send = tuple(max(0, min(x1, (q + 1) * shard_len) - max(x0, q * shard_len))
                     for q in range(world))
        a, b = max(x0, lo), min(x1, hi)
        plan.append(Bucket(x0, x1, send, max(0, a - lo), max(0, b - a)))
    return plan


class Exchange:
    """The collectives of the ZeRO-2 step on byte views of the buffers.

    NCCL moves device buffers directly.  gloo has no all-to-all of device
    buffers, so with gloo device buffers are staged through host memory (the
    path that lets several ranks share one GPU in tests: no kernel then waits
    on another rank)."""

    def __init__(self, group=None):
        dist = _dist()
        self.group = group
        self.dist = dist
        self.world = _world(group)
        # with a process group every exchange is a collective, one rank included
        # (a one-rank NCCL group runs the same calls); without one they are copies
        self.active = dist.is_available() and dist.is_initialized()
        self.staged = self.active and dist.get_backend(group) == "gloo"

    @staticmethod
    def _bytes(t):
        import torch
        if not t.is_contiguous():
            raise ValueError("exchanged buffers must be contiguous")
        return t.view(torch.uint8) if t.dtype != torch.uint8 else t

    def all_to_all(self, out, inp, out_splits, in_splits, async_op: bool = False):
        """out: `sum(out_splits)` elements received in rank order; inp: `sum(in_splits)`
        elements, in_splits[q] of them for rank q (16-bit elements).  With
        async_op (device buffers, not staged) returns the collective's work
        handle: its wait() orders the current stream after the transfer."""
        if not self.active:
            out.copy_(inp)
            return None
        item = inp.element_size()
        ob, ib = self._bytes(out), self._bytes(inp)
        osz = [x * item for x in out_splits]
        isz = [x * item for x in in_splits]
        if not self.staged or not out.is_cuda:
            return self.dist.all_to_all_single(ob, ib, osz, isz, group=self.group,
                                               async_op=async_op)
        ho = ob.cpu()
        self.dist.all_to_all_single(ho, ib.cpu(), osz, isz, group=self.group)
        ob.copy_(ho)

    def all_gather(self, out, inp):
        """out = every rank's `inp`, concatenated in rank order."""
        if not self.active:
            out.copy_(inp)
            return None
        ob, ib = self._bytes(out), self._bytes(inp)
        if not self.staged or not out.is_cuda:
            return self.dist.all_gather_into_tensor(ob, ib, group=self.group)
        ho = ob.cpu()
        self.dist.all_gather_into_tensor(ho, ib.cpu(), group=self.group)
        ob.copy_(ho)

    def all_reduce(self, t, op: str):
        if not self.active:
            return None
        o = self.dist.ReduceOp.MAX if op == "max" else self.dist.ReduceOp.SUM
        if not self.staged or not t.is_cuda:
            return self.dist.all_reduce(t, op=o, group=self.group)
        h = t.cpu()
        self.dist.all_reduce(h, op=o, group=self.group)
        t.copy_(h)


class Zero2Step:
    """One rank's ZeRO-2 optimizer step over its own full flat gradients.

    ops: the local compute of this rank's shard, an object with
      accumulate(rows, offset, length, first, flag): acc[offset:offset+length]
          = (first ? 0 : acc[...]) + rows[0] + ... + rows[world-1] in fp32, in
          rank order, OR-ing any non-finite sum into flag;
      sumsq(d_sumsq): the squared norm of the shard's mean gradient;
      apply(flag, d_sumsq): the update from acc (clipped when d_sumsq is not
          None), writing nothing if flag != 0;
      scaler_update(flag) -> int: the loss-scale update; returns the overflow;
      half_shard: this rank's half copy of its shard (the all-gather's input).
    Ops that hold a second state set (oop = True) also provide
      update_oop(rows, offset, length, flag): the last micro-step's sums of a
          range (acc, or +0 when G = 1, + the rows in rank order), the flag,
          and the update from the current set into the other one, written
          whatever the flag;
      commit_oop(flag) -> int: the loss-scale update; on a clean step the
          written set becomes current.  Returns the overflow.
    Unclipped steps then take the last micro-step out of place, bucket by
    bucket as the exchange delivers it: the sum is never written back, and no
    pass over the shard follows the exchange (the clipping norm needs every
    final sum before the update, so clipped steps materialise).
    The library's kernels are the ops on GPUs (ZsShardOps); the tests also
    drive this choreography with the oracle as the ops, on CPU."""

    def __init__(self, ops, psi_pad: int, shard_len: int, rank: int, bucket_elems: int,
                 recv, flag, d_sumsq=None, exchange: Exchange | None = None):
        self.ops = ops
        self.x = exchange or Exchange()
        self.world = self.x.world
        self.rank = rank
        self.E = shard_len
        self.plan = bucket_plan(psi_pad, shard_len, self.world, rank, bucket_elems)
        self.longest = max(b.length for b in self.plan)
        slot = self.world * self.longest
        if recv.numel() < slot:
            raise ValueError("recv must hold world * (longest bucket part) elements")
        # 16-bit receive slots, reused bucket after bucket in stream order; with
        # room for two (and device collectives), the exchange of the next
        # bucket overlaps the sum of this one (§2.2 overlap_comm)
        self.overlap = (recv.numel() >= 2 * slot and self.x.active and not self.x.staged
                        and recv.is_cuda)
        self.slots = [recv[:slot], recv[slot:2 * slot]] if self.overlap else [recv[:slot]]
        self.flag = flag
        self.d_sumsq = d_sumsq

    def exchanged_bytes(self, accum_steps: int, elem_bytes: int = 2) -> dict:
        """Bytes this rank sends and receives per step (gradients, then the
        all-gather of the half copy on an applied step)."""
        sent = sum(sum(b.send) - b.send[self.rank] for b in self.plan) * accum_steps * elem_bytes
        recv = sum(b.length for b in self.plan) * (self.world - 1) * accum_steps * elem_bytes
        gather = self.E * (self.world - 1) * elem_bytes
        return {"grad_sent": sent, "grad_received": recv, "param_gather_received": gather}

    def micro_step(self, grad_flat, first: bool, oop_last: bool = False):
        """Exchange one micro-step's flat gradient bucket by bucket and sum the
        received slices of this rank's shard onto the accumulator (oop_last:
        the step's last micro-step, summed and applied out of place per bucket)."""
        pending = None

        def consume(p):
            work, b, rows = p
            if work is not None:
                work.wait()
            if not b.length:
                return
            r = [rows[q] for q in range(self.world)]
            if oop_last:
                self.ops.update_oop(r, b.offset, b.length, self.flag)
            else:
                self.ops.accumulate(r, b.offset, b.length, first, self.flag)

        for i, b in enumerate(self.plan):
            buf = self.slots[i % len(self.slots)]
            rows = buf[:self.world * b.length].view(self.world, b.length)
            # a slot is rewritten only after the sum that read it was queued: the
            # collective waits for the current stream's work before it starts
            work = self.x.all_to_all(rows.view(-1), grad_flat[b.x0:b.x1],
                                     [b.length] * self.world, list(b.send),
                                     async_op=self.overlap)
            if pending is not None:
                consume(pending)
            pending = (work, b, rows)
            if not self.overlap:
                consume(pending)
                pending = None
        if pending is not None:
            consume(pending)

    def finish(self, half_full, clip: bool = False) -> int:
        """The step's boundary: agree on the flag, update, rescale, rebuild the
        half parameters.  Returns the overflow (1: every rank skipped)."""
        self.x.all_reduce(self.flag, "max")
        d = None
        if clip:
            d = self.d_sumsq
            self.ops.sumsq(d)
            self.x.all_reduce(d, "sum")
        self.ops.apply(self.flag, d)
        ovf = self.ops.scaler_update(self.flag)
        if not ovf:
            self.x.all_gather(half_full, self.ops.half_shard)
        return ovf

    def finish_oop(self, half_full) -> int:
        """The boundary of an out-of-place step: agree on the flag, commit (or
        keep the current set), rescale, rebuild the half parameters."""
        self.x.all_reduce(self.flag, "max")
        ovf = self.ops.commit_oop(self.flag)
        if not ovf:
            self.x.all_gather(half_full, self.ops.half_shard)
        return ovf

    def step(self, grads, half_full, clip: bool = False) -> int:
        """A whole step: grads[k] is this rank's flat gradient of micro-step k."""
        self.flag.zero_()
        oop = getattr(self.ops, "oop", False) and not clip
        for k, g in enumerate(grads):
            self.micro_step(g, k == 0, oop_last=oop and k == len(grads) - 1)
        return self.finish_oop(half_full) if oop else self.finish(half_full, clip)


class ZsShardOps:
    """Zero2Step's local compute through the library (the C ABI): the
    accumulate is zs_reduce_check on the received rows, the norm
    zs_grad_sumsq, the update zs_apply / zs_apply_clipped from the
    accumulator, the scale zs_scaler_update.  With a second state set
    (`second` = (master, m, v, half_shard)) unclipped steps apply the last
    micro-step out of place (zs_update_oop per bucket, then the commit)."""

    def __init__(self, zs, ctx, dt, count: int, world: int, accum_steps: int, acc, master, m, v,
                 half_shard, hp, scaler, max_norm: float = 0.0, second=None):
        self.zs, self.ctx, self.dt = zs, ctx, dt
        self.count, self.world, self.g = count, world, accum_steps
        self.acc = acc
        self.sets = [(master, m, v, half_shard)]
        if second is not None:
            self.sets.append(tuple(second))
        self.cur = 0
        self.oop = second is not None
        self.hp, self.scaler, self.max_norm = hp, scaler, max_norm
        self.t = 0

    # the current state set
    master = property(lambda self: self.sets[self.cur][0])
    m = property(lambda self: self.sets[self.cur][1])
    v = property(lambda self: self.sets[self.cur][2])
    half_shard = property(lambda self: self.sets[self.cur][3])

    def _div(self) -> float:
        return float(self.world * self.g * self.scaler.scale)

    def accumulate(self, rows, offset, length, first, flag):
        self.zs.zs_reduce_check(self.ctx, rows, self.dt, length, self.acc[offset:offset + length],
                                first, flag)

    def sumsq(self, d_sumsq):
        self.zs.zs_grad_sumsq(self.ctx, None, self.dt, self.acc, self.count, self._div(), d_sumsq)

    def apply(self, flag, d_sumsq):
        zs = self.zs
        if d_sumsq is not None:
            zs.zs_apply_clipped(self.ctx, flag, d_sumsq, self.max_norm, None, self.dt, self.acc,
                                self.count, self._div(), self.master, self.m, self.v,
                                self.half_shard, self.hp, self.t + 1)
        else:
            zs.zs_apply(self.ctx, flag, None, self.dt, self.acc, self.count, self._div(),
                        self.master, self.m, self.v, self.half_shard, self.hp, self.t + 1)

    def scaler_update(self, flag) -> int:
        ovf = self.zs.zs_scaler_update(self.ctx, flag, self.scaler)
        if not ovf:
            self.t += 1
        return ovf

    def update_oop(self, rows, offset, length, flag):
        src, dst = self.sets[self.cur], self.sets[self.cur ^ 1]
        r = slice(offset, offset + length)
        acc = self.acc[r] if self.g > 1 else None
        self.zs.zs_update_oop(self.ctx, rows, self.dt, length, acc, self._div(), src[0][r],
                              src[1][r], src[2][r], dst[0][r], dst[1][r], dst[2][r], dst[3][r],
                              self.hp, self.t + 1, flag)

    def commit_oop(self, flag) -> int:
        ovf = self.scaler_update(flag)
        if not ovf:
            self.cur ^= 1
        return ovf
