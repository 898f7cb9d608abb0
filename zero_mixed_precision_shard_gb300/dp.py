"""Data-parallel orchestration of one shard step across real ranks.

With one process per GPU, each rank owns one shard (ZeRO-1/2: DeepSpeed
Complete Guide, §2.1 and §2.2) and must skip or apply the step together with
every other rank: an overflow seen by any rank skips the step everywhere and
lowers every rank's loss scale identically (§4.2).  The one exchange this
adds to the shard step is a MAX all-reduce of the int32 overflow flag between
the reduce/check phase and the update phase; on GPUs it stays on the device
(no host round trip before the update).  With gradient clipping a second
scalar joins it: the SUM all-reduce of the shards' squared gradient norms.
"""
from __future__ import annotations


def dp_shard_step(reduce_last, apply, scaler_update, flag, group=None) -> int:
    """Run one step of this rank's shard.

    reduce_last(flag): OR this rank's overflow of the step into `flag` (a
        one-element int32 tensor; it arrives holding 0 or the OR of earlier
        micro-steps).
    apply(flag): the update, which writes nothing if flag != 0.
    scaler_update(flag) -> int: the loss-scale update; returns the overflow.
    Every rank must call this once per step, in the same order."""
    import torch.distributed as dist
    reduce_last(flag)
    if dist.is_available() and dist.is_initialized() and dist.get_world_size(group) > 1:
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
    import torch.distributed as dist
    reduce_last(flag)
    sumsq(d_sumsq)
    if dist.is_available() and dist.is_initialized() and dist.get_world_size(group) > 1:
        dist.all_reduce(flag, op=dist.ReduceOp.MAX, group=group)
        dist.all_reduce(d_sumsq, op=dist.ReduceOp.SUM, group=group)
    apply_clipped(flag, d_sumsq)
    return scaler_update(flag)
