"""Data-parallel orchestration of one shard step across real ranks.

With one process per GPU, each rank owns one shard (ZeRO-1/2: DeepSpeed
Complete Guide, §2.1 and §2.2) and must skip or apply the step together with
every other rank: an overflow seen by any rank skips the step everywhere and
lowers every rank's loss scale identically (§4.2).  The one exchange this
adds to the shard step is a MAX all-reduce of the int32 overflow flag between
the reduce/check phase and the update phase; on GPUs it stays on the device
(no host round trip before the update).
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
