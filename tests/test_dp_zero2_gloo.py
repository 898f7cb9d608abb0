"""The ZeRO-2 exchange choreography on CPU (DeepSpeed Complete Guide, §2.1,
§2.2): gloo ranks each hold their own full flat gradient per micro-step, send
every bucket's part of shard q to rank q (an all-to-all of half slices),
sum what they receive onto their shard's accumulator, agree on the overflow
flag (and the norm when clipping), update, and all-gather the half copy.
The per-rank compute here is the oracle, so the test checks the exchanges:
every rank's shard state, and the gathered half parameters, must equal the
oracle's single-process union of all shards bit for bit, with an overflow on
one rank skipping the step on all; in place, and with the last micro-step
summed and applied out of place bucket by bucket, then committed by the
agreed flag.  Also the bucket plan's host arithmetic.
No GPU."""
import datetime
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
from zero_mixed_precision_shard_gb300.dp import Zero2Step, bucket_plan

PSI, G, STEPS = 5000, 2, 6
INJECT = {3: (1, 1, 4321)}  # step -> (micro, rank, flat index): rank 1's gradient


def full_grads(world, step, scale, psi_pad):
    """grads[r][k]: rank r's flat gradient (fp16 bits) of micro-step k."""
    rng = np.random.default_rng(1000 + step)
    out = []
    for r in range(world):
        per = []
        for k in range(G):
            x = np.zeros(psi_pad, np.float32)
            x[:PSI] = rng.standard_normal(PSI) * 1e-3 * scale
            b = x.astype(np.float16).view(np.uint16)
            if step in INJECT and INJECT[step][:2] == (k, r):
                b[INJECT[step][2]] = 0x7C00
            per.append(b)
        out.append(per)
    return out


def master_init(psi_pad):
    m = np.zeros(psi_pad, np.float32)
    m[:PSI] = np.random.default_rng(99).standard_normal(PSI) * 0.02
    return m


HP = (1e-3, 0.9, 0.999, 1e-8, 0.01)


def reference_union(world, max_norm, steps=STEPS):
    psi_pad, E = oracle.partition(PSI, world)
    m0 = master_init(psi_pad)
    states = [oracle.ShardState.from_master(m0[q * E:(q + 1) * E], 0) for q in range(world)]
    hp = oracle.make_hparams(*HP)
    sc = oracle.make_scaler(1024.0, window=2)
    t, flags = 0, []
    for s in range(1, steps + 1):
        g = full_grads(world, s, sc.scale, psi_pad)
        per = [[[np.ascontiguousarray(g[r][k][q * E:(q + 1) * E]) for r in range(world)]
                for k in range(G)] for q in range(world)]
        f, t, _ = oracle.multi_shard_step(per, 0, states, hp, t, sc, max_norm=max_norm)
        flags.append(f)
    return flags, states, sc.scale, t


class OracleOps:
    """Zero2Step's local compute, done by the oracle on host arrays."""

    def __init__(self, master_shard, world, max_norm):
        self.st = oracle.ShardState.from_master(master_shard, 0)
        self.acc = np.zeros(master_shard.shape[0], np.float32)
        self.hp = oracle.make_hparams(*HP)
        self.sc = oracle.make_scaler(1024.0, window=2)
        self.world, self.max_norm, self.t = world, max_norm, 0

    @property
    def half_shard(self):
        return torch.from_numpy(self.st.half.view(np.int16))   # shares memory

    def div(self):
        return float(self.world * G * self.sc.scale)

    def accumulate(self, rows, offset, length, first, flag):
        a = self.acc[offset:offset + length]
        oracle.reduce_accumulate([r.numpy().view(np.uint16) for r in rows], 0, a, first)
        flag[0] = flag[0] | oracle.any_nonfinite_f32(a)

    def sumsq(self, d):
        d[0] = oracle.grad_sumsq(self.acc, self.div())

    def apply(self, flag, d):
        if int(flag[0]) == 0:
            coef = oracle.clip_coef(float(d[0]), self.max_norm) if d is not None else 1.0
            oracle.adamw_apply_clipped(self.acc, self.div(), coef, self.st.master, self.st.m,
                                       self.st.v, self.st.half, 0, self.hp, self.t + 1)

    def scaler_update(self, flag):
        ovf = int(flag[0])
        oracle.scaler_update(self.sc, ovf)
        if not ovf:
            self.t += 1
        return ovf


class OracleOpsOOP(OracleOps):
    """The same compute, with the last micro-step summed and applied out of
    place into a second state set per bucket and committed by the flag."""
    oop = True

    def __init__(self, master_shard, world, max_norm):
        super().__init__(master_shard, world, max_norm)
        self.other = self.st.copy()

    def update_oop(self, rows, offset, length, flag):
        r = slice(offset, offset + length)
        a = np.zeros(length, np.float32) if G == 1 else self.acc[r].copy()
        oracle.reduce_accumulate([x.numpy().view(np.uint16) for x in rows], 0, a, G == 1)
        flag[0] = flag[0] | oracle.any_nonfinite_f32(a)
        dst = self.other
        for k in ("master", "m", "v"):
            getattr(dst, k)[r] = getattr(self.st, k)[r]
        oracle.adamw_apply(a, self.div(), dst.master[r], dst.m[r], dst.v[r], dst.half[r], 0,
                           self.hp, self.t + 1)

    def commit_oop(self, flag):
        ovf = self.scaler_update(flag)
        if not ovf:
            self.st, self.other = self.other, self.st
        return ovf


def worker(rank, world, port, outdir, max_norm, bucket, oop=False):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    psi_pad, E = oracle.partition(PSI, world)
    m0 = master_init(psi_pad)
    ops = (OracleOpsOOP if oop else OracleOps)(m0[rank * E:(rank + 1) * E], world, max_norm)
    half_full = torch.from_numpy(oracle.f32_to_half(m0, 0).view(np.int16).copy())
    recv = torch.zeros(world * min(E, bucket), dtype=torch.int16)
    z = Zero2Step(ops, psi_pad, E, rank, bucket, recv, torch.zeros(1, dtype=torch.int32),
                  torch.zeros(1, dtype=torch.float64))
    flags = []
    for s in range(1, STEPS + 1):
        g = full_grads(world, s, ops.sc.scale, psi_pad)[rank]
        flags.append(z.step([torch.from_numpy(x.view(np.int16)) for x in g], half_full,
                            clip=max_norm > 0))
    np.savez(os.path.join(outdir, f"rank{rank}.npz"), master=ops.st.master, m=ops.st.m,
             v=ops.st.v, half=ops.st.half, half_full=half_full.numpy().view(np.uint16),
             flags=np.array(flags), scale=ops.sc.scale, t=ops.t)
    dist.destroy_process_group()


def free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


@pytest.mark.parametrize("world,max_norm,bucket,oop", [(2, 0.0, 1 << 20, False),
                                                       (2, 0.01, 640, False),
                                                       (3, 0.0, 1024, False),
                                                       (3, 0.05, 64, False),
                                                       (2, 0.0, 640, True), (3, 0.0, 64, True),
                                                       (3, 0.05, 1024, True)])
def test_zero2_ranks_equal_the_oracle_union(tmp_path, world, max_norm, bucket, oop):
    """oop: the last micro-step out of place per bucket (unclipped steps; a
    clipped step with such ops materialises as before)."""
    mp.spawn(worker, args=(world, free_port(), str(tmp_path), max_norm, bucket, oop),
             nprocs=world, join=True)
    flags, states, scale, t = reference_union(world, max_norm)
    assert flags == [0, 0, 1, 0, 0, 0]
    union_half = np.concatenate([st.half for st in states])
    for r in range(world):
        d = np.load(tmp_path / f"rank{r}.npz")
        assert d["flags"].tolist() == flags       # every rank skipped step 3
        assert float(d["scale"]) == scale and int(d["t"]) == t
        for k in ("master", "m", "v", "half"):
            assert d[k].tobytes() == getattr(states[r], k).tobytes(), k
        assert d["half_full"].tobytes() == union_half.tobytes()   # the all-gather


@pytest.mark.parametrize("psi_pad,world,bucket", [(64 * 12, 3, 64), (64 * 12, 3, 100),
                                                  (64 * 12, 3, 10 ** 6), (2 ** 20, 2, 2 ** 17),
                                                  (64 * 8 * 7, 8, 640)])
def test_bucket_plan_covers_every_shard_once(psi_pad, world, bucket):
    E = psi_pad // world
    for rank in range(world):
        plan = bucket_plan(psi_pad, E, world, rank, bucket)
        assert plan[0].x0 == 0 and plan[-1].x1 == psi_pad
        assert all(a.x1 == b.x0 for a, b in zip(plan, plan[1:]))
        assert all((b.x1 - b.x0) <= bucket and b.x0 % 64 == 0 for b in plan)
        assert all(sum(b.send) == b.x1 - b.x0 for b in plan)
        mine = [(b.offset, b.length) for b in plan if b.length]
        assert mine[0][0] == 0 and sum(ln for _, ln in mine) == E
        assert all(o1 + l1 == o2 for (o1, l1), (o2, _) in zip(mine, mine[1:]))
        # what rank r sends to `rank` is exactly what `rank` receives from each rank
        assert all(b.send[rank] == b.length for b in plan)
        assert all(b.offset % 64 == 0 and b.length % 64 == 0 for b in plan)
    with pytest.raises(ValueError):
        bucket_plan(psi_pad, E, world, 0, 63)


def test_zero2_single_rank_without_a_process_group():
    """One rank and no process group: the exchanges are copies, and the step is
    the oracle's single-shard step."""
    assert not dist.is_initialized()
    psi_pad, E = oracle.partition(PSI, 1)
    m0 = master_init(psi_pad)
    ops = OracleOps(m0.copy(), 1, 0.0)
    half_full = torch.zeros(psi_pad, dtype=torch.int16)
    z = Zero2Step(ops, psi_pad, E, 0, 1024, torch.zeros(1024, dtype=torch.int16),
                  torch.zeros(1, dtype=torch.int32))
    st = oracle.ShardState.from_master(m0, 0)
    sc = oracle.make_scaler(1024.0, window=2)
    t = 0
    for s in range(1, 4):
        g = full_grads(1, s, ops.sc.scale, psi_pad)[0]
        f = z.step([torch.from_numpy(x.view(np.int16)) for x in g], half_full)
        f_o, t, _ = oracle.shard_step([[x] for x in g], 0, st, oracle.make_hparams(*HP), t, sc)
        assert f == f_o
    assert ops.st.master.tobytes() == st.master.tobytes()
    assert half_full.numpy().view(np.uint16).tobytes() == st.half.tobytes()


FAIL_AT = 5


def failing_worker(rank, world, port, outdir):
    """Rank 1 fails on the host before step FAIL_AT's exchange (an exception,
    then the process exits); rank 0 must learn it from its next collective,
    which ends with an error within the group's timeout instead of waiting
    forever, its state that of the steps before."""
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world,
                            timeout=datetime.timedelta(seconds=20))
    psi_pad, E = oracle.partition(PSI, world)
    m0 = master_init(psi_pad)
    ops = OracleOps(m0[rank * E:(rank + 1) * E], world, 0.0)
    half_full = torch.from_numpy(oracle.f32_to_half(m0, 0).view(np.int16).copy())
    z = Zero2Step(ops, psi_pad, E, rank, 1024, torch.zeros(world * 1024, dtype=torch.int16),
                  torch.zeros(1, dtype=torch.int32))
    applied, error = 0, ""
    try:
        for s in range(1, STEPS + 1):
            if rank == 1 and s == FAIL_AT:
                raise RuntimeError("rank 1 failed before its exchange")
            g = full_grads(world, s, ops.sc.scale, psi_pad)[rank]
            z.step([torch.from_numpy(x.view(np.int16)) for x in g], half_full)
            applied = s
    except Exception as e:  # the failure as each rank sees it
        error = f"{type(e).__name__}: {e}"[:300]
    np.savez(os.path.join(outdir, f"rank{rank}.npz"), master=ops.st.master, applied=applied,
             error=error, t=ops.t)
    os._exit(0)   # no teardown of a broken group


def test_a_rank_that_fails_ends_the_others_next_exchange(tmp_path):
    mp.spawn(failing_worker, args=(2, free_port(), str(tmp_path)), nprocs=2, join=True)
    r0, r1 = (np.load(tmp_path / f"rank{r}.npz") for r in range(2))
    assert "rank 1 failed" in str(r1["error"]) and int(r1["applied"]) == FAIL_AT - 1
    assert str(r0["error"]) != ""                     # its exchange ended with an error
    assert int(r0["applied"]) == FAIL_AT - 1
    # rank 0 holds exactly the state of the steps before the failure (one of them skipped)
    _, states, _, t = reference_union(2, 0.0, steps=FAIL_AT - 1)
    assert int(r0["t"]) == t == FAIL_AT - 2
    assert r0["master"].tobytes() == states[0].master.tobytes()
