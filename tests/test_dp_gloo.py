"""The multi-rank path on CPU: two gloo ranks each own one shard of a small
model and step it with dp_shard_step (and dp_shard_step_clipped), using the
oracle for the per-rank work.  An overflow injected on one rank must make both
ranks skip, clipping must use the norm of the whole model, and the union of
the two shards must equal the single-process step of all shards.  No GPU."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle

PSI, N, G, STEPS = 3000, 2, 2, 6
INJECT = {3: (1, 1, 2900)}  # step -> (micro, rank, flat index): lands in rank 1's shard


def make_grads(step, scale, psi_pad):
    rng = np.random.default_rng(step)
    out = []
    for k in range(G):
        micro = []
        for r in range(N):
            x = np.zeros(psi_pad, np.float32)
            x[:PSI] = rng.standard_normal(PSI) * 1e-3 * scale
            b = x.astype(np.float16).view(np.uint16)
            if step in INJECT and INJECT[step][:2] == (k, r):
                b[INJECT[step][2]] = 0x7C00
            micro.append(b)
        out.append(micro)
    return out


def reference_union(max_norm=0.0):
    psi_pad, E = oracle.partition(PSI, N)
    master0 = np.zeros(psi_pad, np.float32)
    master0[:PSI] = np.random.default_rng(99).standard_normal(PSI) * 0.02
    states = [oracle.ShardState.from_master(master0[q * E:(q + 1) * E], 0) for q in range(N)]
    hp = oracle.make_hparams(1e-3, 0.9, 0.999, 1e-8, 0.01)
    sc = oracle.make_scaler(1024.0, window=2)
    t = 0
    flags = []
    for s in range(1, STEPS + 1):
        full = make_grads(s, sc.scale, psi_pad)
        per = [[[np.ascontiguousarray(x[q * E:(q + 1) * E]) for x in micro] for micro in full]
               for q in range(N)]
        f, t, _ = oracle.multi_shard_step(per, 0, states, hp, t, sc, max_norm=max_norm)
        flags.append(f)
    return flags, states, sc.scale, t


def worker(rank, port, outdir, max_norm=0.0):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=N)
    from zero_mixed_precision_shard_gb300.dp import dp_shard_step, dp_shard_step_clipped
    psi_pad, E = oracle.partition(PSI, N)
    master0 = np.zeros(psi_pad, np.float32)
    master0[:PSI] = np.random.default_rng(99).standard_normal(PSI) * 0.02
    st = oracle.ShardState.from_master(master0[rank * E:(rank + 1) * E], 0)
    hp = oracle.make_hparams(1e-3, 0.9, 0.999, 1e-8, 0.01)
    sc = oracle.make_scaler(1024.0, window=2)
    t = [0]
    flags = []
    for s in range(1, STEPS + 1):
        full = make_grads(s, sc.scale, psi_pad)
        mine = [[np.ascontiguousarray(x[rank * E:(rank + 1) * E]) for x in micro]
                for micro in full]
        acc = np.zeros(E, np.float32)
        flag = torch.zeros(1, dtype=torch.int32)

        def reduce_last(f):
            local = 0
            for k, micro in enumerate(mine):
                oracle.reduce_accumulate(micro, 0, acc, first=(k == 0))
                local |= oracle.any_nonfinite(micro, 0, E)
            local |= oracle.any_nonfinite_f32(acc)
            f[0] = f[0] | local

        def apply(f):
            if int(f[0]) == 0:
                oracle.adamw_apply(acc, float(N * G * sc.scale), st.master, st.m, st.v, st.half,
                                   0, hp, t[0] + 1)

        def scaler_update(f):
            ovf = int(f[0])
            oracle.scaler_update(sc, ovf)
            if not ovf:
                t[0] += 1
            return ovf

        def sumsq(d):
            d[0] = oracle.grad_sumsq(acc, float(N * G * sc.scale))

        def apply_clipped(f, d):
            if int(f[0]) == 0:
                coef = oracle.clip_coef(float(d[0]), max_norm)
                oracle.adamw_apply_clipped(acc, float(N * G * sc.scale), coef, st.master, st.m,
                                           st.v, st.half, 0, hp, t[0] + 1)

        if max_norm > 0:
            d_sumsq = torch.zeros(1, dtype=torch.float64)
            flags.append(dp_shard_step_clipped(reduce_last, sumsq, apply_clipped, scaler_update,
                                               flag, d_sumsq))
        else:
            flags.append(dp_shard_step(reduce_last, apply, scaler_update, flag))
    np.savez(os.path.join(outdir, f"rank{rank}.npz"), master=st.master, m=st.m, v=st.v,
             half=st.half, flags=np.array(flags), scale=sc.scale, t=t[0])
    dist.destroy_process_group()


def free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


@pytest.mark.parametrize("max_norm", [0.0, 0.01])
def test_two_gloo_ranks_skip_together(tmp_path, max_norm):
    mp.spawn(worker, args=(free_port(), str(tmp_path), max_norm), nprocs=N, join=True)
    flags, states, scale, t = reference_union(max_norm)
    assert flags == [0, 0, 1, 0, 0, 0]
    for r in range(N):
        d = np.load(tmp_path / f"rank{r}.npz")
        assert d["flags"].tolist() == flags      # rank 0 skipped although it saw no overflow
        assert float(d["scale"]) == scale and int(d["t"]) == t
        for k in ("master", "m", "v", "half"):
            assert d[k].tobytes() == getattr(states[r], k).tobytes()


def test_single_process_without_group_is_a_plain_step():
    from zero_mixed_precision_shard_gb300.dp import dp_shard_step, dp_shard_step_clipped
    calls = []
    flag = torch.zeros(1, dtype=torch.int32)
    ovf = dp_shard_step(lambda f: calls.append("r"), lambda f: calls.append("a"),
                        lambda f: (calls.append("s"), 0)[1], flag)
    assert calls == ["r", "a", "s"] and ovf == 0
