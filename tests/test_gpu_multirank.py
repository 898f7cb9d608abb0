"""The multi-GPU path with two ranks sharing the one GPU over a gloo process
group (the exchanges go through host memory; no kernel waits on another rank).

First the ZeRO-2 step itself (DeepSpeed Complete Guide, §2.1, §2.2) through
the library: each rank holds its own full flat fp16 gradient per micro-step,
sends every bucket's part of shard q to rank q, sums what it receives with
the library's reduce kernel, agrees on the flag (and the clipping norm),
updates its shard and all-gathers the half copy; both ranks' state and the
gathered half parameters are compared with the oracle's union of all shards,
in place and with the last micro-step applied out of place per bucket.
Then the benchmark's multi-GPU run, launched as a multi-GPU run is (torchrun,
one process per rank): the one JSON line reports the whole job."""
import json
import os
import socket
import subprocess
import sys

import numpy as np
import pytest

import bench

pytestmark = pytest.mark.gpu

PSI, G, STEPS, LR = 200_003, 2, 6, 3e-4
HP = (LR, 0.9, 0.999, 1e-8, 0.01)
INJECT = {3: (1, 1, 150_001)}   # step -> (micro, rank, flat index): in rank 1's gradient


def full_grads(world, step, scale, psi_pad):
    """grads[r][k]: rank r's flat fp16 gradient (bit patterns) of micro-step k."""
    rng = np.random.default_rng(500 + step)
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


def second_set(E, dev, oop):
    """The out-of-place step's second master/m/v/half set (None: in place)."""
    import torch
    if not oop:
        return None
    p = torch.zeros(E, dtype=torch.float32, device=dev)
    return (p, torch.zeros_like(p), torch.zeros_like(p),
            torch.zeros(E, dtype=torch.int16, device=dev))


def zero2_worker(rank, world, port, outdir, max_norm, bucket, oop=False):
    import torch
    import torch.distributed as dist

    import oracle
    import zero_mixed_precision_shard_gb300 as zs
    from zero_mixed_precision_shard_gb300.dp import Zero2Step, ZsShardOps
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    torch.cuda.set_device(0)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    part = zs.zs_init_partition(PSI, world)
    psi_pad, E = part.psi_pad, part.shard_len
    m0 = np.zeros(psi_pad, np.float32)
    m0[:PSI] = np.random.default_rng(7).standard_normal(PSI) * 0.02
    ctx = zs.Ctx()
    dev = torch.device("cuda", 0)
    master = torch.from_numpy(m0[rank * E:(rank + 1) * E].copy()).to(dev)
    m, v = torch.zeros_like(master), torch.zeros_like(master)
    acc = torch.zeros_like(master)
    half_shard = torch.zeros(E, dtype=torch.int16, device=dev)
    half_full = torch.from_numpy(oracle.f32_to_half(m0, 0).view(np.int16).copy()).to(dev)
    sc = zs.zs_scaler_init(1024.0, 1.0, 2, 1, True)
    ops = ZsShardOps(zs, ctx, zs.ZS_FP16, E, world, G, acc, master, m, v, half_shard,
                     zs.make_hparams(*HP), sc, max_norm, second=second_set(E, dev, oop))
    recv = torch.zeros(world * min(E, bucket), dtype=torch.int16, device=dev)
    z = Zero2Step(ops, psi_pad, E, rank, bucket, recv,
                  torch.zeros(1, dtype=torch.int32, device=dev),
                  torch.zeros(1, dtype=torch.float64, device=dev))
    flags = []
    for s in range(1, STEPS + 1):
        g = full_grads(world, s, sc.scale, psi_pad)[rank]
        dg = [torch.from_numpy(x.view(np.int16)).to(dev) for x in g]
        flags.append(z.step(dg, half_full, clip=max_norm > 0))
    torch.cuda.synchronize()
    np.savez(os.path.join(outdir, f"rank{rank}.npz"), master=ops.master.cpu().numpy(),
             m=ops.m.cpu().numpy(), v=ops.v.cpu().numpy(),
             half=ops.half_shard.cpu().numpy().view(np.uint16),
             half_full=half_full.cpu().numpy().view(np.uint16), flags=np.array(flags),
             scale=sc.scale, t=ops.t, sent=z.exchanged_bytes(G)["grad_sent"])
    ctx.close()
    dist.destroy_process_group()


def oracle_union(world, max_norm):
    import oracle
    psi_pad, E = oracle.partition(PSI, world)
    m0 = np.zeros(psi_pad, np.float32)
    m0[:PSI] = np.random.default_rng(7).standard_normal(PSI) * 0.02
    states = [oracle.ShardState.from_master(m0[q * E:(q + 1) * E], 0) for q in range(world)]
    hp = oracle.make_hparams(*HP)
    sc = oracle.make_scaler(1024.0, window=2)
    t, flags = 0, []
    for s in range(1, STEPS + 1):
        g = full_grads(world, s, sc.scale, psi_pad)
        per = [[[np.ascontiguousarray(g[r][k][q * E:(q + 1) * E]) for r in range(world)]
                for k in range(G)] for q in range(world)]
        f, t, _ = oracle.multi_shard_step(per, 0, states, hp, t, sc, max_norm=max_norm)
        flags.append(f)
    return flags, states, sc.scale, t


def nccl_one_rank_worker(rank, port, outdir, max_norm, bucket, oop=False):
    """zero2_worker's step over a one-rank NCCL group: every exchange is a real
    NCCL call on device buffers (the all-to-alls posted asynchronously into two
    receive slots, each waited on by the stream before its sum)."""
    import torch
    import torch.distributed as dist

    import oracle
    import zero_mixed_precision_shard_gb300 as zs
    from zero_mixed_precision_shard_gb300.dp import Zero2Step, ZsShardOps
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    dist.init_process_group("nccl", rank=0, world_size=1, device_id=dev)
    part = zs.zs_init_partition(PSI, 1)
    psi_pad, E = part.psi_pad, part.shard_len
    m0 = np.zeros(psi_pad, np.float32)
    m0[:PSI] = np.random.default_rng(7).standard_normal(PSI) * 0.02
    ctx = zs.Ctx()
    master = torch.from_numpy(m0.copy()).to(dev)
    m, v = torch.zeros_like(master), torch.zeros_like(master)
    acc = torch.zeros_like(master)
    half_shard = torch.zeros(E, dtype=torch.int16, device=dev)
    half_full = torch.zeros(psi_pad, dtype=torch.int16, device=dev)
    sc = zs.zs_scaler_init(1024.0, 1.0, 2, 1, True)
    ops = ZsShardOps(zs, ctx, zs.ZS_FP16, E, 1, G, acc, master, m, v, half_shard,
                     zs.make_hparams(*HP), sc, max_norm, second=second_set(E, dev, oop))
    recv = torch.zeros(2 * min(E, bucket), dtype=torch.int16, device=dev)
    z = Zero2Step(ops, psi_pad, E, 0, bucket, recv,
                  torch.zeros(1, dtype=torch.int32, device=dev),
                  torch.zeros(1, dtype=torch.float64, device=dev))
    assert z.overlap and z.x.active and not z.x.staged
    flags = []
    for s in range(1, STEPS + 1):
        g = full_grads(1, s, sc.scale, psi_pad)[0]
        if s in INJECT:
            g[INJECT[s][0]][INJECT[s][2]] = 0x7C00     # one rank: the inf is its own
        dg = [torch.from_numpy(x.view(np.int16)).to(dev) for x in g]
        flags.append(z.step(dg, half_full, clip=max_norm > 0))
    torch.cuda.synchronize()
    np.savez(os.path.join(outdir, "rank0.npz"), master=ops.master.cpu().numpy(),
             m=ops.m.cpu().numpy(), v=ops.v.cpu().numpy(),
             half=ops.half_shard.cpu().numpy().view(np.uint16),
             half_full=half_full.cpu().numpy().view(np.uint16), flags=np.array(flags),
             scale=sc.scale, t=ops.t)
    ctx.close()
    dist.destroy_process_group()


@pytest.mark.parametrize("max_norm,bucket,oop", [(0.0, 50_048, False), (0.01, 1 << 22, False),
                                                (0.0, 50_048, True)])
def test_zero2_step_over_a_one_rank_nccl_group(tmp_path, max_norm, bucket, oop):
    """The NCCL form of the exchanges (device all-to-all with two slots and
    asynchronous posts, device all-reduce and all-gather), on the one GPU as a
    one-rank group, against the oracle's step of the single shard (oop: the
    last micro-step applied out of place per bucket, then committed)."""
    import torch.multiprocessing as mp

    import oracle
    from _helpers import assert_close, half_ulps
    mp.spawn(nccl_one_rank_worker, args=(free_port(), str(tmp_path), max_norm, bucket, oop),
             nprocs=1, join=True)
    psi_pad, E = oracle.partition(PSI, 1)
    m0 = np.zeros(psi_pad, np.float32)
    m0[:PSI] = np.random.default_rng(7).standard_normal(PSI) * 0.02
    st = oracle.ShardState.from_master(m0, 0)
    sc = oracle.make_scaler(1024.0, window=2)
    hp = oracle.make_hparams(*HP)
    t, flags = 0, []
    for s in range(1, STEPS + 1):
        g = full_grads(1, s, sc.scale, psi_pad)[0]
        if s in INJECT:
            g[INJECT[s][0]][INJECT[s][2]] = 0x7C00
        f, t, _ = oracle.shard_step([[x] for x in g], 0, st, hp, t, sc, max_norm=max_norm)
        flags.append(f)
    assert flags == [0, 0, 1, 0, 0, 0]
    d = np.load(tmp_path / "rank0.npz")
    assert d["flags"].tolist() == flags
    assert float(d["scale"]) == sc.scale and int(d["t"]) == t
    for k in ("master", "m", "v"):
        assert_close(d[k], getattr(st, k), k)
    assert half_ulps(d["half"], st.half).max() <= 1
    assert d["half_full"].tobytes() == d["half"].tobytes()    # the one-rank all-gather


@pytest.mark.parametrize("max_norm,bucket,oop", [(0.0, 1 << 22, False), (0.01, 30_016, False),
                                                (0.0, 30_016, True)])
def test_two_cuda_ranks_zero2_step_equals_the_oracle_union(tmp_path, max_norm, bucket, oop):
    import torch.multiprocessing as mp
    from _helpers import assert_close, half_ulps
    world = 2
    mp.spawn(zero2_worker, args=(world, free_port(), str(tmp_path), max_norm, bucket, oop),
             nprocs=world, join=True)
    flags, states, scale, t = oracle_union(world, max_norm)
    assert flags == [0, 0, 1, 0, 0, 0]
    got = [np.load(tmp_path / f"rank{r}.npz") for r in range(world)]
    gathered = np.concatenate([d["half"] for d in got])
    for r, d in enumerate(got):
        assert d["flags"].tolist() == flags          # rank 0 skipped step 3 too
        assert float(d["scale"]) == scale and int(d["t"]) == t
        for k in ("master", "m", "v"):
            assert_close(d[k], getattr(states[r], k), f"rank {r} {k}")
        assert half_ulps(d["half"], states[r].half).max() <= 1
        # the all-gather: every rank holds both ranks' half shards
        assert d["half_full"].tobytes() == gathered.tobytes()
        # each micro-step sends the other rank its shard's part of the flat gradient
        assert int(d["sent"]) == G * 2 * (len(gathered) // world)


def free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def torchrun(args, n=2):
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={n}",
           "--master-addr=127.0.0.1", f"--master-port={free_port()}",
           os.path.join(bench.ROOT, "bench.py"), "--gpus", str(n), "--dist-backend", "gloo"] + args
    out = subprocess.run(cmd, capture_output=True, text=True, timeout=900, cwd=bench.ROOT)
    assert out.returncode == 0, out.stderr[-3000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, out.stdout[-2000:]      # rank 0 alone prints
    return json.loads(lines[0])


@pytest.mark.parametrize("workload,elements,extra", [("llama7b-n1", 1 << 22, []),
                                                     ("gpt2-small-n8", 1 << 20, []),
                                                     ("llama7b-n1", 1 << 22, ["--clip", "1.0"])])
def test_two_ranks_on_one_gpu(workload, elements, extra):
    d = torchrun(["--workload", workload, "--elements", str(elements), "--steps", "3",
                  "--warmup", "3", "--e2e-steps", "1", "--skip-cpu", "--skip-probe"] + extra)
    assert d["n_gpus"] == 2 and d["scaling"] == "strong"
    c = d["config"]
    assert c["parallelism"].startswith("ZeRO-2 dp2")
    assert ("norm SUM" in c["parallelism"]) == bool(extra)
    # whole job: every parameter of the (truncated) model over the slowest rank's step
    assert d["value"] == pytest.approx(elements / (d["ms_per_step"] * 1e-3), rel=1e-6)
    wl = bench.synth.WORKLOADS[workload]
    E = c["shard_len"]
    # each rank sends the other rank its shard's part of every micro-step's gradient
    assert c["exchange_bytes_per_rank_per_step"]["grad_sent"] == wl.g * E * 2
    assert c["exchange_bytes_per_rank_per_step"]["grad_received"] == wl.g * E * 2
    assert d["gpu_launches"] >= 2 * 3 * (wl.g + 1)
    # unclipped: the last micro-step applied out of place per bucket (the second
    # state set fits); clipped: the materialised sums, then the update
    last = "apply" if extra else "update_oop"
    assert set(c["kernels"]) >= {"reduce_first", last} and ("update_oop" in c["api"]) != bool(extra)
    e = d["e2e"]
    assert e["h2d_bytes_per_step"] == 2 * wl.g * 2 * E * 2 and e["value"] > 0
    assert d["cpu_baseline"] is None                 # rank 0 at N = 1 only
