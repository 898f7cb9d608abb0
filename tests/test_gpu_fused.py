"""The fused step: zs_shard_step, zs_shard_step_async, zs_shard_step_oop,
zs_shard_step_async_oop and the clipped forms as ONE cooperative kernel
wherever one thread per 8 (unclipped shards small enough: 4) owned elements
fits a co-resident grid.  Each thread holds its elements' last
micro-step sums and state in registers across a bounded grid barrier that
resolves the step's overflow flag (DeepSpeed Complete Guide, §2.2 and §4.2:
nothing is committed on an overflowing step).

Checked: flags, scales and every state buffer equal to the multi-kernel path's
bit for bit, step after step (the same fp32 arithmetic in the same order),
with an overflow on the last and on an earlier micro-step; the state held to
the oracle's bound; that exactly one fused launch ran per step within the
capacity and none past it; CUDA-graph replay of the cooperative launch; and
the bounded wait -- a barrier that waits for a CTA that never comes gives up
within its limit, writes nothing, and the context reports ZS_ERR_TIMEOUT and
stays usable."""
import numpy as np
import pytest
import torch

import oracle
from _helpers import (STRESS_LR, assert_close, assert_half_close, dev16, half_ulps, host16,
                      lib_half)

pytestmark = pytest.mark.gpu

FP16, BF16 = 0, 1
HP = (STRESS_LR, 0.9, 0.999, 1e-8, 0.01)


@pytest.fixture(scope="module")
def zs():
    import zero_mixed_precision_shard_gb300 as pkg
    torch.cuda.set_device(0)
    return pkg


@pytest.fixture(scope="module")
def ctxs(zs):
    on, off = zs.Ctx(), zs.Ctx()
    off.set_fused(zs.ZS_FUSED_OFF)
    on.set_timing(True)
    off.set_timing(True)
    yield on, off
    on.close()
    off.close()


def fused_launches(zs, ctx):
    return ctx.timing(zs.ZS_KERNEL_FUSED)[1]


def rand_grads(rng, n, count, dtype, scale):
    return [lib_half((rng.standard_normal(count) * 1e-3 * scale *
                      np.exp2(rng.integers(-4, 4, count))).astype(np.float32), dtype)
            for _ in range(n)]


def state_set(master0, count):
    master = torch.from_numpy(master0.copy()).cuda()
    return {"p": master, "m": torch.zeros_like(master), "v": torch.zeros_like(master),
            "h": torch.zeros(count, dtype=torch.int16, device="cuda")}


def same_state(a, b, where):
    for k in ("p", "m", "v", "h"):
        assert torch.equal(a[k], b[k]), (where, k)


def inject(grads, s, G, n, count, dtype):
    """An inf on the last micro-step at step 3, on the first at step 7; at
    step 5 NaNs every 997 elements of the last micro-step, so that every CTA
    of a large grid arrives at the barrier with a non-finite sum."""
    if s in (3, 7):
        k = G - 1 if s == 3 else 0
        grads[k][n - 1][count // 3] = 0x7C00 if dtype == FP16 else 0x7F80
    if s == 5:
        grads[G - 1][0][::997] = 0x7E00 if dtype == FP16 else 0x7FC0


@pytest.mark.parametrize("dtype", [FP16, BF16])
@pytest.mark.parametrize("n,G,count", [(1, 1, 1), (1, 1, 7), (2, 1, 8), (2, 1, 4099),
                                       (3, 2, 65_541), (5, 3, 10_007), (64, 1, 777),
                                       (2, 1, 524_288), (256, 1, 1_000),
                                       # either side of the switch from 4- to 8-element
                                       # units (4 CTAs per SM x 152 SMs x 256 x 4)
                                       (1, 1, 622_591), (2, 2, 622_597), (3, 1, 900_001)])
@pytest.mark.parametrize("hyst,consec", [(1, False), (2, False), (2, True)])
def test_fused_sync_steps_equal_the_multi_kernel_path_and_the_oracle(zs, ctxs, dtype, n, G,
                                                                     count, hyst, consec):
    """Ten steps, overflows at steps 3, 5 and 7, under the loss scaler's
    hysteresis 1 and 2 (consecutive or not): the fused step's last CTA runs
    the same scaler as the multi-kernel path."""
    on, off = ctxs
    rng = np.random.default_rng(1000 * n + 10 * G + dtype + count % 97)
    master0 = (rng.standard_normal(count) * 0.02).astype(np.float32)
    hp, hp_o = zs.make_hparams(*HP), oracle.make_hparams(*HP)
    dyn = dtype == FP16
    sc_o = oracle.make_scaler(1024.0 if dyn else 1.0, 1.0, 3, hyst, dyn, consec)
    sc = {c: zs.zs_scaler_init(sc_o.scale, 1.0, 3, hyst, dyn, consec) for c in ("on", "off")}
    st = oracle.ShardState.from_master(master0, dtype)
    sets = {"on": state_set(master0, count), "off": state_set(master0, count)}
    accs = {c: torch.zeros(count, dtype=torch.float32, device="cuda") for c in ("on", "off")}
    t = t_o = 0
    f0 = fused_launches(zs, on)
    for s in range(1, 11):
        grads = [rand_grads(rng, n, count, dtype, sc_o.scale) for _ in range(G)]
        inject(grads, s, G, n, count, dtype)
        ovf_o, t_o, _ = oracle.shard_step(grads, dtype, st, hp_o, t_o, sc_o)
        dg = [[dev16(x) for x in micro] for micro in grads]
        out = {}
        for name, ctx in (("on", on), ("off", off)):
            b, acc = sets[name], accs[name]
            for k in range(G - 1):
                zs.zs_grad_accum(ctx, dg[k], dtype, count, acc, k == 0)
            out[name] = zs.zs_shard_step(ctx, dg[G - 1], dtype, count, acc if G > 1 else None,
                                         G, b["p"], b["m"], b["v"], b["h"], hp, t + 1, sc[name])
        assert out["on"] == out["off"] == (ovf_o, sc_o.scale), f"step {s}"
        assert (sc["on"].clean_count, sc["on"].hyst_left) == (sc_o.clean_count, sc_o.hyst_left)
        same_state(sets["on"], sets["off"], s)
        if not ovf_o:
            t += 1
    assert t == t_o
    assert fused_launches(zs, on) - f0 == 10          # one launch per step, skipped ones too
    got = sets["on"]
    assert_close(got["p"].cpu().numpy(), st.master, "master")
    assert_close(got["m"].cpu().numpy(), st.m, "m")
    assert_close(got["v"].cpu().numpy(), st.v, "v")
    assert_half_close(host16(got["h"]), got["p"].cpu().numpy(), st.half, st.master, dtype)


def test_fused_oop_sync_equals_in_place(zs, ctxs):
    """zs_shard_step_oop through the fused kernel: the written set equals the
    in-place step's state; on an overflow nothing is written anywhere."""
    on, _ = ctxs
    rng = np.random.default_rng(5)
    n, G, count, dtype = 2, 2, 30_011, FP16
    master0 = (rng.standard_normal(count) * 0.02).astype(np.float32)
    hp = zs.make_hparams(*HP)
    sc_a, sc_b = zs.zs_scaler_init(512.0, 1.0, 2, 1, True), zs.zs_scaler_init(512.0, 1.0, 2, 1, True)
    ref = state_set(master0, count)
    bufs = [state_set(master0, count), state_set(np.zeros_like(master0), count)]
    acc_a = torch.zeros(count, dtype=torch.float32, device="cuda")
    acc_b = torch.zeros_like(acc_a)
    cur, t = 0, 0
    f0 = fused_launches(zs, on)
    for s in range(1, 9):
        grads = [rand_grads(rng, n, count, dtype, sc_a.scale) for _ in range(G)]
        inject(grads, s, G, n, count, dtype)
        dg = [[dev16(x) for x in micro] for micro in grads]
        zs.zs_grad_accum(on, dg[0], dtype, count, acc_a, True)
        ovf_a, _ = zs.zs_shard_step(on, dg[1], dtype, count, acc_a, G, ref["p"], ref["m"], ref["v"],
                                    ref["h"], hp, t + 1, sc_a)
        zs.zs_grad_accum(on, dg[0], dtype, count, acc_b, True)
        src, dst = bufs[cur], bufs[cur ^ 1]
        before = {k: x.clone() for k, x in dst.items()}
        ovf_b, _ = zs.zs_shard_step_oop(on, dg[1], dtype, count, acc_b, G, src["p"], src["m"],
                                        src["v"], dst["p"], dst["m"], dst["v"], dst["h"], hp,
                                        t + 1, sc_b)
        assert ovf_a == ovf_b and sc_a.scale == sc_b.scale, f"step {s}"
        if ovf_b:
            same_state(dst, before, s)                  # the fused form writes nothing
        else:
            cur ^= 1
            t += 1
        same_state(bufs[cur], ref, s)
    assert fused_launches(zs, on) - f0 == 16


def run_async(zs, ctx, api, graph, n, G, count, rng_seed, steps=10):
    """Ten async steps (one overflow) under a WarmupDecayLR schedule; returns
    the state after each step and the oracle's final state."""
    dtype = FP16
    rng = np.random.default_rng(rng_seed)
    master0 = (rng.standard_normal(count) * 0.02).astype(np.float32)
    st = oracle.ShardState.from_master(master0, dtype)
    sc_o = oracle.make_scaler(512.0, 1.0, 2, 1, True)
    kind, mn, mx, wu, tot = (oracle.LR_WARMUP_DECAY, float(np.float32(1e-5)),
                             float(np.float32(STRESS_LR)), 3, 9)
    sched = zs.make_schedule(kind, mn, mx, wu, tot)
    hp = zs.make_hparams(mx, 0.9, 0.999, 1e-8, 0.01)
    state = zs.DeviceState(zs.zs_scaler_init(sc_o.scale, 1.0, 2, 1, True))
    sets = [state_set(master0, count), state_set(np.zeros_like(master0), count)]
    acc = torch.zeros(count, dtype=torch.float32, device="cuda")
    pad = (count + 7) // 8 * 8
    gbuf = torch.zeros((G, n, pad), dtype=torch.int16, device="cuda")
    ptrs = [zs.pointer_array(gbuf[k, r, :count] for r in range(n)) for k in range(G)]
    pairs = {k: zs.pointer_array([sets[0][k], sets[1][k]]) for k in ("p", "m", "v", "h")}
    s0 = sets[0]

    def step_calls():
        for k in range(G - 1):
            zs.zs_grad_accum(ctx, ptrs[k], dtype, count, acc, k == 0)
        if api == "async":
            zs.zs_shard_step_async(ctx, ptrs[G - 1], dtype, count, acc, G, s0["p"], s0["m"],
                                   s0["v"], s0["h"], hp, sched, state)
        else:
            zs.zs_shard_step_async_oop(ctx, ptrs[G - 1], dtype, count, acc, G, pairs["p"],
                                       pairs["m"], pairs["v"], pairs["h"], hp, sched, state)

    g = None
    t_o = 0
    snaps = []
    for s in range(1, steps + 1):
        grads = [[lib_half((rng.standard_normal(count) * 1e-2 * sc_o.scale).astype(np.float32),
                           dtype) for _ in range(n)] for _ in range(G)]
        if s == 5:
            grads[G - 1][n - 1][count - 1] = 0x7C00
        host = np.stack([np.stack(mc) for mc in grads]).view(np.int16)
        gbuf[:, :, :count].copy_(torch.from_numpy(host))
        lr_t = oracle.lr_at(kind, mn, mx, wu, tot, t_o + 1)
        ovf_o, t_o, _ = oracle.shard_step(grads, dtype, st,
                                          oracle.make_hparams(lr_t, 0.9, 0.999, 1e-8, 0.01),
                                          t_o, sc_o)
        if graph and g is None:
            step_calls()                 # the first step uncaptured, then capture the rest
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                step_calls()
        elif graph:
            g.replay()
        else:
            step_calls()
        d = state.read()
        assert d.overflow == ovf_o and d.scaler.scale == sc_o.scale, f"step {s}"
        assert d.step == t_o and d.iterations == s
        cur = sets[d.buf if api == "async_oop" else 0]
        if api == "async_oop":
            assert d.buf == t_o % 2
        snaps.append({k: x.clone() for k, x in cur.items()})
    return snaps, st


@pytest.mark.parametrize("api", ["async", "async_oop"])
@pytest.mark.parametrize("graph", [False, True])
@pytest.mark.parametrize("n,G,count", [(1, 3, 20_011), (8, 2, 40_003), (2, 1, 524_288)])
def test_fused_async_steps_equal_the_multi_kernel_path_and_the_oracle(zs, ctxs, api, graph, n,
                                                                      G, count):
    on, off = ctxs
    seed = n + 10 * G + (100 if graph else 0) + (7 if api == "async_oop" else 0)
    f0 = fused_launches(zs, on)
    got, st = run_async(zs, on, api, graph, n, G, count, seed)
    if not graph:   # launches inside a graph replay are not timed
        assert fused_launches(zs, on) - f0 == 10
    ref, _ = run_async(zs, off, api, graph, n, G, count, seed)
    for s, (a, b) in enumerate(zip(got, ref), start=1):
        same_state(a, b, s)
    last = got[-1]
    assert_close(last["p"].cpu().numpy(), st.master, "master")
    assert_close(last["m"].cpu().numpy(), st.m, "m")
    assert_close(last["v"].cpu().numpy(), st.v, "v")
    assert half_ulps(host16(last["h"]), st.half).max() <= 1


@pytest.mark.parametrize("extra", [0, 1, 8])
def test_fused_capacity_boundary(zs, ctxs, extra):
    """At the capacity the step is one fused launch; past it the multi-kernel
    path runs; both give the same state."""
    on, off = ctxs
    cap = on.fused_capacity
    assert cap == off.fused_capacity and cap >= 524_288
    count = cap + extra
    rng = np.random.default_rng(extra)
    master0 = (rng.standard_normal(count) * 0.02).astype(np.float32)
    hp = zs.make_hparams(*HP)
    grads = [dev16(x) for x in rand_grads(rng, 2, count, FP16, 1024.0)]
    res = {}
    for name, ctx in (("on", on), ("off", off)):
        b = state_set(master0, count)
        sc = zs.zs_scaler_init(1024.0, 1.0, 10, 1, True)
        f0 = fused_launches(zs, ctx)
        r0 = ctx.timing(zs.ZS_KERNEL_APPLY_RECOMPUTE)[1]
        res[name] = (zs.zs_shard_step(ctx, grads, FP16, count, None, 1, b["p"], b["m"], b["v"],
                                      b["h"], hp, 1, sc), b)
        fused = fused_launches(zs, ctx) - f0
        multi = ctx.timing(zs.ZS_KERNEL_APPLY_RECOMPUTE)[1] - r0
        if name == "on" and extra == 0:
            assert (fused, multi) == (1, 0)
        else:
            assert (fused, multi) == (0, 1)
    assert res["on"][0] == res["off"][0] == (0, 1024.0)
    same_state(res["on"][1], res["off"][1], "boundary")


def test_fused_wait_that_runs_out_reports_a_timeout(zs):
    """ZS_FUSED_TEST_TIMEOUT makes the barrier wait for a CTA that never comes:
    every CTA gives up after the limit (20 ms here) and writes nothing; the
    synchronising call returns ZS_ERR_TIMEOUT with the scaler untouched; the
    context resets its barrier and flag and its next step is the oracle's."""
    ctx = zs.Ctx()
    try:
        ctx.set_fused(zs.ZS_FUSED_TEST_TIMEOUT, 20_000_000)
        rng = np.random.default_rng(3)
        n, count, dtype = 2, 50_003, FP16
        master0 = (rng.standard_normal(count) * 0.02).astype(np.float32)
        grads = rand_grads(rng, n, count, dtype, 1024.0)
        grads[1][17] = 0x7C00            # a flag bit the failed step leaves behind
        dg = [dev16(x) for x in grads]
        hp = zs.make_hparams(*HP)
        sc = zs.zs_scaler_init(1024.0, 1.0, 10, 1, True)
        b = state_set(master0, count)
        before = {k: x.clone() for k, x in b.items()}
        with pytest.raises(zs.ZsError) as e:
            zs.zs_shard_step(ctx, dg, dtype, count, None, 1, b["p"], b["m"], b["v"], b["h"], hp,
                             1, sc)
        assert e.value.status == zs.ZS_ERR_TIMEOUT
        same_state(b, before, "after the timeout")
        assert sc.scale == 1024.0 and sc.clean_count == 0
        # the async form returns at once; the next call on the context reports it
        state = zs.DeviceState(zs.zs_scaler_init(1024.0, 1.0, 10, 1, True))
        zs.zs_shard_step_async(ctx, dg, dtype, count, None, 1, b["p"], b["m"], b["v"], b["h"],
                               hp, None, state)
        torch.cuda.synchronize()
        with pytest.raises(zs.ZsError) as e:
            zs.zs_grad_accum(ctx, dg, dtype, count, torch.zeros(count, device="cuda"), True)
        assert e.value.status == zs.ZS_ERR_TIMEOUT
        d = state.read()
        assert (d.step, d.iterations, d.scaler.scale) == (0, 0, 1024.0)
        same_state(b, before, "after the async timeout")
        # usable again: a clean step from the same state equals the oracle's
        ctx.set_fused(zs.ZS_FUSED_ON)
        grads[1][17] = grads[1][18]
        dg = [dev16(x) for x in grads]
        st = oracle.ShardState.from_master(master0, dtype)
        sc_o = oracle.make_scaler(1024.0, 1.0, 10, 1, True)
        ovf_o, _, _ = oracle.shard_step([grads], dtype, st, oracle.make_hparams(*HP), 0, sc_o)
        assert zs.zs_shard_step(ctx, dg, dtype, count, None, 1, b["p"], b["m"], b["v"], b["h"],
                                hp, 1, sc) == (ovf_o, sc_o.scale) == (0, 1024.0)
        assert_close(b["p"].cpu().numpy(), st.master, "master")
        assert_close(b["v"].cpu().numpy(), st.v, "v")
    finally:
        ctx.close()


def test_set_fused_rejects_unknown_modes(zs):
    ctx = zs.Ctx()
    try:
        with pytest.raises(zs.ZsError) as e:
            ctx.set_fused(3)
        assert e.value.status == zs.ZS_ERR_ARG
    finally:
        ctx.close()


@pytest.mark.parametrize("mode", ["fused", "multi"])
@pytest.mark.parametrize("hyst", [1, 2])
def test_device_state_step_equals_the_synchronising_step_bitwise(zs, mode, hyst):
    """The device forms compute the step's constants (bias corrections by
    square-and-multiply in fp64, the same operations as the host) on the
    device: zs_shard_step_async and zs_shard_step give the same state bit for
    bit, step after step, skipped steps included."""
    ctx = zs.Ctx()
    try:
        ctx.set_fused(zs.ZS_FUSED_ON if mode == "fused" else zs.ZS_FUSED_OFF)
        rng = np.random.default_rng(11)
        n, G, count, dtype = 2, 2, 20_011, FP16
        master0 = (rng.standard_normal(count) * 0.02).astype(np.float32)
        hp = zs.make_hparams(*HP)
        sc = zs.zs_scaler_init(1024.0, 1.0, 2, hyst, True)
        state = zs.DeviceState(zs.zs_scaler_init(1024.0, 1.0, 2, hyst, True))
        a, b = state_set(master0, count), state_set(master0, count)
        acc_a = torch.zeros(count, dtype=torch.float32, device="cuda")
        acc_b = torch.zeros_like(acc_a)
        t = 0
        for s in range(1, 13):
            grads = [rand_grads(rng, n, count, dtype, sc.scale) for _ in range(G)]
            inject(grads, s, G, n, count, dtype)
            dg = [[dev16(x) for x in micro] for micro in grads]
            zs.zs_grad_accum(ctx, dg[0], dtype, count, acc_a, True)
            ovf, _ = zs.zs_shard_step(ctx, dg[1], dtype, count, acc_a, G, a["p"], a["m"], a["v"],
                                      a["h"], hp, t + 1, sc)
            zs.zs_grad_accum(ctx, dg[0], dtype, count, acc_b, True)
            zs.zs_shard_step_async(ctx, dg[1], dtype, count, acc_b, G, b["p"], b["m"], b["v"],
                                   b["h"], hp, None, state)
            d = state.read()
            assert (d.overflow, d.scaler.scale) == (ovf, sc.scale), s
            assert (d.scaler.hyst_left, d.scaler.clean_count) == (sc.hyst_left, sc.clean_count)
            t += 0 if ovf else 1
            assert d.step == t
            same_state(a, b, s)
    finally:
        ctx.close()


@pytest.mark.parametrize("form", ["sync", "async"])
@pytest.mark.parametrize("n,G,count,max_norm", [(1, 3, 50_001, 0.05), (2, 1, 8_191, 0.01),
                                                (5, 2, 524_288, 0.02), (3, 1, 7, 1e-6)])
def test_fused_clipped_steps_equal_the_multi_kernel_path(zs, ctxs, form, n, G, count, max_norm):
    """The clipped forms through the fused kernel: each CTA's total of squares
    travels with the grid barrier and the last CTA folds the totals in the
    norm pass's order, so the norm, the coefficient and every state buffer
    equal the multi-kernel path's bit for bit, step after step (an overflow
    included), and the state stays within the oracle's bound."""
    on, off = ctxs
    dtype = FP16
    rng = np.random.default_rng(7 * n + G + count % 101)
    master0 = (rng.standard_normal(count) * 0.02).astype(np.float32)
    hp, hp_o = zs.make_hparams(*HP), oracle.make_hparams(*HP)
    st = oracle.ShardState.from_master(master0, dtype)
    sc_o = oracle.make_scaler(1024.0, 1.0, 3, 1, True)
    sets = {c: state_set(master0, count) for c in ("on", "off")}
    accs = {c: torch.zeros(count, dtype=torch.float32, device="cuda") for c in ("on", "off")}
    scs = {c: zs.zs_scaler_init(1024.0, 1.0, 3, 1, True) for c in ("on", "off")}
    states = {c: zs.DeviceState(zs.zs_scaler_init(1024.0, 1.0, 3, 1, True)) for c in ("on", "off")}
    norms = {c: torch.zeros(1, dtype=torch.float64, device="cuda") for c in ("on", "off")}
    f0 = fused_launches(zs, on)
    t = t_o = 0
    for s in range(1, 7):
        grads = [rand_grads(rng, n, count, dtype, sc_o.scale) for _ in range(G)]
        if s == 3:
            grads[G - 1][n - 1][count // 2] = 0x7C00
        ovf_o, t_o, _, norm_o = oracle.shard_step(grads, dtype, st, hp_o, t_o, sc_o,
                                                  max_norm=max_norm, return_norm=True)
        dg = [[dev16(x) for x in micro] for micro in grads]
        res = {}
        for name, ctx in (("on", on), ("off", off)):
            b, acc = sets[name], accs[name]
            for k in range(G - 1):
                zs.zs_grad_accum(ctx, dg[k], dtype, count, acc, k == 0)
            a = acc if G > 1 else None
            if form == "sync":
                res[name] = zs.zs_shard_step_clipped(ctx, dg[G - 1], dtype, count, a, G, b["p"],
                                                     b["m"], b["v"], b["h"], hp, t + 1,
                                                     scs[name], max_norm)
            else:
                zs.zs_shard_step_async_clipped(ctx, dg[G - 1], dtype, count, a, G, b["p"],
                                               b["m"], b["v"], b["h"], hp, None, max_norm,
                                               states[name], norms[name])
                d = states[name].read()
                res[name] = (d.overflow, d.scaler.scale, norms[name].item())
        assert res["on"][:2] == res["off"][:2] == (ovf_o, sc_o.scale), s
        if not ovf_o:
            assert res["on"][2] == res["off"][2], s          # the norm, bit for bit
            assert abs(res["on"][2] - norm_o) <= 1e-6 * norm_o
            t += 1
        same_state(sets["on"], sets["off"], s)
    assert t == t_o
    assert fused_launches(zs, on) - f0 == 6
    got = sets["on"]
    assert_close(got["p"].cpu().numpy(), st.master, "master")
    assert_close(got["m"].cpu().numpy(), st.m, "m")
    assert_close(got["v"].cpu().numpy(), st.v, "v")


@pytest.mark.parametrize("count,dtype", [(524_291, FP16), (900_001, BF16)])
def test_many_fused_steps_equal_the_multi_kernel_path(zs, count, dtype):
    """501 device-state out-of-place steps, 50 to each CUDA graph replay (the
    benchmark's launch pattern for a short step), 4- and 8-element units:
    every one of them resolved by the fused grid barrier the way the
    multi-kernel path resolves it.  Two replays run with an inf in the
    gradients (100 overflowing steps in a row, under hysteresis 2); at the end
    the current state set, the scale and the step counts are equal bit for bit."""
    n, per, replays = 2, 50, 10
    rng = np.random.default_rng(count)
    master0 = (rng.standard_normal(count) * 0.02).astype(np.float32)
    pad = (count + 7) // 8 * 8
    host = np.zeros((n, pad), np.uint16)
    host[:, :count] = np.stack(rand_grads(rng, n, count, dtype, 1024.0))
    gbuf = torch.from_numpy(host.view(np.int16)).cuda()
    hp = zs.make_hparams(*HP)
    inf = 0x7C00 if dtype == FP16 else 0x7F80
    runs = []
    for mode in (zs.ZS_FUSED_ON, zs.ZS_FUSED_OFF):
        ctx = zs.Ctx()
        ctx.set_fused(mode)
        sets = [state_set(master0, count), state_set(np.zeros_like(master0), count)]
        pairs = [zs.pointer_array([sets[0][k], sets[1][k]]) for k in ("p", "m", "v", "h")]
        ptrs = zs.pointer_array(gbuf[r, :count] for r in range(n))
        dyn = dtype == FP16
        state = zs.DeviceState(zs.zs_scaler_init(1024.0 if dyn else 1.0, 1.0, 7, 2, dyn))

        def step():
            zs.zs_shard_step_async_oop(ctx, ptrs, dtype, count, None, 1, *pairs, hp, None, state)
        step()                                   # uncaptured: caches the launch shapes
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for _ in range(per):
                step()
        runs.append((ctx, sets, state, g))
    for r in range(replays):
        if r in (3, 7):
            gbuf[1, 12_345] = inf
        for _, _, _, g in runs:
            g.replay()
        torch.cuda.synchronize()
        if r in (3, 7):
            gbuf[1, 12_345] = int(host[1, 12_345].astype(np.int16))
    (c_on, s_on, d_on, _), (c_off, s_off, d_off, _) = runs
    a, b = d_on.read(), d_off.read()
    assert a.iterations == b.iterations == 1 + per * replays
    assert (a.step, a.buf, a.scaler.scale, a.scaler.hyst_left, a.scaler.clean_count) == \
        (b.step, b.buf, b.scaler.scale, b.scaler.hyst_left, b.scaler.clean_count)
    assert a.step == 1 + per * (replays - 2)                 # the two inf replays skipped
    same_state(s_on[a.buf & 1], s_off[b.buf & 1], "after 501 steps")
    assert not torch.equal(s_on[a.buf & 1]["p"], torch.from_numpy(master0).cuda())
    for ctx, _, _, g in runs:
        del g
        ctx.close()
