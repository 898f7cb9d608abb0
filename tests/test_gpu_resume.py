"""Checkpoint/resume and run-to-run determinism of the shard step.  All state
is caller-owned (master, m, v, half copy, scaler, Adam's step count; for the
device-resident forms the zs_device_state and the current set), so saving it
after 5 steps, reloading it into fresh buffers and a fresh context and running
5 more steps must equal 10 straight steps bit for bit."""
import io

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def zs():
    import zero_mixed_precision_shard_gb300 as pkg
    torch.cuda.set_device(0)
    return pkg


def make_grads(step, n, g, count, scale):
    """[g][n] slices of `count` halves; rows padded to 8 elements so every
    slice starts 16-byte aligned."""
    rng = np.random.default_rng(1000 + step)
    pad = (count + 7) // 8 * 8
    x = np.zeros((g, n, pad), np.float16)
    x[:, :, :count] = (rng.standard_normal((g, n, count)) * 1e-2 * scale).astype(np.float16)
    if step == 4:
        x[0, n - 1, 7] = np.inf
    return torch.from_numpy(x.view(np.int16)).cuda()[:, :, :count]


def run(zs, ctx, state, first_step, last_step, n, g, count):
    master, m, v, half, acc, scaler, t = state
    hp = zs.make_hparams(1e-3, 0.9, 0.999, 1e-8, 0.01)
    for s in range(first_step, last_step + 1):
        gb = make_grads(s, n, g, count, scaler.scale)
        for k in range(g - 1):
            zs.zs_grad_accum(ctx, [gb[k, r] for r in range(n)], zs.ZS_FP16, count, acc, k == 0)
        ovf, _ = zs.zs_shard_step(ctx, [gb[g - 1, r] for r in range(n)], zs.ZS_FP16, count, acc, g,
                                  master, m, v, half, hp, t + 1, scaler)
        if not ovf:
            t += 1
    return master, m, v, half, acc, scaler, t


def fresh(zs, n, g, count):
    rng = np.random.default_rng(5)
    master = torch.from_numpy((rng.standard_normal(count) * 0.02).astype(np.float32)).cuda()
    return (master, torch.zeros_like(master), torch.zeros_like(master),
            torch.zeros(count, dtype=torch.int16, device="cuda"),
            torch.zeros(count, dtype=torch.float32, device="cuda"),
            zs.zs_scaler_init(1024.0, 1.0, 3, 1, True), 0)


@pytest.mark.parametrize("n,g", [(2, 3), (8, 1)])
def test_resume_equals_straight_run(zs, n, g):
    count = 40_009
    ctx = zs.Ctx()
    straight = run(zs, ctx, fresh(zs, n, g, count), 1, 10, n, g, count)
    half_way = run(zs, ctx, fresh(zs, n, g, count), 1, 5, n, g, count)
    master, m, v, half, _, scaler, t = half_way
    buf = io.BytesIO()
    torch.save({"master": master.cpu(), "m": m.cpu(), "v": v.cpu(), "half": half.cpu(),
                "scaler": list(bytes(scaler)), "t": t}, buf)
    ctx.close()
    buf.seek(0)
    ck = torch.load(buf)
    ctx2 = zs.Ctx()
    sc = zs.zs_scaler.from_buffer_copy(bytes(ck["scaler"]))
    restored = (ck["master"].cuda(), ck["m"].cuda(), ck["v"].cuda(), ck["half"].cuda(),
                torch.zeros(count, dtype=torch.float32, device="cuda"), sc, ck["t"])
    resumed = run(zs, ctx2, restored, 6, 10, n, g, count)
    for a, b in zip(straight[:4], resumed[:4]):
        assert torch.equal(a, b)
    assert straight[5].scale == resumed[5].scale and straight[6] == resumed[6] == 9
    ctx2.close()


def test_runs_are_bitwise_deterministic(zs):
    n, g, count = 16, 2, 300_007
    outs = []
    for _ in range(2):
        ctx = zs.Ctx()
        outs.append(run(zs, ctx, fresh(zs, n, g, count), 1, 6, n, g, count))
        ctx.close()
    for a, b in zip(outs[0][:5], outs[1][:5]):
        assert torch.equal(a, b)


def run_device(zs, ctx, bufs, dstate, first_step, last_step, n, g, count, sched):
    """zs_grad_accum + zs_shard_step_async_oop (the benchmark's default form):
    bufs[k] = the pair of buffers of master, m, v and half; the device state
    names the current set."""
    hp = zs.make_hparams(1e-3, 0.9, 0.999, 1e-8, 0.01)
    pairs = [zs.pointer_array(p) for p in bufs]
    acc = torch.zeros(count, dtype=torch.float32, device="cuda")
    for s in range(first_step, last_step + 1):
        gb = make_grads(s, n, g, count, dstate.read().scaler.scale)
        for k in range(g - 1):
            zs.zs_grad_accum(ctx, [gb[k, r] for r in range(n)], zs.ZS_FP16, count, acc, k == 0)
        zs.zs_shard_step_async_oop(ctx, [gb[g - 1, r] for r in range(n)], zs.ZS_FP16, count,
                                   acc if g > 1 else None, g, *pairs, hp, sched, dstate)
    torch.cuda.synchronize()


@pytest.mark.parametrize("fused", [True, False])
@pytest.mark.parametrize("n,g", [(2, 3), (16, 2)])
def test_device_state_resume_equals_straight_run(zs, n, g, fused):
    """The device-resident out-of-place form under a WarmupDecayLR schedule:
    the checkpoint is the current state set and the device state (scale,
    hysteresis, Adam's step, iterations, learning rate), saved with torch.
    Restored into fresh buffers and a fresh context, the current set loaded as
    set 0, five more steps equal ten straight ones bit for bit."""
    count = 40_009
    sched = zs.make_schedule(zs.ZS_LR_WARMUP_DECAY, 0.0, 1e-3, 3, 12)

    def fresh_bufs():
        rng = np.random.default_rng(5)
        m0 = torch.from_numpy((rng.standard_normal(count) * 0.02).astype(np.float32)).cuda()
        return [[m0, torch.empty_like(m0)],
                [torch.zeros_like(m0), torch.empty_like(m0)],
                [torch.zeros_like(m0), torch.empty_like(m0)],
                [torch.zeros(count, dtype=torch.int16, device="cuda"),
                 torch.empty(count, dtype=torch.int16, device="cuda")]]

    def new_ctx():
        c = zs.Ctx()
        c.set_fused(zs.ZS_FUSED_ON if fused else zs.ZS_FUSED_OFF)
        return c

    ctx = new_ctx()
    straight, st_a = fresh_bufs(), zs.DeviceState(zs.zs_scaler_init(1024.0, 1.0, 3, 2, True))
    run_device(zs, ctx, straight, st_a, 1, 10, n, g, count, sched)
    half_way, st_b = fresh_bufs(), zs.DeviceState(zs.zs_scaler_init(1024.0, 1.0, 3, 2, True))
    run_device(zs, ctx, half_way, st_b, 1, 5, n, g, count, sched)
    d = st_b.read()
    cur = d.buf & 1
    buf = io.BytesIO()
    torch.save({"state": [p[cur].cpu() for p in half_way], "device_state": list(bytes(d))}, buf)
    ctx.close()
    buf.seek(0)
    ck = torch.load(buf)
    ctx2 = new_ctx()
    restored = [[x.cuda(), torch.empty_like(x.cuda())] for x in ck["state"]]
    ds = zs.zs_device_state.from_buffer_copy(bytes(ck["device_state"]))
    ds.buf = 0                                     # the loaded set is set 0
    st_c = zs.DeviceState(ds.scaler)
    st_c.buf.copy_(torch.frombuffer(bytearray(bytes(ds)), dtype=torch.uint8))
    run_device(zs, ctx2, restored, st_c, 6, 10, n, g, count, sched)
    a, c = st_a.read(), st_c.read()
    assert (a.step, a.iterations, a.scaler.scale, a.scaler.hyst_left, a.lr) == \
        (c.step, c.iterations, c.scaler.scale, c.scaler.hyst_left, c.lr)
    assert a.iterations == 10 and a.step == 9           # step 4 overflowed
    for pa, pc in zip(straight, restored):
        assert torch.equal(pa[a.buf & 1], pc[c.buf & 1])
    ctx2.close()
