"""Checkpoint/resume and run-to-run determinism of the shard step.  All state
is caller-owned (master, m, v, half copy, scaler, Adam's step count), so
saving it after 5 steps, reloading it into fresh buffers and a fresh context
and running 5 more steps must equal 10 straight steps bit for bit."""
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
