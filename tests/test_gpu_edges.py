"""Degenerate inputs of the update, each against the oracle: bf16 gradients
up to and past the magnitude whose square leaves the fp32 range (up to the
bf16 maximum), zero gradients with decay, lr = 0, betas of 0, a large eps, a
very late Adam step, and fp16 gradients in the subnormal range."""
import numpy as np
import pytest
import torch

import oracle
from _helpers import STRESS_LR, dev16, host16, lib_half, ulps

pytestmark = pytest.mark.gpu

FP16, BF16 = 0, 1
REL, ABS = 1e-6, 1e-9


@pytest.fixture(scope="module")
def zs():
    import zero_mixed_precision_shard_gb300 as pkg
    torch.cuda.set_device(0)
    return pkg


@pytest.fixture(scope="module", params=["fused", "multi"])
def ctx(zs, request):
    """Every test runs with the fused single-kernel step (where the shard fits
    one co-resident grid) and with the multi-kernel path."""
    c = zs.Ctx()
    c.set_fused(zs.ZS_FUSED_ON if request.param == "fused" else zs.ZS_FUSED_OFF)
    yield c
    c.close()


def close(got, want, name):
    """1e-6 relative + 1e-9 absolute; equal infinities where the fp32 state no
    longer holds the value."""
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    assert (np.isinf(got) == np.isinf(want)).all(), name
    assert (np.sign(got[np.isinf(got)]) == np.sign(want[np.isinf(want)])).all(), name
    assert not np.isnan(got).any() and not np.isnan(want).any(), name
    f = np.isfinite(want)
    err = np.abs(got[f] - want[f])
    tol = REL * np.abs(want[f]) + ABS
    assert (err <= tol).all(), (name, float((err / tol).max()))


def run_steps(zs, ctx, dtype, n, G, grads_per_step, hp_vals, scale, master0):
    count = master0.shape[0]
    st = oracle.ShardState.from_master(master0, dtype)
    hp_o, hp = oracle.make_hparams(*hp_vals), zs.make_hparams(*hp_vals)
    dyn = dtype == FP16 and scale != 1.0
    sc_o = oracle.make_scaler(scale, 1.0, 1000, 1, dyn)
    sc = zs.zs_scaler_init(scale, 1.0, 1000, 1, dyn)
    master = torch.from_numpy(master0.copy()).cuda()
    m, v = torch.zeros_like(master), torch.zeros_like(master)
    half = torch.zeros(count, dtype=torch.int16, device="cuda")
    acc = torch.zeros_like(master)
    t = t_o = 0
    for grads in grads_per_step:
        ovf_o, t_o, _ = oracle.shard_step(grads, dtype, st, hp_o, t_o, sc_o)
        dg = [[dev16(x) for x in micro] for micro in grads]
        for k in range(G - 1):
            zs.zs_grad_accum(ctx, dg[k], dtype, count, acc, k == 0)
        ovf, ns = zs.zs_shard_step(ctx, dg[G - 1], dtype, count, acc, G, master, m, v, half, hp,
                                   t + 1, sc)
        assert ovf == ovf_o and ns == sc_o.scale
        if not ovf:
            t += 1
    assert t == t_o
    return st, master.cpu().numpy(), m.cpu().numpy(), v.cpu().numpy(), host16(half)


def big_bf16_steps(rng, n, G, count, big, steps=3):
    out = []
    for s in range(steps):
        vals = [[(rng.standard_normal(count) * 1e-2).astype(np.float32) for _ in range(n)]
                for _ in range(G)]
        if s == 0:
            for i, x in big.items():   # every rank and micro-step holds x: the mean is x
                for k in range(G):
                    for r in range(n):
                        vals[k][r][i] = x
        out.append([[lib_half(x, BF16) for x in micro] for micro in vals])
    return out


@pytest.mark.parametrize("n,G", [(1, 1), (2, 2), (4, 1)])
def test_bf16_gradients_up_to_the_fp32_square(zs, ctx, n, G):
    """bf16 mean gradients up to 1.5e19 in magnitude (squares up to 2.25e38,
    inside fp32): the fp32 update matches the fp64 oracle at every step, v
    finite on both sides."""
    rng = np.random.default_rng(40 + n + G)
    count = 10_007
    master0 = (rng.standard_normal(count) * 0.02).astype(np.float32)
    big = {5: 1.5e19, 6: -1.5e19, 7: 1e15, 100: -3e12, 101: 1e10, count - 1: 1.2e19}
    steps = big_bf16_steps(rng, n, G, count, big)
    st, p, m, v, h = run_steps(zs, ctx, BF16, n, G, steps, (STRESS_LR, 0.9, 0.999, 1e-8, 0.01),
                               1.0, master0)
    close(p, st.master, "master")
    close(m, st.m, "m")
    close(v, st.v, "v")
    assert np.isfinite(st.v).all() and ulps(h, st.half).max() <= 1
    # those elements moved by about lr in the first step, as Adam's first step does
    assert (np.abs(p[[5, 6]] - master0[[5, 6]]) > 0.5 * STRESS_LR).all()


@pytest.mark.parametrize("n,G", [(1, 1), (2, 2)])
def test_bf16_gradients_past_the_fp32_square(zs, ctx, n, G):
    """Beyond that, up to the bf16 maximum: g*g passes the fp32 maximum, and
    from ~5.8e20 (1-beta2)*g*g does too, so the stored v is +inf on both sides
    (the oracle rounds its fp64 v to fp32 for storage) -- but the first step's
    Adam term is still the exact moment's, about lr: the kernel takes the root
    of the new v as |g| * sqrt(beta2*v_old/g^2 + (1-beta2)) and scales the
    root, not v, by the bias correction.  Afterwards the Adam term is 0 on both
    sides (m_hat / inf) and decay alone moves those weights; no NaN anywhere."""
    rng = np.random.default_rng(77 + n + G)
    count = 4_099
    master0 = (rng.standard_normal(count) * 0.02).astype(np.float32)
    # every rank and micro-step holds x, so the fp32 sum holds n*G*x: the
    # largest stay below the fp32 maximum in that sum (else the step overflows)
    top = 1.0 / (n * G)
    big = {5: 2e19, 6: -7e19, 7: 5e20, 8: 1e30, 9: 3.3e38 * top, 10: -3.3e38 * top,
           count - 1: 3.38e38 * top}
    idx = sorted(big)
    steps = big_bf16_steps(rng, n, G, count, big)
    st, p, m, v, h = run_steps(zs, ctx, BF16, n, G, steps, (STRESS_LR, 0.9, 0.999, 1e-8, 0.01),
                               1.0, master0)
    close(p, st.master, "master")
    close(m, st.m, "m")
    close(v, st.v, "v")       # +inf where the fp32 state cannot hold v, on both sides
    assert ulps(h, st.half).max() <= 1
    assert np.isfinite(p).all() and np.isfinite(m).all() and not np.isnan(v).any()
    assert np.isinf(v[[8, 9, 10, count - 1]]).all() and np.isfinite(v[[5, 6, 7]]).all()
    # the first step moved those weights by about lr, as Adam's first step does
    assert (np.abs(p[idx] - master0[idx]) > 0.5 * STRESS_LR).all()


@pytest.mark.parametrize("hp_vals", [(STRESS_LR, 0.9, 0.999, 1e-8, 0.1),   # zero gradients, decay
                                     (0.0, 0.9, 0.999, 1e-8, 0.1),         # lr = 0
                                     (STRESS_LR, 0.0, 0.0, 1e-8, 0.0),     # betas of 0
                                     (STRESS_LR, 0.9, 0.999, 1e-3, 0.01)])  # large eps
def test_degenerate_hyper_parameters(zs, ctx, hp_vals):
    rng = np.random.default_rng(9)
    count = 4_099
    master0 = (rng.standard_normal(count) * 0.02).astype(np.float32)
    zero = hp_vals[1] == 0.9 and hp_vals[3] == 1e-8
    steps = []
    for s in range(4):
        x = np.zeros(count, np.float32) if zero else \
            (rng.standard_normal(count) * 1e-3 * 1024).astype(np.float32)
        steps.append([[lib_half(x, FP16), lib_half(-0.5 * x, FP16)]])
    st, p, m, v, h = run_steps(zs, ctx, FP16, 2, 1, steps, hp_vals, 1024.0, master0)
    close(p, st.master, "master")
    close(m, st.m, "m")
    close(v, st.v, "v")
    assert ulps(h, st.half).max() <= 1
    if hp_vals[0] == 0.0:
        assert p.tobytes() == master0.tobytes()              # lr = 0 moves nothing
    if zero:   # the Adam term is 0: decay alone, (1 - lr*wd) per step
        want = master0.astype(np.float64) * (1 - hp_vals[0] * hp_vals[4]) ** 4
        assert np.abs(p - want).max() <= 1e-6 * np.abs(want).max()


def test_late_step_and_subnormal_fp16_gradients(zs, ctx):
    """Adam step 10^6 (bias corrections ~1) via zs_apply, on fp16 gradients in
    the subnormal range under a 2^16 loss scale."""
    rng = np.random.default_rng(12)
    count = 8_193
    sub = (rng.integers(-1023, 1024, count) * 2.0 ** -24).astype(np.float32)   # fp16 subnormals
    g = lib_half(sub, FP16)
    assert (np.abs(sub) < 2.0 ** -14).all()
    master = (rng.standard_normal(count) * 0.02).astype(np.float32)
    m0 = (rng.standard_normal(count) * 1e-9).astype(np.float32)
    v0 = (rng.random(count) * 1e-19).astype(np.float32)
    acc = np.zeros(count, np.float32)
    oracle.reduce_accumulate([g], FP16, acc, first=True)
    hp_vals = (1e-4, 0.9, 0.999, 1e-8, 0.01)
    st = oracle.ShardState(master.copy(), m0.copy(), v0.copy(), np.zeros(count, np.uint16))
    oracle.adamw_apply(acc, 65536.0, st.master, st.m, st.v, st.half, FP16,
                       oracle.make_hparams(*hp_vals), 10 ** 6)
    d = [torch.from_numpy(a.copy()).cuda() for a in (master, m0, v0)]
    half = torch.zeros(count, dtype=torch.int16, device="cuda")
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    zs.zs_apply(ctx, flag, [dev16(g)], FP16, None, count, 65536.0, d[0], d[1], d[2], half,
                zs.make_hparams(*hp_vals), 10 ** 6)
    close(d[0].cpu().numpy(), st.master, "master")
    close(d[1].cpu().numpy(), st.m, "m")
    close(d[2].cpu().numpy(), st.v, "v")
    assert ulps(host16(half), st.half).max() <= 1
