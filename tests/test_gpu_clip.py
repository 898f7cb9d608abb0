"""Global-norm gradient clipping on the GPU against the oracle: the squared
norm (deterministic, within 1e-6 relative), the clipped update (state within
1e-6 relative + 1e-9 absolute, half within 1 ulp), the unclipped case equal
to the plain step bit for bit, and the two-phase form across shards."""
import numpy as np
import pytest
import torch

import oracle
from _helpers import STRESS_LR, assert_close, dev16, lib_half, ulps

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
    one co-resident grid; the norm then travels with its grid barrier) and
    with the multi-kernel path."""
    c = zs.Ctx()
    c.set_fused(zs.ZS_FUSED_ON if request.param == "fused" else zs.ZS_FUSED_OFF)
    yield c
    c.close()


def close(got, want, name):
    """1e-6 relative + 1e-9 absolute (these tests run at lr 3e-4)."""
    assert_close(got, want, name)


@pytest.mark.parametrize("dtype", [FP16, BF16])
@pytest.mark.parametrize("count", [1, 13, 4096, 1_000_003])
@pytest.mark.parametrize("form", ["acc", "slices", "acc+slices"])
def test_sumsq_matches_oracle(zs, ctx, dtype, count, form):
    rng = np.random.default_rng(count)
    n, div = 3, 3 * 2 * 512.0
    acc0 = (rng.standard_normal(count) * 0.3 * div).astype(np.float32)
    sl = [lib_half((rng.standard_normal(count) * 0.2 * 512).astype(np.float32), dtype)
          for _ in range(n)]
    final = np.zeros(count, np.float32) if form == "slices" else acc0.copy()
    if form != "acc":
        oracle.reduce_accumulate(sl, dtype, final, first=(form == "slices"))
    want = oracle.grad_sumsq(final, div)
    out = torch.zeros(1, dtype=torch.float64, device="cuda")
    acc = None if form == "slices" else torch.from_numpy(acc0).cuda()
    grads = None if form == "acc" else [dev16(s) for s in sl]
    zs.zs_grad_sumsq(ctx, grads, dtype, acc, count, div, out)
    got = out.item()
    assert abs(got - want) <= 1e-6 * want
    out2 = torch.zeros(1, dtype=torch.float64, device="cuda")
    zs.zs_grad_sumsq(ctx, grads, dtype, acc, count, div, out2)
    assert out2.item() == got   # deterministic


@pytest.mark.parametrize("dtype", [FP16, BF16])
@pytest.mark.parametrize("n,G,count,max_norm", [(1, 3, 50_001, 0.05), (2, 1, 8_191, 0.01),
                                                 (8, 2, 100_000, 0.1), (4, 1, 4_099, 1e6)])
def test_clipped_shard_steps(zs, ctx, dtype, n, G, count, max_norm):
    rng = np.random.default_rng(n * 7 + G)
    master0 = (rng.standard_normal(count) * 0.02).astype(np.float32)
    st = oracle.ShardState.from_master(master0, dtype)
    hp_v = (STRESS_LR, 0.9, 0.999, 1e-8, 0.01)
    hp_o, hp = oracle.make_hparams(*hp_v), zs.make_hparams(*hp_v)
    dyn = dtype == FP16
    sc_o = oracle.make_scaler(512.0 if dyn else 1.0, 1.0, 1000, 1, dyn)
    sc = zs.zs_scaler_init(sc_o.scale, 1.0, 1000, 1, dyn)
    master = torch.from_numpy(master0.copy()).cuda()
    m, v = torch.zeros_like(master), torch.zeros_like(master)
    half = torch.zeros(count, dtype=torch.int16, device="cuda")
    acc = torch.zeros(count, dtype=torch.float32, device="cuda")
    t = t_o = 0
    for s in range(1, 5):
        grads = [[lib_half((rng.standard_normal(count) * 1e-2 * sc_o.scale).astype(np.float32),
                           dtype) for _ in range(n)] for _ in range(G)]
        if s == 3:
            grads[0][0][5] = 0x7C00 if dtype == FP16 else 0x7F80
        ovf_o, t_o, _, norm_o = oracle.shard_step(grads, dtype, st, hp_o, t_o, sc_o,
                                                  max_norm=max_norm, return_norm=True)
        dg = [[dev16(x) for x in micro] for micro in grads]
        for k in range(G - 1):
            zs.zs_grad_accum(ctx, dg[k], dtype, count, acc, k == 0)
        ovf, ns, norm = zs.zs_shard_step_clipped(ctx, dg[G - 1], dtype, count, acc, G, master, m,
                                                 v, half, hp, t + 1, sc, max_norm)
        if not ovf:
            t += 1
        assert ovf == ovf_o and ns == sc_o.scale
        assert abs(norm - norm_o) <= 1e-6 * norm_o + 1e-30
    assert t == t_o == 3
    close(master.cpu().numpy(), st.master, "master")
    close(m.cpu().numpy(), st.m, "m")
    close(v.cpu().numpy(), st.v, "v")
    assert ulps(half.cpu().numpy().view(np.uint16), st.half).max() <= 1


def test_large_max_norm_equals_plain_step_bitwise(zs, ctx):
    rng = np.random.default_rng(5)
    n, count = 2, 30_011
    outs = []
    for clipped in (False, True):
        r2 = np.random.default_rng(6)
        master = torch.from_numpy((r2.standard_normal(count) * 0.02).astype(np.float32)).cuda()
        m, v = torch.zeros_like(master), torch.zeros_like(master)
        half = torch.zeros(count, dtype=torch.int16, device="cuda")
        sc = zs.zs_scaler_init(256.0, 1.0, 1000, 1, True)
        hp = zs.make_hparams(STRESS_LR, 0.9, 0.999, 1e-8, 0.0)
        g = [dev16(lib_half((r2.standard_normal(count) * 2.56).astype(np.float32), FP16))
             for _ in range(n)]
        if clipped:
            zs.zs_shard_step_clipped(ctx, g, FP16, count, None, 1, master, m, v, half, hp, 1, sc,
                                     1e9)
        else:
            zs.zs_shard_step(ctx, g, FP16, count, None, 1, master, m, v, half, hp, 1, sc)
        outs.append((master, m, v, half))
    for a, b in zip(*outs):
        assert torch.equal(a, b)
    del rng


def test_two_phase_clipping_across_shards(zs, ctx):
    """Four shards, one global norm: per-shard sums of squares added on the
    device, then each shard's clipped update; against the oracle's union."""
    rng = np.random.default_rng(21)
    psi, n = 40_000, 4
    psi_pad, E = oracle.partition(psi, n)
    hp_v = (STRESS_LR, 0.9, 0.999, 1e-8, 0.0)
    master0 = (rng.standard_normal(psi_pad) * 0.02).astype(np.float32)
    full = [lib_half((rng.standard_normal(psi_pad) * 0.3 * 256).astype(np.float32), FP16)
            for _ in range(n)]
    states = [oracle.ShardState.from_master(master0[q * E:(q + 1) * E], FP16) for q in range(n)]
    per = [[[np.ascontiguousarray(f[q * E:(q + 1) * E]) for f in full]] for q in range(n)]
    oracle.multi_shard_step(per, FP16, states, oracle.make_hparams(*hp_v), 0,
                            oracle.make_scaler(256.0), max_norm=0.5)
    fd = [dev16(f) for f in full]
    dev = [[torch.from_numpy(master0[q * E:(q + 1) * E].copy()).cuda(),
            torch.zeros(E, device="cuda"), torch.zeros(E, device="cuda"),
            torch.zeros(E, dtype=torch.int16, device="cuda")] for q in range(n)]
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    part = torch.zeros(n, dtype=torch.float64, device="cuda")
    div = float(n * 256.0)
    for q in range(n):
        zs.zs_reduce_check(ctx, [f[q * E:(q + 1) * E] for f in fd], FP16, E, None, True, flag)
        zs.zs_grad_sumsq(ctx, [f[q * E:(q + 1) * E] for f in fd], FP16, None, E, div, part[q:])
    total = part.sum().reshape(1).contiguous()
    for q in range(n):
        zs.zs_apply_clipped(ctx, flag, total, 0.5, [f[q * E:(q + 1) * E] for f in fd], FP16, None,
                            E, div, dev[q][0], dev[q][1], dev[q][2], dev[q][3],
                            zs.make_hparams(*hp_v), 1)
    for q in range(n):
        close(dev[q][0].cpu().numpy(), states[q].master, "master")
        close(dev[q][1].cpu().numpy(), states[q].m, "m")
        close(dev[q][2].cpu().numpy(), states[q].v, "v")
        assert ulps(dev[q][3].cpu().numpy().view(np.uint16), states[q].half).max() <= 1


@pytest.mark.parametrize("n,G", [(1, 1), (2, 2), (4, 2), (16, 1)])
def test_fused_norm_of_huge_sums(zs, ctx, n, G):
    """bf16 gradients near 1e30 (finite; their squares pass the fp32 maximum)
    beside ordinary ones: the norm fused into the last pass, on the re-read
    (n < 4) and the materialising (n >= 4) forms, matches the oracle's fp64
    norm, and the clipped step matches the oracle's state."""
    rng = np.random.default_rng(100 + n * 3 + G)
    count = 70_003
    master0 = (rng.standard_normal(count) * 0.02).astype(np.float32)
    st = oracle.ShardState.from_master(master0, BF16)
    hp_v = (STRESS_LR, 0.9, 0.999, 1e-8, 0.01)
    hp_o, hp = oracle.make_hparams(*hp_v), zs.make_hparams(*hp_v)
    sc_o = oracle.make_scaler(1.0, 1.0, 1000, 1, False)
    sc = zs.zs_scaler_init(1.0, 1.0, 1000, 1, False)
    master = torch.from_numpy(master0.copy()).cuda()
    m, v = torch.zeros_like(master), torch.zeros_like(master)
    half = torch.zeros(count, dtype=torch.int16, device="cuda")
    acc = torch.zeros(count, dtype=torch.float32, device="cuda")
    t = t_o = 0
    for s in range(1, 3):
        vals = [[(rng.standard_normal(count) * 1e-2).astype(np.float32) for _ in range(n)]
                for _ in range(G)]
        # both sides of the 1e18 split, in one 8-element vector and alone, and the tail
        for pos, x in ((5, 1e30), (6, 2e18), (7, 9e17), (4_001, -3e29), (40_000, 1.5e18),
                       (count - 1, 7e25)):
            vals[G - 1][n - 1][pos] = x * (1 + s)
        grads = [[lib_half(x, BF16) for x in micro] for micro in vals]
        ovf_o, t_o, _, norm_o = oracle.shard_step(grads, BF16, st, hp_o, t_o, sc_o,
                                                  max_norm=1.0, return_norm=True)
        dg = [[dev16(x) for x in micro] for micro in grads]
        for k in range(G - 1):
            zs.zs_grad_accum(ctx, dg[k], BF16, count, acc, k == 0)
        ovf, ns, norm = zs.zs_shard_step_clipped(ctx, dg[G - 1], BF16, count, acc, G, master,
                                                 m, v, half, hp, t + 1, sc, 1.0)
        if not ovf:
            t += 1
        assert ovf == ovf_o == 0 and ns == sc_o.scale
        assert norm_o > 1e29
        assert abs(norm - norm_o) <= 1e-6 * norm_o
    assert t == t_o == 2
    close(master.cpu().numpy(), st.master, "master")
    close(m.cpu().numpy(), st.m, "m")
    close(v.cpu().numpy(), st.v, "v")
    assert ulps(half.cpu().numpy().view(np.uint16), st.half).max() <= 1
