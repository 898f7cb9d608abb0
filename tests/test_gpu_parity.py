"""Parity of the CUDA path (through the C ABI) with the CPU oracle on the same
seeded inputs: bit-exact accumulators and flags, AdamW state within
1e-6 relative + 1e-9 absolute, half copies within 1 ulp, exact scales and skip
decisions.  Sizes span several CTAs' worth of vectors plus ragged tails."""
import numpy as np
import pytest
import torch

import oracle
import synth
from _helpers import STRESS_LR, assert_close, dev16, half_ulps, host16, lib_half, tol_ratio

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


def rand_grads(rng, n, count, dtype, scale=1024.0):
    out = []
    for r in range(n):
        x = rng.standard_normal(count) * 1e-3 * scale * np.exp2(rng.integers(-6, 6, count))
        x[rng.random(count) < 0.01] = 0.0
        x[rng.random(count) < 0.01] = -0.0
        out.append(lib_half(x.astype(np.float32), dtype))
    return out


def assert_state_close(got, want, name):
    """1e-6 relative + 1e-9 absolute, at every learning rate."""
    assert_close(got, want, name)


# ---------------------------------------------------------------- reduce

CASES = [(n, c) for n in (1, 2, 3, 4, 5, 8, 9, 16, 64) for c in (0, 1, 7, 8, 9, 1000, 65541)]
CASES += [(256, 4099), (255, 17)]


@pytest.mark.parametrize("dtype", [FP16, BF16])
@pytest.mark.parametrize("n,count", CASES)
def test_grad_accum_bit_exact(zs, ctx, dtype, n, count):
    rng = np.random.default_rng(1000 * n + count)
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    acc_d = torch.full((max(count, 1),), 123.0, dtype=torch.float32, device="cuda")
    acc_o = np.zeros(count, np.float32)
    for k in range(3):
        g = rand_grads(rng, n, count, dtype)
        zs.zs_reduce_check(ctx, [dev16(s) for s in g], dtype, count, acc_d, k == 0, flag)
        oracle.reduce_accumulate(g, dtype, acc_o, first=(k == 0))
    got = acc_d[:count].cpu().numpy()
    assert got.tobytes() == acc_o.tobytes()
    assert flag.item() == 0
    # check-only form: flag only, nothing written
    before = acc_d.clone()
    zs.zs_reduce_check(ctx, [dev16(s) for s in g], dtype, count, None, True, flag)
    assert flag.item() == 0 and torch.equal(before, acc_d)


def finite_patterns(dtype):
    """Every finite half bit pattern (both signs, zeros and subnormals included)."""
    b = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    exp = 0x7C00 if dtype == FP16 else 0x7F80
    return b[(b & exp) != exp]


# fp32 accumulator values the patterns are added onto: signed zeros, an fp32
# subnormal, values that absorb small halves or cancel large ones, and values
# near the fp32 maximum (bf16 halves there sum past it)
ACC_BASES = [0.0, -0.0, 1e-40, -1.0, 3.0517578125e-05, 65504.0 * 7, -2.5e9, 1.7e38, -3.0e38]


@pytest.mark.parametrize("dtype", [FP16, BF16])
@pytest.mark.parametrize("n", [1, 3])
def test_every_half_pattern_accumulates_exactly(zs, ctx, dtype, n):
    """Each finite half pattern added onto fp32 accumulators of several kinds
    (and onto +0 for the first micro-step), n ranks in order: the fp32 sums
    must equal the oracle's bit for bit, the flag its any-non-finite test."""
    pat = finite_patterns(dtype)
    count = pat.size * len(ACC_BASES) + 5           # + a ragged tail
    g = [np.resize(np.roll(pat, 997 * r), count) for r in range(n)]
    acc0 = np.resize(np.repeat(np.array(ACC_BASES, np.float32), pat.size), count)
    for first in (True, False):
        acc_o = acc0.copy()
        oracle.reduce_accumulate(g, dtype, acc_o, first)
        want_flag = oracle.any_nonfinite_f32(acc_o)
        acc_d = torch.from_numpy(acc0.copy()).cuda()
        flag = torch.zeros(1, dtype=torch.int32, device="cuda")
        zs.zs_reduce_check(ctx, [dev16(x) for x in g], dtype, count, acc_d, first, flag)
        got = acc_d.cpu().numpy()
        assert got.tobytes() == acc_o.tobytes(), np.flatnonzero(got.view(np.uint32)
                                                                != acc_o.view(np.uint32))[:8]
        assert flag.item() == want_flag


@pytest.mark.parametrize("dtype", [FP16, BF16])
@pytest.mark.parametrize("where", ["first", "body", "tail", "last_rank"])
@pytest.mark.parametrize("kind", ["inf", "-inf", "nan"])
@pytest.mark.parametrize("n", [1, 5])
def test_overflow_flag(zs, ctx, dtype, where, kind, n):
    rng = np.random.default_rng(7)
    count = 8 * 1000 + 5
    g = rand_grads(rng, n, count, dtype)
    bits = {"inf": 0x7C00 if dtype == FP16 else 0x7F80,
            "-inf": 0xFC00 if dtype == FP16 else 0xFF80,
            "nan": 0x7E00 if dtype == FP16 else 0x7FC0}[kind]
    r, i = {"first": (0, 0), "body": (2, 4321), "tail": (1, count - 2),
            "last_rank": (n - 1, count // 2)}[where]
    r = min(r, n - 1)
    g[r][i] = bits
    assert oracle.any_nonfinite(g, dtype, count) == 1
    for acc in (torch.zeros(count, dtype=torch.float32, device="cuda"), None):
        flag = torch.zeros(1, dtype=torch.int32, device="cuda")
        zs.zs_reduce_check(ctx, [dev16(s) for s in g], dtype, count, acc, True, flag)
        assert flag.item() == 1


def test_bf16_finite_sum_overflow_is_flagged(zs, ctx):
    big = lib_half(np.full(16, 3.0e38, np.float32), BF16)
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    acc = torch.zeros(16, dtype=torch.float32, device="cuda")
    zs.zs_reduce_check(ctx, [dev16(big), dev16(big)], BF16, 16, acc, True, flag)
    assert flag.item() == 1 and torch.isinf(acc).all()
    acc_o = np.zeros(16, np.float32)
    oracle.reduce_accumulate([big, big], BF16, acc_o, True)
    assert oracle.any_nonfinite_f32(acc_o) == 1


# ---------------------------------------------------------------- apply

def random_state(rng, count):
    master = (rng.standard_normal(count) * 0.02).astype(np.float32)
    m = (rng.standard_normal(count) * 1e-4).astype(np.float32)
    v = (rng.random(count) * 1e-7).astype(np.float32)
    return master, m, v


@pytest.mark.parametrize("dtype", [FP16, BF16])
@pytest.mark.parametrize("count", [1, 9, 4096, 100003])
@pytest.mark.parametrize("t,wd", [(1, 0.0), (2, 0.01), (10, 0.1), (1000, 0.0)])
def test_apply_matches_oracle(zs, ctx, dtype, count, t, wd):
    rng = np.random.default_rng(count + t)
    master, m, v = random_state(rng, count)
    n, g, S = 8, 4, 65536.0
    acc = (rng.standard_normal(count) * 1e-3 * n * g * S).astype(np.float32)
    acc[:min(count, 3)] = 0.0
    hp_o = oracle.make_hparams(1e-4, 0.9, 0.999, 1e-8, wd)
    st = oracle.ShardState(master.copy(), m.copy(), v.copy(), np.zeros(count, np.uint16))
    oracle.adamw_apply(acc, n * g * S, st.master, st.m, st.v, st.half, dtype, hp_o, t)
    d = [torch.from_numpy(a.copy()).cuda() for a in (acc, master, m, v)]
    half = torch.zeros(count, dtype=torch.int16, device="cuda")
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    hp = zs.make_hparams(1e-4, 0.9, 0.999, 1e-8, wd)
    zs.zs_apply(ctx, flag, None, dtype, d[0], count, n * g * S, d[1], d[2], d[3], half, hp, t)
    assert_state_close(d[1].cpu().numpy(), st.master, "master")
    assert_state_close(d[2].cpu().numpy(), st.m, "m")
    assert_state_close(d[3].cpu().numpy(), st.v, "v")
    assert half_ulps(host16(half), st.half).max() <= 1
    # a set flag writes nothing
    flag.fill_(1)
    snap = [x.clone() for x in d[1:]] + [half.clone()]
    zs.zs_apply(ctx, flag, None, dtype, d[0], count, n * g * S, d[1], d[2], d[3], half, hp, t + 1)
    for a, b in zip(snap, d[1:] + [half]):
        assert torch.equal(a, b)


@pytest.mark.parametrize("dtype", [FP16, BF16])
@pytest.mark.parametrize("with_acc", [False, True])
def test_apply_recompute_matches_oracle(zs, ctx, dtype, with_acc):
    rng = np.random.default_rng(11)
    n, count, S = 3, 50001, 256.0
    master, m, v = random_state(rng, count)
    g_prev = rand_grads(rng, n, count, dtype, S)
    g_last = rand_grads(rng, n, count, dtype, S)
    acc_o = np.zeros(count, np.float32)
    G = 1
    if with_acc:
        oracle.reduce_accumulate(g_prev, dtype, acc_o, True)
        G = 2
    oracle.reduce_accumulate(g_last, dtype, acc_o, not with_acc)
    hp_o = oracle.make_hparams(STRESS_LR, 0.9, 0.999, 1e-8, 0.01)
    st = oracle.ShardState(master.copy(), m.copy(), v.copy(), np.zeros(count, np.uint16))
    oracle.adamw_apply(acc_o, n * G * S, st.master, st.m, st.v, st.half, dtype, hp_o, 3)
    acc = None
    if with_acc:
        acc = torch.zeros(count, dtype=torch.float32, device="cuda")
        f0 = torch.zeros(1, dtype=torch.int32, device="cuda")
        zs.zs_reduce_check(ctx, [dev16(s) for s in g_prev], dtype, count, acc, True, f0)
    d = [torch.from_numpy(a.copy()).cuda() for a in (master, m, v)]
    half = torch.zeros(count, dtype=torch.int16, device="cuda")
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    hp = zs.make_hparams(STRESS_LR, 0.9, 0.999, 1e-8, 0.01)
    zs.zs_apply(ctx, flag, [dev16(s) for s in g_last], dtype, acc, count, n * G * S, d[0], d[1],
                d[2], half, hp, 3)
    assert_state_close(d[0].cpu().numpy(), st.master, "master")
    assert_state_close(d[1].cpu().numpy(), st.m, "m")
    assert_state_close(d[2].cpu().numpy(), st.v, "v")
    assert half_ulps(host16(half), st.half).max() <= 1


# ---------------------------------------------------------------- whole steps

def run_shard_steps(zs, ctx, dtype, n, G, count, steps, seed, inject=None, acc_mode="auto",
                    window=3, hysteresis=1, consecutive=False, lr=STRESS_LR, check_state=True):
    """Drive zs_grad_accum + zs_shard_step on the GPU and oracle.shard_step on
    the host for `steps` steps; the oracle's scale drives input generation.
    Flags, scales and counters must be equal at every step; with check_state,
    master/m/v must be within the parity bar at the end."""
    rng = np.random.default_rng(seed)
    master0 = (rng.standard_normal(count) * 0.02).astype(np.float32)
    st = oracle.ShardState.from_master(master0, dtype)
    hp_vals = (lr, 0.9, 0.999, 1e-8, 0.01)
    hp_o = oracle.make_hparams(*hp_vals)
    dynamic = dtype == FP16
    sc_o = oracle.make_scaler(1024.0 if dynamic else 1.0, 1.0, window, hysteresis, dynamic,
                              consecutive)
    sc = zs.zs_scaler_init(sc_o.scale, 1.0, window, hysteresis, dynamic, consecutive)
    hp = zs.make_hparams(*hp_vals)
    master = torch.from_numpy(master0.copy()).cuda()
    m = torch.zeros_like(master)
    v = torch.zeros_like(master)
    half = torch.zeros(count, dtype=torch.int16, device="cuda")
    acc = torch.zeros(count, dtype=torch.float32, device="cuda")
    if acc_mode == "none":
        acc = None
    t_o = t = 0
    flags = []
    for s in range(1, steps + 1):
        grads = [rand_grads(rng, n, count, dtype, sc_o.scale) for _ in range(G)]
        if inject and s in inject:
            k, r, i, bits = inject[s]
            grads[k][r][i] = bits
        ovf_o, t_o, _ = oracle.shard_step(grads, dtype, st, hp_o, t_o, sc_o)
        dg = [[dev16(x) for x in micro] for micro in grads]
        for k in range(G - 1):
            zs.zs_grad_accum(ctx, dg[k], dtype, count, acc, k == 0)
        ovf, new_scale = zs.zs_shard_step(ctx, dg[G - 1], dtype, count, acc, G, master, m, v,
                                          half, hp, t + 1, sc)
        if not ovf:
            t += 1
        assert ovf == ovf_o, f"step {s}"
        assert new_scale == sc_o.scale and sc.scale == sc_o.scale, f"step {s}"
        assert (sc.clean_count, sc.hyst_left) == (sc_o.clean_count, sc_o.hyst_left)
        flags.append(ovf)
    assert t == t_o
    if check_state:
        assert_state_close(master.cpu().numpy(), st.master, "master")
        assert_state_close(m.cpu().numpy(), st.m, "m")
        assert_state_close(v.cpu().numpy(), st.v, "v")
        assert half_ulps(host16(half), st.half).max() <= 1
    return flags, (master, m, v, half), st


@pytest.mark.parametrize("dtype", [FP16, BF16])
@pytest.mark.parametrize("n,G,count", [(1, 1, 4099), (2, 3, 10007), (4, 1, 8192 + 3),
                                       (8, 2, 20011), (16, 1, 777)])
def test_shard_step_sequence(zs, ctx, dtype, n, G, count):
    inf = 0x7C00 if dtype == FP16 else 0x7F80
    inject = {3: (G - 1, n - 1, count - 1, inf), 5: (0, 0, count // 2, 0x7E00 if dtype == FP16
                                                      else 0x7FC0)}
    flags, _, _ = run_shard_steps(zs, ctx, dtype, n, G, count, 10, seed=n * 100 + G,
                                  inject=inject)
    assert flags == [0, 0, 1, 0, 1, 0, 0, 0, 0, 0]


@pytest.mark.parametrize("dtype", [FP16, BF16])
@pytest.mark.parametrize("lr", [1e-4, 1e-3])
def test_shard_step_drift_by_learning_rate(zs, ctx, dtype, lr, capsys):
    """The fp32 state's distance from the fp64 oracle after 10 steps, printed as
    a fraction of the parity bar.  At lr 1e-4 it is held to the bar.  At
    lr 1e-3 (above every workload's) only the exact results are checked and the
    ratio is reported: each step both sides round p to fp32, and where their
    unrounded values straddle a rounding boundary p differs by one ulp, an
    absolute amount that grows with how far p moves, so with lr."""
    inf = 0x7C00 if dtype == FP16 else 0x7F80
    flags, (master, m, v, half), st = run_shard_steps(
        zs, ctx, dtype, 8, 2, 20011, 10, seed=77, inject={4: (1, 7, 5, inf)}, lr=lr,
        check_state=False)
    assert flags == [0, 0, 0, 1, 0, 0, 0, 0, 0, 0]
    ratios = {k: tol_ratio(d.cpu().numpy(), w) for k, d, w in
              (("master", master, st.master), ("m", m, st.m), ("v", v, st.v))}
    with capsys.disabled():
        print(f"\n  lr {lr:g} {'fp16' if dtype == FP16 else 'bf16'}: worst error / bound "
              + ", ".join(f"{k} {r:.3f}" for k, r in ratios.items()))
    assert half_ulps(host16(half), st.half).max() <= 1
    if lr <= 3e-4:
        assert max(ratios.values()) <= 1.0, ratios


def test_hysteresis_two(zs, ctx):
    """hysteresis 2: the scale halves on every second overflow since the last
    decrease; the device scaler must follow the oracle's step by step."""
    inf = 0x7C00
    inject = {s: (0, 0, 17, inf) for s in (1, 3, 4, 5, 9)}
    flags, _, _ = run_shard_steps(zs, ctx, FP16, 2, 1, 1001, 10, seed=3, inject=inject,
                                  window=2, hysteresis=2)
    assert flags == [1, 0, 1, 1, 1, 0, 0, 0, 1, 0]


@pytest.mark.parametrize("consecutive", [False, True])
def test_consecutive_hysteresis(zs, ctx, consecutive):
    """hysteresis 2 with and without consecutive_hysteresis: the device scaler
    follows the oracle step by step (the two settings diverge at step 3)."""
    inject = {s: (0, 0, 17, 0x7C00) for s in (1, 3, 4, 7, 9, 10)}
    flags, _, _ = run_shard_steps(zs, ctx, FP16, 2, 1, 1001, 11, seed=4, inject=inject,
                                  window=100, hysteresis=2, consecutive=consecutive)
    assert flags == [1, 0, 1, 1, 0, 0, 1, 0, 1, 1, 0]


@pytest.mark.parametrize("n", [4, 8])
def test_materialise_and_recompute_agree_bitwise(zs, ctx, n):
    _, a, _ = run_shard_steps(zs, ctx, FP16, n, 1, 5003, 4, seed=5, acc_mode="auto")
    _, b, _ = run_shard_steps(zs, ctx, FP16, n, 1, 5003, 4, seed=5, acc_mode="none")
    for x, y in zip(a, b):
        assert torch.equal(x, y)


def test_zero_count_step_still_updates_scale(zs, ctx):
    sc = zs.zs_scaler_init(1024.0, 1.0, 1, 1, True)
    e = torch.zeros(8, dtype=torch.float32, device="cuda")
    h = torch.zeros(8, dtype=torch.int16, device="cuda")
    g = [torch.zeros(8, dtype=torch.int16, device="cuda")]
    ovf, s = zs.zs_shard_step(ctx, g, FP16, 0, None, 1, e, e, e, h, zs.make_hparams(1e-3), 1, sc)
    assert ovf == 0 and s == 2048.0


def test_flat_1m_two_ranks_all_shards(zs, ctx):
    """The 2-rank flat workload (Ψ = 2^20, fp16, +inf at step 5 on rank 1) in
    full: both shards per step with one global flag (two-phase calls),
    against the oracle's union of shard steps."""
    wl = synth.WORKLOADS["flat-1m-n2"]
    psi_pad, E = oracle.partition(wl.psi, wl.n)
    idx = np.arange(wl.psi, dtype=np.int64)
    master0 = synth.host_master(wl, idx)
    states = [oracle.ShardState.from_master(master0[q * E:(q + 1) * E], FP16) for q in range(2)]
    hp_o = oracle.make_hparams(wl.lr, wl.beta1, wl.beta2, wl.eps, wl.weight_decay)
    sc_o = oracle.make_scaler(wl.scale0, wl.min_scale, wl.window, wl.hysteresis, wl.dynamic)
    hp = zs.make_hparams(wl.lr, wl.beta1, wl.beta2, wl.eps, wl.weight_decay)
    sc = zs.zs_scaler_init(wl.scale0, wl.min_scale, wl.window, wl.hysteresis, wl.dynamic)
    dev = [dict(master=torch.from_numpy(master0[q * E:(q + 1) * E].copy()).cuda(),
                m=torch.zeros(E, device="cuda"), v=torch.zeros(E, device="cuda"),
                half=torch.zeros(E, dtype=torch.int16, device="cuda")) for q in range(2)]
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    t_o = t = 0
    flags = []
    for s in range(1, wl.steps + 1):
        full = [synth.host_grad_bits(wl, idx, s, 1, r, sc_o.scale) for r in range(2)]
        per = [[[np.ascontiguousarray(f[q * E:(q + 1) * E]) for f in full]] for q in range(2)]
        ovf_o, t_o, _ = oracle.multi_shard_step(per, FP16, states, hp_o, t_o, sc_o)
        full_d = [dev16(f) for f in full]
        flag.zero_()
        for q in range(2):  # n = 2 < 4: check pass, then the update re-reads the slices
            zs.zs_reduce_check(ctx, [f[q * E:(q + 1) * E] for f in full_d], FP16, E, None, True,
                               flag)
        for q in range(2):
            zs.zs_apply(ctx, flag, [f[q * E:(q + 1) * E] for f in full_d], FP16, None, E,
                        float(wl.n * wl.g * sc.scale), dev[q]["master"], dev[q]["m"],
                        dev[q]["v"], dev[q]["half"], hp, t + 1)
        ovf = zs.zs_scaler_update(ctx, flag, sc)
        if not ovf:
            t += 1
        assert ovf == ovf_o and sc.scale == sc_o.scale
        flags.append(ovf)
    assert flags == [0, 0, 0, 0, 1, 0, 0, 0, 0, 0] and sc.scale == 2.0 ** 15 and t == t_o == 9
    for q in range(2):
        assert_state_close(dev[q]["master"].cpu().numpy(), states[q].master, "master")
        assert_state_close(dev[q]["m"].cpu().numpy(), states[q].m, "m")
        assert_state_close(dev[q]["v"].cpu().numpy(), states[q].v, "v")
        assert half_ulps(host16(dev[q]["half"]), states[q].half).max() <= 1


def test_bucketed_calls_equal_whole_shard(zs, ctx):
    rng = np.random.default_rng(9)
    n, count, bucket = 8, 100_000, 9_992
    g = [rand_grads(rng, n, count, FP16) for _ in range(2)]
    master, m, v = random_state(rng, count)
    hp = zs.make_hparams(1e-3, 0.9, 0.999, 1e-8, 0.01)
    outs = []
    for bsz in (count, bucket):
        acc = torch.zeros(count, dtype=torch.float32, device="cuda")
        d = [torch.from_numpy(a.copy()).cuda() for a in (master, m, v)]
        half = torch.zeros(count, dtype=torch.int16, device="cuda")
        flag = torch.zeros(1, dtype=torch.int32, device="cuda")
        gd = [[dev16(x) for x in micro] for micro in g]
        for b in range(0, count, bsz):
            e = min(count, b + bsz)
            for k in range(2):
                zs.zs_reduce_check(ctx, [x[b:e] for x in gd[k]], FP16, e - b, acc[b:e], k == 0,
                                   flag)
        for b in range(0, count, bsz):
            e = min(count, b + bsz)
            zs.zs_apply(ctx, flag, None, FP16, acc[b:e], e - b, n * 2 * 1024.0, d[0][b:e],
                        d[1][b:e], d[2][b:e], half[b:e], hp, 1)
        outs.append([acc] + d + [half])
    for x, y in zip(*outs):
        assert torch.equal(x, y)


def test_argument_errors(zs, ctx):
    x = torch.zeros(64, dtype=torch.float32, device="cuda")
    h = torch.zeros(64, dtype=torch.int16, device="cuda")
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    with pytest.raises(zs.ZsError) as e:
        zs.zs_grad_accum(ctx, [h[1:]], FP16, 8, x, True)
    assert e.value.status == zs.ZS_ERR_ALIGN
    with pytest.raises(zs.ZsError) as e:
        zs.zs_grad_accum(ctx, [h], 7, 8, x, True)
    assert e.value.status == zs.ZS_ERR_DTYPE
    with pytest.raises(zs.ZsError) as e:
        zs.zs_grad_accum(ctx, [], FP16, 8, x, True)
    assert e.value.status == zs.ZS_ERR_ARG
    with pytest.raises(zs.ZsError) as e:
        zs.zs_apply(ctx, flag, None, FP16, x, 8, 1.0, x, x, x, h, zs.make_hparams(1e-3), 0)
    assert e.value.status == zs.ZS_ERR_ARG
    assert "step" in zs.lib.zs_last_error(ctx.handle).decode()
    with pytest.raises(zs.ZsError) as e:
        zs.zs_grad_accum(ctx, [h] * 257, FP16, 8, x, True)
    assert e.value.status == zs.ZS_ERR_ARG


def test_copy_probe_copies(zs, ctx):
    src = torch.arange(1 << 20, dtype=torch.int32, device="cuda")
    dst = torch.zeros_like(src)
    zs.zs_copy_peak(ctx, src, dst, src.numel() * 4, False)
    assert torch.equal(src, dst)
    zs.zs_copy_peak(ctx, src, dst, src.numel() * 4, True)


def test_timing_counters_over_many_launches(zs):
    """Per-kernel event timing: every launch is counted, finished records are
    folded without blocking, and the totals survive more than a thousand
    launches with timing left on."""
    ctx = zs.Ctx()
    count = 4096
    g = [torch.zeros(count, dtype=torch.int16, device="cuda")]
    acc = torch.zeros(count, dtype=torch.float32, device="cuda")
    ctx.set_timing(True)
    for k in range(1500):
        zs.zs_grad_accum(ctx, g, FP16, count, acc, k == 0)
    ms, n_later, el = ctx.timing(zs.ZS_KERNEL_REDUCE)
    _, n_first, _ = ctx.timing(zs.ZS_KERNEL_REDUCE_FIRST)
    assert n_first == 1 and n_later == 1499 and el == 1499 * count and ms > 0
    ctx.timing_reset()
    assert ctx.timing(zs.ZS_KERNEL_REDUCE) == (0.0, 0, 0)
    assert ctx.launch_count == 1500
    ctx.close()


def test_context_flag_is_the_step_flag(zs):
    """zs_ctx_overflow_flag exposes the flag zs_grad_accum ORs into: a caller
    can hand it to the two-phase calls (or all-reduce it) and zs_shard_step
    clears it."""
    ctx = zs.Ctx()
    count = 1000
    bad = np.zeros(count, np.uint16)
    bad[3] = 0x7C00
    acc = torch.zeros(count, dtype=torch.float32, device="cuda")
    zs.zs_grad_accum(ctx, [dev16(bad)], FP16, count, acc, True)
    sc = zs.zs_scaler_init(64.0, 1.0, 1000, 1, True)
    assert zs.zs_scaler_update(ctx, ctx.overflow_flag_ptr, sc) == 1 and sc.scale == 32.0
    master = torch.zeros(count, dtype=torch.float32, device="cuda")
    m, v = torch.zeros_like(master), torch.zeros_like(master)
    half = torch.zeros(count, dtype=torch.int16, device="cuda")
    good = dev16(np.zeros(count, np.uint16))
    ovf, _ = zs.zs_shard_step(ctx, [good], FP16, count, acc, 2, master, m, v, half,
                              zs.make_hparams(1e-3), 1, sc)
    assert ovf == 1   # micro-step 1's inf still counts
    ovf, _ = zs.zs_shard_step(ctx, [good], FP16, count, None, 1, master, m, v, half,
                              zs.make_hparams(1e-3), 1, sc)
    assert ovf == 0   # the previous step cleared the flag
    ctx.close()


def test_two_contexts_on_two_streams(zs):
    """Contexts are independent: two shards stepped concurrently on two
    streams (each context with its own flag) equal the same steps run one
    after the other."""
    rng = np.random.default_rng(55)
    count, n = 200_003, 4
    grads = [[rand_grads(rng, n, count, FP16, 256.0)] for _ in range(2)]
    grads[1][0][2][9] = 0x7C00   # shard 1 overflows, shard 0 does not
    master0 = [(rng.standard_normal(count) * 0.02).astype(np.float32) for _ in range(2)]

    def run(concurrent):
        ctxs = [zs.Ctx(), zs.Ctx()]
        streams = [torch.cuda.Stream(), torch.cuda.Stream()]
        outs = []
        bufs = []
        for q in range(2):
            master = torch.from_numpy(master0[q].copy()).cuda()
            bufs.append((master, torch.zeros_like(master), torch.zeros_like(master),
                         torch.zeros(count, dtype=torch.int16, device="cuda"),
                         torch.zeros(count, dtype=torch.float32, device="cuda"),
                         [dev16(x) for x in grads[q][0]]))
        torch.cuda.synchronize()
        scalers = [zs.zs_scaler_init(256.0, 1.0, 1000, 1, True) for _ in range(2)]
        res = [None, None]
        import threading

        def work(q):
            master, m, v, half, acc, g = bufs[q]
            res[q] = zs.zs_shard_step(ctxs[q], g, FP16, count, acc, 1, master, m, v, half,
                                      zs.make_hparams(1e-4), 1, scalers[q], streams[q])
        if concurrent:
            ts = [threading.Thread(target=work, args=(q,)) for q in range(2)]
            for t in ts:
                t.start()
            for t in ts:
                t.join()
        else:
            for q in range(2):
                work(q)
        torch.cuda.synchronize()
        for q in range(2):
            outs.append([b.clone() for b in bufs[q][:4]])
            ctxs[q].close()
        return res, outs

    r1, o1 = run(True)
    r2, o2 = run(False)
    assert r1 == r2 and r1[0][0] == 0 and r1[1][0] == 1
    for a, b in zip(o1, o2):
        for x, y in zip(a, b):
            assert torch.equal(x, y)


def test_default_stream_is_the_current_torch_stream(zs):
    """A call given no stream launches on the calling thread's current torch
    stream: the default one, or the one a `torch.cuda.stream` block makes
    current (the work is then ordered on it alone)."""
    assert zs._stream(None) == torch.cuda.current_stream().cuda_stream
    side = torch.cuda.Stream()
    ctx = zs.Ctx()
    try:
        count = 1 << 20
        g = [torch.full((count,), 0x3C00, dtype=torch.int16, device="cuda")]   # fp16 1.0
        acc = torch.zeros(count, dtype=torch.float32, device="cuda")
        torch.cuda.synchronize()
        with torch.cuda.stream(side):
            assert zs._stream(None) == side.cuda_stream != torch.cuda.default_stream().cuda_stream
            for k in range(3):
                zs.zs_grad_accum(ctx, g, FP16, count, acc, k == 0)
        side.synchronize()
        assert torch.all(acc == 3.0)
        assert zs._stream(None) == torch.cuda.current_stream().cuda_stream
    finally:
        ctx.close()


def test_timing_skips_launches_captured_into_a_graph(zs):
    """With timing on, a launch captured into a CUDA graph records no events
    (they would be timed once per capture, and could not be waited on after
    the graph is gone): the counters hold the uncaptured launches only and stay
    readable after the graph is destroyed."""
    ctx = zs.Ctx()
    ctx.set_timing(True)
    count = 4096
    g = [torch.zeros(count, dtype=torch.int16, device="cuda")]
    acc = torch.zeros(count, dtype=torch.float32, device="cuda")
    zs.zs_grad_accum(ctx, g, FP16, count, acc, True)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        zs.zs_grad_accum(ctx, g, FP16, count, acc, False)
    graph.replay()
    graph.replay()
    torch.cuda.synchronize()
    assert ctx.timing(zs.ZS_KERNEL_REDUCE_FIRST)[1] == 1
    assert ctx.timing(zs.ZS_KERNEL_REDUCE)[1] == 0
    del graph
    zs.zs_grad_accum(ctx, g, FP16, count, acc, False)
    assert ctx.timing(zs.ZS_KERNEL_REDUCE)[1] == 1
    ctx.close()
