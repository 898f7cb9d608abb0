"""The half-precision accumulator variant on the GPU against the oracle:
bit-exact half accumulators and flags (including sums that round past the
fp16 maximum), and multi-step state within 1e-6 relative + 1e-9 absolute."""
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
    """Every test runs with the fused single-kernel step (the shards here fit
    one co-resident grid) and with the multi-kernel path."""
    c = zs.Ctx()
    c.set_fused(zs.ZS_FUSED_ON if request.param == "fused" else zs.ZS_FUSED_OFF)
    yield c
    c.close()


def close(got, want, name):
    """1e-6 relative + 1e-9 absolute (these tests run at lr 3e-4)."""
    assert_close(got, want, name)


@pytest.mark.parametrize("dtype", [FP16, BF16])
@pytest.mark.parametrize("n,count", [(1, 1), (1, 65541), (2, 9), (5, 10007), (16, 4099)])
def test_halfacc_accumulate_bit_exact(zs, ctx, dtype, n, count):
    rng = np.random.default_rng(n + count)
    acc_d = torch.zeros(count, dtype=torch.int16, device="cuda")
    acc_o = np.zeros(count, np.uint16)
    for k in range(3):
        g = [lib_half((rng.standard_normal(count) * 300).astype(np.float32), dtype)
             for _ in range(n)]
        zs.zs_grad_accum_halfacc(ctx, [dev16(x) for x in g], dtype, count, acc_d, k == 0)
        oracle.reduce_accumulate_half(g, dtype, acc_o, k == 0)
    assert acc_d.cpu().numpy().view(np.uint16).tobytes() == acc_o.tobytes()


@pytest.mark.parametrize("dtype", [FP16, BF16])
@pytest.mark.parametrize("n", [1, 2])
def test_halfacc_every_pattern_bit_exact(zs, ctx, dtype, n):
    """Every finite half pattern as the carried accumulator, with n ranks' halves
    (the patterns in other orders) added on: the rounded sums must equal the
    oracle's bit for bit, sums past the half maximum included."""
    b = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    exp = 0x7C00 if dtype == FP16 else 0x7F80
    pat = b[(b & exp) != exp]
    count = pat.size + 3
    acc0 = np.resize(pat, count)
    g = [np.resize(np.roll(pat[::-1], 4099 * r), count) for r in range(n)]
    acc_o = acc0.copy()
    oracle.reduce_accumulate_half(g, dtype, acc_o, False)
    acc_d = dev16(acc0)
    zs.zs_grad_accum_halfacc(ctx, [dev16(x) for x in g], dtype, count, acc_d, False)
    assert acc_d.cpu().numpy().view(np.uint16).tobytes() == acc_o.tobytes()
    # the first micro-step: +0 then the ranks in order
    acc_o = np.zeros(count, np.uint16)
    oracle.reduce_accumulate_half(g, dtype, acc_o, True)
    zs.zs_grad_accum_halfacc(ctx, [dev16(x) for x in g], dtype, count, acc_d, True)
    assert acc_d.cpu().numpy().view(np.uint16).tobytes() == acc_o.tobytes()


def test_halfacc_sum_rounding_past_fp16_max_overflows(zs, ctx):
    count = 17
    big = lib_half(np.full(count, 40000.0, np.float32), FP16)
    acc = torch.zeros(count, dtype=torch.int16, device="cuda")
    master = torch.full((count,), 0.5, dtype=torch.float32, device="cuda")
    m, v = torch.zeros_like(master), torch.zeros_like(master)
    half = torch.zeros(count, dtype=torch.int16, device="cuda")
    sc = zs.zs_scaler_init(1024.0, 1.0, 1000, 1, True)
    zs.zs_grad_accum_halfacc(ctx, [dev16(big)], FP16, count, acc, True)
    ovf, ns = zs.zs_shard_step_halfacc(ctx, [dev16(big)], FP16, count, acc, 2, master, m, v, half,
                                       zs.make_hparams(1e-3), 1, sc)
    assert ovf == 1 and ns == 512.0
    assert torch.all(master == 0.5)


@pytest.mark.parametrize("dtype", [FP16, BF16])
@pytest.mark.parametrize("n,G,count", [(1, 8, 30_011), (4, 2, 20_000), (16, 1, 5_003)])
def test_halfacc_shard_steps(zs, ctx, dtype, n, G, count):
    rng = np.random.default_rng(n * 3 + G)
    master0 = (rng.standard_normal(count) * 0.02).astype(np.float32)
    st = oracle.ShardState.from_master(master0, dtype)
    dyn = dtype == FP16
    sc_o = oracle.make_scaler(256.0 if dyn else 1.0, 1.0, 3, 1, dyn)
    sc = zs.zs_scaler_init(sc_o.scale, 1.0, 3, 1, dyn)
    hp_v = (STRESS_LR, 0.9, 0.999, 1e-8, 0.01)
    hp_o, hp = oracle.make_hparams(*hp_v), zs.make_hparams(*hp_v)
    master = torch.from_numpy(master0.copy()).cuda()
    m, v = torch.zeros_like(master), torch.zeros_like(master)
    half = torch.zeros(count, dtype=torch.int16, device="cuda")
    acc = torch.zeros(count, dtype=torch.int16, device="cuda")
    t = t_o = 0
    for s in range(1, 9):
        grads = [[lib_half((rng.standard_normal(count) * 1e-2 * sc_o.scale).astype(np.float32),
                           dtype) for _ in range(n)] for _ in range(G)]
        if s == 4:
            grads[0][n - 1][count // 3] = 0x7E00 if dtype == FP16 else 0x7FC0
        ovf_o, t_o, _ = oracle.shard_step_halfacc(grads, dtype, st, hp_o, t_o, sc_o)
        dg = [[dev16(x) for x in micro] for micro in grads]
        for k in range(G - 1):
            zs.zs_grad_accum_halfacc(ctx, dg[k], dtype, count, acc, k == 0)
        ovf, ns = zs.zs_shard_step_halfacc(ctx, dg[G - 1], dtype, count, acc, G, master, m, v,
                                           half, hp, t + 1, sc)
        if not ovf:
            t += 1
        assert ovf == ovf_o and ns == sc_o.scale, f"step {s}"
    assert t == t_o
    close(master.cpu().numpy(), st.master, "master")
    close(m.cpu().numpy(), st.m, "m")
    close(v.cpu().numpy(), st.v, "v")
    assert ulps(half.cpu().numpy().view(np.uint16), st.half).max() <= 1


@pytest.mark.parametrize("dtype", [FP16, BF16])
@pytest.mark.parametrize("n,G,count", [(1, 8, 30_011), (4, 2, 20_000), (16, 1, 5_003)])
def test_halfacc_oop_steps_equal_the_in_place_step_and_the_oracle(zs, ctx, dtype, n, G, count):
    """zs_shard_step_halfacc_oop: the last micro-step's sums rounded to the
    accumulator's format, flagged and applied out of place in one pass.  The
    written set equals the in-place half-accumulator step's state bit for bit,
    step after step (an overflow, and a sum that rounds past the half maximum,
    included: the current set stays untouched), and the oracle's within the bound."""
    rng = np.random.default_rng(n * 5 + G + 50 * dtype)
    master0 = (rng.standard_normal(count) * 0.02).astype(np.float32)
    st = oracle.ShardState.from_master(master0, dtype)
    dyn = dtype == FP16
    sc_o = oracle.make_scaler(256.0 if dyn else 1.0, 1.0, 3, 1, dyn)
    sc_a = zs.zs_scaler_init(sc_o.scale, 1.0, 3, 1, dyn)
    sc_b = zs.zs_scaler_init(sc_o.scale, 1.0, 3, 1, dyn)
    hp_v = (STRESS_LR, 0.9, 0.999, 1e-8, 0.01)
    hp_o, hp = oracle.make_hparams(*hp_v), zs.make_hparams(*hp_v)

    def state(m0):
        p = torch.from_numpy(m0.copy()).cuda()
        return [p, torch.zeros_like(p), torch.zeros_like(p),
                torch.zeros(count, dtype=torch.int16, device="cuda")]
    ref = state(master0)
    sets = [state(master0), state(np.zeros_like(master0))]
    acc_a = torch.zeros(count, dtype=torch.int16, device="cuda")
    acc_b = torch.zeros_like(acc_a)
    cur = t = t_o = 0
    big = 40_000.0 if dtype == FP16 else 2.0e38    # two of them round past the half maximum
    for s in range(1, 9):
        grads = [[lib_half((rng.standard_normal(count) * 1e-2 * sc_o.scale).astype(np.float32),
                           dtype) for _ in range(n)] for _ in range(G)]
        if s == 4:
            grads[0][n - 1][count // 3] = 0x7E00 if dtype == FP16 else 0x7FC0
        if s == 6 and n * G > 1:
            grads[0][0][7] = grads[G - 1][n - 1][7] = lib_half(np.float32([big]), dtype)[0]
        ovf_o, t_o, _ = oracle.shard_step_halfacc(grads, dtype, st, hp_o, t_o, sc_o)
        dg = [[dev16(x) for x in micro] for micro in grads]
        for k in range(G - 1):
            zs.zs_grad_accum_halfacc(ctx, dg[k], dtype, count, acc_a, k == 0)
            zs.zs_grad_accum_halfacc(ctx, dg[k], dtype, count, acc_b, k == 0)
        ovf_a, ns_a = zs.zs_shard_step_halfacc(ctx, dg[G - 1], dtype, count, acc_a, G, *ref, hp,
                                               t + 1, sc_a)
        src, dst = sets[cur], sets[cur ^ 1]
        before = [x.clone() for x in src]
        ovf_b, ns_b = zs.zs_shard_step_halfacc_oop(ctx, dg[G - 1], dtype, count,
                                                   acc_b if G > 1 else None, G, *src[:3],
                                                   *dst, hp, t + 1, sc_b)
        assert ovf_a == ovf_b == ovf_o and ns_a == ns_b == sc_o.scale, f"step {s}"
        if ovf_b:
            assert all(torch.equal(x, y) for x, y in zip(before, src))
        else:
            cur ^= 1
            t += 1
        for k in range(3):
            assert torch.equal(sets[cur][k], ref[k]), (s, k)
        if t:
            assert torch.equal(sets[cur][3], ref[3])
    assert t == t_o
    close(sets[cur][0].cpu().numpy(), st.master, "master")
    close(sets[cur][1].cpu().numpy(), st.m, "m")
    close(sets[cur][2].cpu().numpy(), st.v, "v")


@pytest.mark.parametrize("form", ["async", "async_oop"])
@pytest.mark.parametrize("graph", [False, True])
@pytest.mark.parametrize("dtype", [FP16, BF16])
def test_halfacc_device_state_steps_equal_the_synchronising_step(zs, ctx, form, graph, dtype):
    """zs_shard_step_halfacc_async (in place) and _async_oop: the scale, Adam's
    step count and the outcome on the device, no host round trip, eager or
    replayed from a CUDA graph.  The same kernels and constants as the
    synchronising half-accumulator step: the state equals it bit for bit,
    step after step (an overflow included), and the oracle's within the bound."""
    n, G, count = 4, 2, 20_011
    rng = np.random.default_rng(77 + dtype + (10 if graph else 0) + (100 if form == "async_oop" else 0))
    master0 = (rng.standard_normal(count) * 0.02).astype(np.float32)
    st = oracle.ShardState.from_master(master0, dtype)
    dyn = dtype == FP16
    sc_o = oracle.make_scaler(256.0 if dyn else 1.0, 1.0, 3, 1, dyn)
    sc = zs.zs_scaler_init(sc_o.scale, 1.0, 3, 1, dyn)
    state = zs.DeviceState(zs.zs_scaler_init(sc_o.scale, 1.0, 3, 1, dyn))
    hp_v = (STRESS_LR, 0.9, 0.999, 1e-8, 0.01)
    hp_o, hp = oracle.make_hparams(*hp_v), zs.make_hparams(*hp_v)

    def state_bufs(m0):
        p = torch.from_numpy(m0.copy()).cuda()
        return [p, torch.zeros_like(p), torch.zeros_like(p),
                torch.zeros(count, dtype=torch.int16, device="cuda")]
    ref = state_bufs(master0)                       # the synchronising step
    sets = [state_bufs(master0), state_bufs(np.zeros_like(master0))]
    pairs = [zs.pointer_array([sets[0][k], sets[1][k]]) for k in range(4)]
    acc_r = torch.zeros(count, dtype=torch.int16, device="cuda")
    acc_d = torch.zeros_like(acc_r)
    pad = (count + 7) // 8 * 8
    gbuf = torch.zeros((G, n, pad), dtype=torch.int16, device="cuda")
    ptrs = [zs.pointer_array(gbuf[k, r, :count] for r in range(n)) for k in range(G)]

    def device_step():
        for k in range(G - 1):
            zs.zs_grad_accum_halfacc(ctx, ptrs[k], dtype, count, acc_d, k == 0)
        if form == "async":
            zs.zs_shard_step_halfacc_async(ctx, ptrs[G - 1], dtype, count, acc_d, G, *sets[0],
                                           hp, None, state)
        else:
            zs.zs_shard_step_halfacc_async_oop(ctx, ptrs[G - 1], dtype, count, acc_d, G,
                                               *pairs, hp, None, state)

    g = None
    t = t_o = 0
    for s in range(1, 9):
        grads = [[lib_half((rng.standard_normal(count) * 1e-2 * sc_o.scale).astype(np.float32),
                           dtype) for _ in range(n)] for _ in range(G)]
        if s == 4:
            grads[G - 1][n - 1][count // 3] = 0x7E00 if dyn else 0x7FC0
        host = np.stack([np.stack(mc) for mc in grads]).view(np.int16)
        gbuf[:, :, :count].copy_(torch.from_numpy(host))
        ovf_o, t_o, _ = oracle.shard_step_halfacc(grads, dtype, st, hp_o, t_o, sc_o)
        dg = [[dev16(x) for x in micro] for micro in grads]
        for k in range(G - 1):
            zs.zs_grad_accum_halfacc(ctx, dg[k], dtype, count, acc_r, k == 0)
        ovf, _ = zs.zs_shard_step_halfacc(ctx, dg[G - 1], dtype, count, acc_r, G, *ref, hp,
                                          t + 1, sc)
        if graph and g is None:
            device_step()                 # the first step uncaptured, then capture the rest
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                device_step()
        elif graph:
            g.replay()
        else:
            device_step()
        d = state.read()
        assert d.overflow == ovf == ovf_o and d.scaler.scale == sc.scale == sc_o.scale, s
        t += 0 if ovf else 1
        assert d.step == t == t_o and d.iterations == s
        cur = sets[d.buf] if form == "async_oop" else sets[0]
        for k in range(3):
            assert torch.equal(cur[k], ref[k]), (s, k)
        if t:
            assert torch.equal(cur[3], ref[3])
    close(ref[0].cpu().numpy(), st.master, "master")
    close(ref[1].cpu().numpy(), st.m, "m")
    close(ref[2].cpu().numpy(), st.v, "v")


@pytest.mark.parametrize("form", ["sync", "oop", "async", "async_oop"])
@pytest.mark.parametrize("dtype", [FP16, BF16])
@pytest.mark.parametrize("n,G,count", [(1, 1, 4099), (2, 3, 65_541), (16, 2, 20_011),
                                       (3, 1, 900_001)])
def test_halfacc_fused_step_equals_the_multi_kernel_path(zs, form, dtype, n, G, count):
    """The half-accumulator forms' last call as one fused kernel (4-element
    units, or 8 for the 900,001-element shard): the last micro-step's sums
    rounded to the accumulator's format before the flag and the update, as the
    half-accumulator passes round them.  Every step's state equals the
    multi-kernel path's bit for bit (a NaN step and a sum that rounds past the
    half maximum included), one fused launch a step."""
    on, off = zs.Ctx(), zs.Ctx()
    try:
        off.set_fused(zs.ZS_FUSED_OFF)
        on.set_timing(True)
        rng = np.random.default_rng(900 + 10 * n + G + dtype + 100 * len(form))
        master0 = (rng.standard_normal(count) * 0.02).astype(np.float32)
        dyn = dtype == FP16
        hp = zs.make_hparams(STRESS_LR, 0.9, 0.999, 1e-8, 0.01)
        big = 40_000.0 if dtype == FP16 else 2.0e38

        def bufs(m0):
            p = torch.from_numpy(m0.copy()).cuda()
            return [p, torch.zeros_like(p), torch.zeros_like(p),
                    torch.zeros(count, dtype=torch.int16, device="cuda")]
        run = {}
        for name, ctx in (("on", on), ("off", off)):
            sets = [bufs(master0), bufs(np.zeros_like(master0))]
            run[name] = {"ctx": ctx, "sets": sets, "cur": 0, "t": 0,
                         "acc": torch.zeros(count, dtype=torch.int16, device="cuda"),
                         "sc": zs.zs_scaler_init(256.0 if dyn else 1.0, 1.0, 3, 1, dyn),
                         "state": zs.DeviceState(zs.zs_scaler_init(256.0 if dyn else 1.0, 1.0,
                                                                   3, 1, dyn)),
                         "pairs": [zs.pointer_array([sets[0][k], sets[1][k]])
                                   for k in range(4)]}
        f0 = on.timing(zs.ZS_KERNEL_FUSED)[1]
        for s in range(1, 7):
            grads = [[lib_half((rng.standard_normal(count) * 1e-2 * 256.0).astype(np.float32),
                               dtype) for _ in range(n)] for _ in range(G)]
            if s == 3:
                grads[G - 1][n - 1][count // 3] = 0x7E00 if dyn else 0x7FC0
            if s == 5 and n * G > 1:
                grads[0][0][7] = grads[G - 1][n - 1][7] = lib_half(np.float32([big]), dtype)[0]
            dg = [[dev16(x) for x in micro] for micro in grads]
            out = {}
            for name, r in run.items():
                ctx, acc, sets = r["ctx"], r["acc"], r["sets"]
                for k in range(G - 1):
                    zs.zs_grad_accum_halfacc(ctx, dg[k], dtype, count, acc, k == 0)
                cur = sets[r["cur"]]
                if form == "sync":
                    out[name] = zs.zs_shard_step_halfacc(ctx, dg[G - 1], dtype, count, acc, G,
                                                         *cur, hp, r["t"] + 1, r["sc"])
                elif form == "oop":
                    dst = sets[r["cur"] ^ 1]
                    out[name] = zs.zs_shard_step_halfacc_oop(
                        ctx, dg[G - 1], dtype, count, acc if G > 1 else None, G, *cur[:3],
                        *dst, hp, r["t"] + 1, r["sc"])
                    if not out[name][0]:
                        r["cur"] ^= 1
                elif form == "async":
                    zs.zs_shard_step_halfacc_async(ctx, dg[G - 1], dtype, count, acc, G, *cur,
                                                   hp, None, r["state"])
                else:
                    zs.zs_shard_step_halfacc_async_oop(ctx, dg[G - 1], dtype, count,
                                                       acc if G > 1 else None, G, *r["pairs"],
                                                       hp, None, r["state"])
                if form in ("async", "async_oop"):
                    d = r["state"].read()
                    out[name] = (d.overflow, d.scaler.scale, d.step)
                    if form == "async_oop":
                        r["cur"] = d.buf & 1
                if not out[name][0]:
                    r["t"] += 1
            assert out["on"] == out["off"], f"step {s}"
            a, b = run["on"], run["off"]
            for k in range(4):
                assert torch.equal(a["sets"][a["cur"]][k], b["sets"][b["cur"]][k]), (s, k)
        assert on.timing(zs.ZS_KERNEL_FUSED)[1] - f0 == 6      # one launch a step
        assert run["on"]["t"] == run["off"]["t"] == (4 if n * G > 1 else 5)
    finally:
        on.close()
        off.close()
