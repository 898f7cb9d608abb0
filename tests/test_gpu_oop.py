"""The out-of-place step (zs_shard_step_oop, zs_shard_step_async_oop): the
last micro-step's sums, the overflow check and the AdamW update in one pass
that writes a second set of state buffers, committed only on a clean step.

It adds the same fp32 sums in the same order and runs the same update
arithmetic as zs_shard_step, so its state must equal the in-place step's bit
for bit, step after step, including the skipped steps (where the current set
must stay untouched); and it is held to the oracle like every other form.
Random stress inputs at lr 3e-4, at most 10 steps, re-read (n < 4) and
materialising (n >= 4) counterparts, fp16 and bf16, ragged tails."""
import numpy as np
import pytest
import torch

import oracle
from _helpers import STRESS_LR, assert_close, dev16, half_ulps, host16, lib_half

pytestmark = pytest.mark.gpu

FP16, BF16 = 0, 1


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


def rand_grads(rng, n, count, dtype, scale):
    return [lib_half((rng.standard_normal(count) * 1e-3 * scale *
                      np.exp2(rng.integers(-4, 4, count))).astype(np.float32), dtype)
            for _ in range(n)]


def state_set(master0, count):
    master = torch.from_numpy(master0.copy()).cuda()
    return {"p": master, "m": torch.zeros_like(master), "v": torch.zeros_like(master),
            "h": torch.zeros(count, dtype=torch.int16, device="cuda")}


@pytest.mark.parametrize("dtype", [FP16, BF16])
@pytest.mark.parametrize("n,G,count", [(1, 1, 4099), (2, 3, 10007), (4, 1, 8200),
                                       (16, 2, 20011), (64, 1, 777)])
def test_oop_steps_equal_the_in_place_step_and_the_oracle(zs, ctx, dtype, n, G, count):
    rng = np.random.default_rng(n * 31 + G + 7 * dtype)
    master0 = (rng.standard_normal(count) * 0.02).astype(np.float32)
    hp_vals = (STRESS_LR, 0.9, 0.999, 1e-8, 0.01)
    hp, hp_o = zs.make_hparams(*hp_vals), oracle.make_hparams(*hp_vals)
    dyn = dtype == FP16
    sc_o = oracle.make_scaler(1024.0 if dyn else 1.0, 1.0, 3, 1, dyn)
    sc_a = zs.zs_scaler_init(sc_o.scale, 1.0, 3, 1, dyn)     # in place
    sc_b = zs.zs_scaler_init(sc_o.scale, 1.0, 3, 1, dyn)     # out of place
    st = oracle.ShardState.from_master(master0, dtype)
    ref = state_set(master0, count)
    bufs = [state_set(master0, count), state_set(np.zeros_like(master0), count)]
    cur = 0
    acc_a = torch.zeros(count, dtype=torch.float32, device="cuda")
    acc_b = torch.zeros(count, dtype=torch.float32, device="cuda")
    t = t_o = 0
    inf = 0x7C00 if dtype == FP16 else 0x7F80
    for s in range(1, 11):
        grads = [rand_grads(rng, n, count, dtype, sc_o.scale) for _ in range(G)]
        if s in (3, 7):
            k = G - 1 if s == 3 else 0            # the last micro-step, then an earlier one
            grads[k][n - 1][count // 3] = inf
        ovf_o, t_o, _ = oracle.shard_step(grads, dtype, st, hp_o, t_o, sc_o)
        dg = [[dev16(x) for x in micro] for micro in grads]
        for k in range(G - 1):
            zs.zs_grad_accum(ctx, dg[k], dtype, count, acc_a, k == 0)
        ovf_a, _ = zs.zs_shard_step(ctx, dg[G - 1], dtype, count, acc_a, G, ref["p"], ref["m"],
                                    ref["v"], ref["h"], hp, t + 1, sc_a)
        for k in range(G - 1):
            zs.zs_grad_accum(ctx, dg[k], dtype, count, acc_b, k == 0)
        src, dst = bufs[cur], bufs[cur ^ 1]
        before = [x.clone() for x in (src["p"], src["m"], src["v"])]
        ovf_b, scale_b = zs.zs_shard_step_oop(ctx, dg[G - 1], dtype, count,
                                              acc_b if G > 1 else None, G, src["p"], src["m"],
                                              src["v"], dst["p"], dst["m"], dst["v"], dst["h"],
                                              hp, t + 1, sc_b)
        assert ovf_a == ovf_b == ovf_o, f"step {s}"
        assert scale_b == sc_a.scale == sc_o.scale
        assert (sc_b.clean_count, sc_b.hyst_left) == (sc_o.clean_count, sc_o.hyst_left)
        if ovf_b:
            for x, y in zip(before, (src["p"], src["m"], src["v"])):
                assert torch.equal(x, y)          # the current set is untouched
        else:
            cur ^= 1
            t += 1
        now = bufs[cur]
        for k in ("p", "m", "v"):
            assert torch.equal(now[k], ref[k]), (s, k)
        if t:
            assert torch.equal(now["h"], ref["h"])
    assert t == t_o
    now = bufs[cur]
    assert_close(now["p"].cpu().numpy(), st.master, "master")
    assert_close(now["m"].cpu().numpy(), st.m, "m")
    assert_close(now["v"].cpu().numpy(), st.v, "v")
    assert half_ulps(host16(now["h"]), st.half).max() <= 1


@pytest.mark.parametrize("dtype", [FP16, BF16])
@pytest.mark.parametrize("graph", [False, True])
@pytest.mark.parametrize("n,G,count", [(1, 3, 20_011), (8, 2, 40_003), (64, 1, 4_103)])
def test_async_oop_steps_match_oracle(zs, ctx, n, G, count, graph, dtype):
    """The device-resident form: the buffer index in the device state flips on
    every applied step; against the oracle with a WarmupDecayLR schedule, an
    overflow and a CUDA-graph replay (fp16 with a dynamic scale, bf16 with a
    static one)."""
    rng = np.random.default_rng(n + 10 * G + (100 if graph else 0) + 1000 * dtype)
    master0 = (rng.standard_normal(count) * 0.02).astype(np.float32)
    st = oracle.ShardState.from_master(master0, dtype)
    dyn = dtype == FP16
    sc_o = oracle.make_scaler(512.0 if dyn else 1.0, 1.0, 2, 1, dyn)
    kind, mn, mx, wu, tot = (oracle.LR_WARMUP_DECAY, float(np.float32(1e-5)),
                             float(np.float32(STRESS_LR)), 3, 9)
    sched = zs.make_schedule(kind, mn, mx, wu, tot)
    hp = zs.make_hparams(mx, 0.9, 0.999, 1e-8, 0.01)
    state = zs.DeviceState(zs.zs_scaler_init(sc_o.scale, 1.0, 2, 1, dyn))
    sets = [state_set(master0, count), state_set(np.zeros_like(master0), count)]
    acc = torch.zeros(count, dtype=torch.float32, device="cuda")
    pad = (count + 7) // 8 * 8
    gbuf = torch.zeros((G, n, pad), dtype=torch.int16, device="cuda")
    ptrs = [zs.pointer_array(gbuf[k, r, :count] for r in range(n)) for k in range(G)]
    pairs = {k: zs.pointer_array([sets[0][k], sets[1][k]]) for k in ("p", "m", "v", "h")}

    def step_calls():
        for k in range(G - 1):
            zs.zs_grad_accum(ctx, ptrs[k], dtype, count, acc, k == 0)
        zs.zs_shard_step_async_oop(ctx, ptrs[G - 1], dtype, count, acc, G, pairs["p"],
                                   pairs["m"], pairs["v"], pairs["h"], hp, sched, state)

    g = None
    t_o = 0
    for s in range(1, 11):
        grads = [[lib_half((rng.standard_normal(count) * 1e-2 * sc_o.scale).astype(np.float32),
                           dtype) for _ in range(n)] for _ in range(G)]
        if s == 5:
            grads[G - 1][n - 1][count - 1] = 0x7C00 if dyn else 0x7F80
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
        assert d.step == t_o and d.iterations == s and d.buf == t_o % 2
    cur = sets[state.read().buf]
    assert_close(cur["p"].cpu().numpy(), st.master, "master")
    assert_close(cur["m"].cpu().numpy(), st.m, "m")
    assert_close(cur["v"].cpu().numpy(), st.v, "v")
    assert half_ulps(host16(cur["h"]), st.half).max() <= 1


def test_oop_rejects_overlapping_buffers(zs, ctx):
    count = 64
    a = torch.zeros(4 * count, dtype=torch.float32, device="cuda")
    h = torch.zeros(count, dtype=torch.int16, device="cuda")
    g = [torch.zeros(count, dtype=torch.int16, device="cuda")]
    sc = zs.zs_scaler_init(1.0, 1.0, 10, 1, False)
    hp = zs.make_hparams(1e-4)
    p_in, m_in, v_in, p_out = a[:count], a[count:2 * count], a[2 * count:3 * count], a[3 * count:]
    # m_out aliasing m_in: refused before any work
    with pytest.raises(zs.ZsError) as e:
        zs.zs_shard_step_oop(ctx, g, FP16, count, None, 1, p_in, m_in, v_in, p_out, m_in,
                             a[count + 8:2 * count + 8], h, hp, 1, sc)
    assert e.value.status == zs.ZS_ERR_ARG


@pytest.mark.parametrize("dtype", [FP16, BF16])
@pytest.mark.parametrize("n,G,count", [(3, 2, 10_007), (2, 1, 8_192), (16, 2, 3_001)])
def test_two_phase_update_oop_equals_the_one_call_form(zs, ctx, n, G, count, dtype):
    """zs_update_oop over two ranges with one flag, then zs_scaler_update on
    that flag: the written set equals zs_shard_step_oop's bit for bit, and
    the flag and scale agree, skipped steps included."""
    rng = np.random.default_rng(n * 7 + G + 100 * dtype)
    master0 = (rng.standard_normal(count) * 0.02).astype(np.float32)
    hp_vals = (STRESS_LR, 0.9, 0.999, 1e-8, 0.01)
    hp = zs.make_hparams(*hp_vals)
    dyn = dtype == FP16
    sc_a = zs.zs_scaler_init(1024.0 if dyn else 1.0, 1.0, 2, 1, dyn)   # one call
    sc_b = zs.zs_scaler_init(1024.0 if dyn else 1.0, 1.0, 2, 1, dyn)   # two phases
    a_sets = [state_set(master0, count), state_set(np.zeros_like(master0), count)]
    b_sets = [state_set(master0, count), state_set(np.zeros_like(master0), count)]
    acc_a = torch.zeros(count, dtype=torch.float32, device="cuda")
    acc_b = torch.zeros_like(acc_a)
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    cut = count // 2 // 64 * 64     # a 64-element boundary: both ranges stay 16-byte aligned
    cur = t = 0
    for s in range(1, 7):
        grads = [rand_grads(rng, n, count, dtype, sc_a.scale) for _ in range(G)]
        if s == 3:
            grads[G - 1][0][count - 5] = 0x7C00 if dyn else 0x7F80   # in the second range
        dg = [[dev16(x) for x in micro] for micro in grads]
        for k in range(G - 1):
            zs.zs_grad_accum(ctx, dg[k], dtype, count, acc_a, k == 0)
        src, dst = a_sets[cur], a_sets[cur ^ 1]
        ovf_a, _ = zs.zs_shard_step_oop(ctx, dg[G - 1], dtype, count, acc_a if G > 1 else None,
                                        G, src["p"], src["m"], src["v"], dst["p"], dst["m"],
                                        dst["v"], dst["h"], hp, t + 1, sc_a)
        flag.zero_()
        for k in range(G - 1):
            zs.zs_reduce_check(ctx, dg[k], dtype, count, acc_b, k == 0, flag)
        src, dst = b_sets[cur], b_sets[cur ^ 1]
        div = float(n * G * sc_b.scale)
        for lo, hi in ((0, cut), (cut, count)):
            r = slice(lo, hi)
            zs.zs_update_oop(ctx, [g[r] for g in dg[G - 1]], dtype, hi - lo,
                             acc_b[r] if G > 1 else None, div, src["p"][r], src["m"][r],
                             src["v"][r], dst["p"][r], dst["m"][r], dst["v"][r], dst["h"][r], hp,
                             t + 1, flag)
        ovf_b = zs.zs_scaler_update(ctx, flag, sc_b)
        assert ovf_a == ovf_b == (1 if s == 3 else 0) and sc_a.scale == sc_b.scale, s
        if not ovf_a:
            cur ^= 1
            t += 1
            for k in ("p", "m", "v", "h"):
                assert torch.equal(a_sets[cur][k], b_sets[cur][k]), (s, k)


def test_update_oop_rejects_bad_arguments(zs, ctx):
    """Rejected before any work: no flag, a non-positive grad_div, the in and
    out sets overlapping, a range start off the 16-byte grid."""
    count = 256
    a = torch.zeros(8 * count, dtype=torch.float32, device="cuda")
    h = torch.zeros(2 * count, dtype=torch.int16, device="cuda")
    g = [torch.zeros(2 * count, dtype=torch.int16, device="cuda")]
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    hp = zs.make_hparams(1e-4)
    sets = [a[k * count:(k + 1) * count] for k in range(6)]

    def call(grads=g, div=2.0, d_flag=flag, s=sets, half=h[:count], n=count):
        zs.zs_update_oop(ctx, grads, FP16, n, None, div, *s, half, hp, 1, d_flag)

    call()                                            # well-formed: accepted
    for kw, status in (({"d_flag": None}, zs.ZS_ERR_ARG), ({"div": 0.0}, zs.ZS_ERR_ARG),
                       ({"div": float("inf")}, zs.ZS_ERR_ARG),
                       ({"s": sets[:3] + [sets[0]] + sets[4:]}, zs.ZS_ERR_ARG),
                       ({"grads": [g[0][1:count + 1]]}, zs.ZS_ERR_ALIGN),
                       ({"s": [a[1:count + 1]] + sets[1:]}, zs.ZS_ERR_ALIGN)):
        with pytest.raises(zs.ZsError) as e:
            call(**kw)
        assert e.value.status == status, kw
    assert flag.item() == 0
