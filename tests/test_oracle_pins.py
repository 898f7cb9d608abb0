"""Pins of the CPU oracle to facts fixed outside it: the pages' printed memory
formulas and figures, closed forms of bias-corrected Adam, exact sums, library
half conversions, a hand-worked loss-scale trace, invariants (shard union,
bucket independence, skip-and-halve), and multi-step runs against a library
AdamW (torch.optim.AdamW, clip_grad_norm_) in fp64.  No GPU."""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from _helpers import lib_half as _lib_half

FP16, BF16 = oracle.FP16, oracle.BF16


# ---------------------------------------------------------------- partition

@pytest.mark.parametrize("psi,n,align", [(1, 1, 64), (1000, 3, 64), (4096, 8, 64), (12345, 7, 8),
                                         (1 << 20, 2, 64), (124_439_808, 8, 64), (0, 4, 64),
                                         (65, 64, 1)])
def test_partition_enumeration(psi, n, align):
    psi_pad, E = oracle.partition(psi, n, align)
    assert psi_pad % (n * align) == 0 and psi_pad >= psi and psi_pad - psi < n * align
    assert E * n == psi_pad
    covered = 0
    for r in range(n):
        b, ve, pe = oracle.shard_range(psi, E, n, r)
        assert b == covered and pe - b == E
        assert b <= ve <= pe and ve == max(b, min(pe, psi))
        covered = pe
    assert covered == psi_pad
    if psi_pad <= 20000:  # brute force: every index owned exactly once
        owner = np.full(psi_pad, -1)
        for r in range(n):
            b, ve, pe = oracle.shard_range(psi, E, n, r)
            assert (owner[b:pe] == -1).all()
            owner[b:pe] = r
        assert (owner >= 0).all()


def test_partition_workload_shapes():
    # Shard lengths of the synthetic workloads (Ψ padded to a multiple of 64·N).
    assert oracle.partition(1 << 20, 2) == (1 << 20, 1 << 19)
    assert oracle.partition(124_439_808, 8) == (124_440_064, 15_555_008)
    assert oracle.partition(1_315_723_264, 16) == (1_315_723_264, 82_232_704)
    assert oracle.partition(6_738_415_616, 64) == (6_738_415_616, 105_287_744)
    assert oracle.partition(6_738_415_616, 1) == (6_738_415_616, 6_738_415_616)


def test_memory_formulas_of_the_pages(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "memory_pages.json")))
    for psi in (64 * 64 * 1000, 6_738_415_616):
        for n in (1, 2, 8, 16, 64):
            psi_pad, E = oracle.partition(psi, n)
            assert psi_pad == psi
            # §2 table, §2.1, §2.2, §2.3 as printed (Ψ divisible by N here)
            assert oracle.state_bytes(psi, E, 0) == 16 * psi
            assert oracle.state_bytes(psi, E, 1) == 4 * psi + 12 * psi // n
            assert oracle.state_bytes(psi, E, 2) == 2 * psi + (2 * psi + 12 * psi) // n
            assert oracle.state_bytes(psi, E, 3) == (2 * psi + 2 * psi + 12 * psi) // n
    for ex in g["model_state_examples"]:
        psi = int(ex["psi"])
        b = oracle.state_bytes(psi, psi, 0)
        assert abs(b - ex["approx_bytes"]) <= ex["printed_digits_rel"] * ex["approx_bytes"]
    psi = 64 * 1_000_000
    _, E = oracle.partition(psi, 64)
    for row in g["n64_per_param"]:
        per = oracle.state_bytes(psi, E, row["stage"]) / psi
        assert abs(per - row["approx"]) <= row["abs_tol"]
        assert abs(16 / per - row["approx_saving"]) <= row["saving_tol"]
    # padding counts against every rank but never against plain DP
    psi_pad, E = oracle.partition(1000, 3)
    assert oracle.state_bytes(1000, E, 3) == 16 * E and 16 * E * 3 >= 16 * 1000


# ---------------------------------------------------------------- half formats

def test_fp16_decode_all_patterns_vs_numpy():
    bits = np.arange(1 << 16, dtype=np.uint16)
    ours = oracle.half_to_double(bits, FP16)
    ref = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert (np.isnan(ours) == nan).all()
    assert (ours[~nan] == ref[~nan]).all()
    assert (np.signbit(ours[~nan]) == np.signbit(ref[~nan])).all()


def test_bf16_decode_all_patterns_vs_torch():
    bits = np.arange(1 << 16, dtype=np.uint16)
    ours = oracle.half_to_double(bits, BF16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).double().numpy()
    nan = np.isnan(ref)
    assert (np.isnan(ours) == nan).all()
    assert (ours[~nan] == ref[~nan]).all()
    assert (np.signbit(ours[~nan]) == np.signbit(ref[~nan])).all()


@pytest.mark.parametrize("dtype", [FP16, BF16])
def test_half_round_trip_all_patterns(dtype):
    bits = np.arange(1 << 16, dtype=np.uint16)
    vals = oracle.half_to_double(bits, dtype)
    ok = ~np.isnan(vals)
    back = oracle.f32_to_half(vals[ok].astype(np.float32), dtype)
    assert (back == bits[ok]).all()


@pytest.mark.parametrize("dtype", [FP16, BF16])
def test_half_encode_random_vs_library(dtype):
    rng = np.random.default_rng(1)
    raw = rng.integers(0, 1 << 32, size=1 << 20, dtype=np.uint64).astype(np.uint32)
    x = raw.view(np.float32)
    x = x[~np.isnan(x)]
    assert (oracle.f32_to_half(x, dtype) == _lib_half(x, dtype)).all()
    # magnitudes around the fp16 range, including subnormals and overflow
    y = (rng.standard_normal(1 << 18) * np.exp2(rng.integers(-30, 18, 1 << 18))).astype(np.float32)
    assert (oracle.f32_to_half(y, dtype) == _lib_half(y, dtype)).all()


@pytest.mark.parametrize("dtype", [FP16, BF16])
def test_half_encode_ties(dtype):
    # midpoints between every pair of adjacent finite halves are fp32-exact ties
    bits = np.arange(0, (0x7C00 if dtype == FP16 else 0x7F80) - 1, dtype=np.uint16)
    lo = oracle.half_to_double(bits, dtype)
    hi = oracle.half_to_double(bits + 1, dtype)
    mid = ((lo + hi) / 2).astype(np.float32)
    assert ((mid.astype(np.float64) == (lo + hi) / 2)).all()
    ours = oracle.f32_to_half(mid, dtype)
    even = np.where(bits % 2 == 0, bits, bits + 1).astype(np.uint16)
    assert (ours == even).all()
    assert (ours == _lib_half(mid, dtype)).all()
    assert (oracle.f32_to_half(-mid, dtype) == (even | 0x8000)).all()


def test_fp16_overflow_threshold():
    # 65504 is the largest finite fp16; the tie 65520 rounds to even = infinity
    assert oracle.f32_to_half(np.float32([65519.996, 65520.0, 1e9]), FP16).tolist() == \
        [0x7BFF, 0x7C00, 0x7C00]


# ---------------------------------------------------------------- reduction

def _h(vals, dtype=FP16):
    return _lib_half(np.array(vals, dtype=np.float32), dtype)


def test_reduce_exact_rationals():
    # integer multiples of 2^-10 with |sum| < 2^13: every fp32 partial sum is exact
    rng = np.random.default_rng(2)
    n, count = 9, 257
    ints = rng.integers(-2000, 2000, size=(3, n, count))
    acc = np.zeros(count, dtype=np.float32)
    for k in range(3):
        slices = [_h(ints[k, r] / 1024.0) for r in range(n)]
        oracle.reduce_accumulate(slices, FP16, acc, first=(k == 0))
    exact = [sum(Fraction(int(ints[k, r, i]), 1024) for k in range(3) for r in range(n))
             for i in range(count)]
    assert all(Fraction(float(a)) == e for a, e in zip(acc, exact))


def test_reduce_order_is_rank_order_from_plus_zero():
    # fp32 spacing at 65504 is 2^-8; 2^-10 alone is absorbed, 4·2^-10 is not.
    big, tiny = 65504.0, 2.0 ** -10
    first_big = [big, tiny, tiny, tiny, tiny, -big]
    first_tiny = [tiny, tiny, tiny, tiny, big, -big]
    for order, expect in ((first_big, 0.0), (first_tiny, 2.0 ** -8)):
        acc = np.zeros(1, dtype=np.float32)
        oracle.reduce_accumulate([_h([x]) for x in order], FP16, acc, first=True)
        assert acc[0] == expect
    # micro-step order: the carried accumulator comes before micro-step 2's ranks
    acc = np.zeros(1, dtype=np.float32)
    oracle.reduce_accumulate([_h([big])], FP16, acc, first=True)
    oracle.reduce_accumulate([_h([tiny]), _h([tiny]), _h([-big])], FP16, acc, first=False)
    assert acc[0] == 0.0
    # start from +0.0: all slices -0.0 give +0.0
    acc = np.full(1, 7.0, dtype=np.float32)
    oracle.reduce_accumulate([_h([-0.0]), _h([-0.0])], FP16, acc, first=True)
    assert acc[0] == 0.0 and not np.signbit(acc[0])
    # not first: the old accumulator is kept
    acc = np.full(1, 7.0, dtype=np.float32)
    oracle.reduce_accumulate([_h([1.0])], FP16, acc, first=False)
    assert acc[0] == 8.0


def test_reduce_bf16_and_nonfinite():
    acc = np.zeros(3, dtype=np.float32)
    oracle.reduce_accumulate([_h([1.0, 3.0e38, 2.0], BF16), _h([0.5, 3.0e38, -2.0], BF16)], BF16,
                             acc, first=True)
    assert acc[0] == 1.5 and np.isinf(acc[1]) and acc[2] == 0.0
    inf = np.array([0x7C00], dtype=np.uint16)
    ninf = np.array([0xFC00], dtype=np.uint16)
    nan = np.array([0x7E00], dtype=np.uint16)
    one = _h([1.0])
    assert oracle.any_nonfinite([one, one], FP16, 1) == 0
    assert oracle.any_nonfinite([one, inf], FP16, 1) == 1
    assert oracle.any_nonfinite([ninf, one], FP16, 1) == 1
    assert oracle.any_nonfinite([nan], FP16, 1) == 1
    assert oracle.any_nonfinite([np.array([0x7F80], np.uint16)], BF16, 1) == 1
    assert oracle.any_nonfinite([np.array([0x7BFF], np.uint16)], FP16, 1) == 0  # 65504


# ---------------------------------------------------------------- Adam / AdamW

def _f32(x):
    return float(np.float32(x))


def _apply(acc, grad_div, master, m, v, hp, t, dtype=FP16):
    st = oracle.ShardState(np.array(master, np.float32), np.array(m, np.float32),
                           np.array(v, np.float32), np.zeros(len(master), np.uint16))
    oracle.adamw_apply(np.array(acc, np.float32), grad_div, st.master, st.m, st.v, st.half,
                       dtype, hp, t)
    return st


def _ulp32(x):
    x = np.abs(np.float32(x))
    return float(np.spacing(x)) if x > 0 else float(np.spacing(np.float32(0)))


def test_adam_first_step_closed_form():
    # t=1 from m=v=0 without decay: Δp = -lr·ĝ/(|ĝ|+eps) (bias-corrected Adam)
    hp = oracle.make_hparams(1e-4, 0.9, 0.999, 1e-8, 0.0)
    lr, eps = hp.lr, hp.eps
    ghat = np.array([1e-3, -1e-3, 3e-8, -1e-8, 2e-9, 1.0, -5e-5, 0.0], dtype=np.float64)
    S, N, G = 65536.0, 2, 1
    acc = (ghat * N * G * S).astype(np.float32)
    ghat = acc.astype(np.float64) / (N * G * S)
    p0 = np.array([0.02, -0.01, 0.5, 1e-3, -2.0, 0.0, 0.03, 0.1], np.float32)
    st = _apply(acc, N * G * S, p0, np.zeros(8), np.zeros(8), hp, 1)
    want = p0.astype(np.float64) - lr * ghat / (np.abs(ghat) + eps)
    for got, w in zip(st.master, want):
        assert abs(float(got) - w) <= 0.5 * _ulp32(w) + 1e-15
    # half copy is the rounded master
    assert (st.half == _lib_half(st.master, FP16)).all()


def test_adam_constant_gradient_every_step():
    # ĝ constant: m_t = (1-β1^t)ĝ and v_t = (1-β2^t)ĝ², so every step moves by lr·ĝ/(|ĝ|+eps)
    hp = oracle.make_hparams(1e-3, 0.9, 0.999, 1e-8, 0.0)
    ghat = np.array([2e-3, -7e-4, 1e-8], np.float64)
    p = np.array([0.1, -0.2, 0.3], np.float32)
    m = np.zeros(3, np.float32)
    v = np.zeros(3, np.float32)
    ref = p.astype(np.float64)
    for t in range(1, 21):
        st = _apply(ghat.astype(np.float32), 1.0, p, m, v, hp, t)
        p, m, v = st.master, st.m, st.v
        ref = ref - hp.lr * ghat / (np.abs(ghat) + hp.eps)
        assert np.all(np.abs(p.astype(np.float64) - ref) <= 4e-7 * np.abs(ref) + 1e-6 * hp.lr * t)


def test_adam_second_step_closed_form():
    # two gradients ĝ1, ĝ2 from m=v=0: m̂2 = (β1ĝ1+ĝ2)/(1+β1), v̂2 = (β2ĝ1²+ĝ2²)/(1+β2)
    hp = oracle.make_hparams(1e-3, 0.9, 0.999, 1e-8, 0.0)
    b1, b2 = hp.beta1, hp.beta2
    g1 = np.array([1e-3, 1e-3, -2e-4, 5e-3], np.float64)
    g2 = np.array([-1e-3, 2e-3, 3e-4, 5e-3], np.float64)
    g1 = g1.astype(np.float32).astype(np.float64)
    g2 = g2.astype(np.float32).astype(np.float64)
    p0 = np.array([0.01, 0.02, -0.03, 0.04], np.float32)
    st = _apply(g1.astype(np.float32), 1.0, p0, np.zeros(4), np.zeros(4), hp, 1)
    p1 = st.master.astype(np.float64)
    st = _apply(g2.astype(np.float32), 1.0, st.master, st.m, st.v, hp, 2)
    mh = (b1 * g1 + g2) / (1 + b1)
    vh = (b2 * g1 ** 2 + g2 ** 2) / (1 + b2)
    want = p1 - hp.lr * mh / (np.sqrt(vh) + hp.eps)
    assert np.all(np.abs(st.master.astype(np.float64) - want) <= 1e-6 * hp.lr + 0.5 * np.spacing(
        np.abs(want).astype(np.float32)))
    # β1 and β2 each matter: a swapped pair would move the alternating element differently
    alt = (b2 * g1[0] + g2[0]) / (1 + b2)
    assert abs(alt - mh[0]) > 1e-5


def test_adamw_decoupled_decay_at_zero_gradient():
    hp = oracle.make_hparams(1e-2, 0.9, 0.999, 1e-8, 0.1)
    p0 = np.array([1.0, -0.5, 0.25, 0.0], np.float32)
    st = _apply(np.zeros(4), 1.0, p0, np.zeros(4), np.zeros(4), hp, 1)
    want = p0.astype(np.float64) * (1 - hp.lr * hp.weight_decay)
    assert np.all(np.abs(st.master - want) <= 0.5 * np.spacing(np.abs(want).astype(np.float32)))
    assert (st.m == 0).all() and (st.v == 0).all()


def test_unscale_divides_by_ranks_micro_steps_and_scale():
    # same ĝ whether it arrives as acc/(N·G·S) for different N, G, S
    hp = oracle.make_hparams(1e-4, 0.9, 0.999, 1e-8, 0.0)
    ghat = 3e-4
    outs = []
    for N, G, S in ((1, 1, 1.0), (8, 4, 65536.0), (64, 1, 2.0 ** 15), (16, 2, 1.0)):
        acc = np.float32(ghat * N * G * S)
        st = _apply([acc], N * G * S, [0.5], [0.0], [0.0], hp, 1)
        outs.append(st.master[0])
    assert len(set(outs)) == 1


# ---------------------------------------------------------------- loss scale

def test_scaler_traces(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "scaler_traces.json")))
    for tr in g["traces"]:
        sc = oracle.make_scaler(tr["scale0"], tr["min_scale"], tr["window"], tr["hysteresis"],
                                tr["dynamic"], tr.get("consecutive_hysteresis", False))
        applied = 0
        got = []
        for s in range(1, tr["steps"] + 1):
            ovf = 1 if s in tr["overflow_steps"] else 0
            applied += 1 - ovf
            oracle.scaler_update(sc, ovf)
            got.append(sc.scale)
        assert got == tr["scale_after"], tr["name"]
        assert applied == tr["applied_updates"]


def test_initial_scale_power_16():
    # initial_scale_power 16 -> 65536 (§4.2)
    assert oracle.make_scaler(2.0 ** 16).scale == 65536.0


# ---------------------------------------------------------------- whole steps

def _rand_slices(rng, n, count, scale, dtype=FP16, sigma=1e-3):
    return [_lib_half((rng.standard_normal(count) * sigma * scale).astype(np.float32), dtype)
            for _ in range(n)]


@pytest.mark.parametrize("dtype", [FP16, BF16])
def test_skip_and_halve_on_injected_nonfinite(dtype):
    rng = np.random.default_rng(3)
    n, g, count = 3, 3, 1000
    hp = oracle.make_hparams(1e-4, 0.9, 0.999, 1e-8, 0.01)
    st = oracle.ShardState.from_master(rng.standard_normal(count) * 0.02, dtype)
    sc = oracle.make_scaler(1024.0)
    grads = [_rand_slices(rng, n, count, sc.scale, dtype) for _ in range(g)]
    ovf, t, _ = oracle.shard_step(grads, dtype, st, hp, 0, sc)
    assert ovf == 0 and t == 1 and sc.scale == 1024.0 and sc.clean_count == 1
    before = st.copy()
    for kind in (0x7C00 if dtype == FP16 else 0x7F80, 0xFC00 if dtype == FP16 else 0xFF80,
                 0x7E00 if dtype == FP16 else 0x7FC0):
        grads = [_rand_slices(rng, n, count, sc.scale, dtype) for _ in range(g)]
        grads[1][2][777] = kind  # micro-step 2, rank 2
        scale_before = sc.scale
        ovf, t2, _ = oracle.shard_step(grads, dtype, st, hp, t, sc)
        assert ovf == 1 and t2 == t and sc.scale == scale_before / 2 and sc.clean_count == 0
        for a, b in ((st.master, before.master), (st.m, before.m), (st.v, before.v),
                     (st.half, before.half)):
            assert a.tobytes() == b.tobytes()


def test_shard_union_equals_unpartitioned_step():
    rng = np.random.default_rng(4)
    psi, n, g = 3000, 4, 2
    psi_pad, E = oracle.partition(psi, n, 64)
    hp = oracle.make_hparams(1e-3, 0.9, 0.999, 1e-8, 0.01)
    master0 = np.zeros(psi_pad, np.float32)
    master0[:psi] = rng.standard_normal(psi) * 0.02
    full = oracle.ShardState.from_master(master0, FP16)
    shards = [oracle.ShardState.from_master(master0[q * E:(q + 1) * E], FP16) for q in range(n)]
    sc_full, sc_sh = oracle.make_scaler(4096.0), oracle.make_scaler(4096.0)
    t_full = t_sh = 0
    for step in range(1, 6):
        grads = []
        for _k in range(g):
            micro = []
            for _r in range(n):
                x = np.zeros(psi_pad, np.float32)
                x[:psi] = rng.standard_normal(psi) * 1e-3 * sc_full.scale
                micro.append(_lib_half(x, FP16))
            grads.append(micro)
        if step == 3:
            grads[0][1][2500] = 0x7C00  # an overflow in shard 3 only
        ovf_full, t_full, _ = oracle.shard_step(grads, FP16, full, hp, t_full, sc_full)
        per_shard = [[[np.ascontiguousarray(s[q * E:(q + 1) * E]) for s in micro] for micro in grads]
                     for q in range(n)]
        ovf_sh, t_sh, _ = oracle.multi_shard_step(per_shard, FP16, shards, hp, t_sh, sc_sh)
        assert ovf_full == ovf_sh == (1 if step == 3 else 0)
        assert t_full == t_sh and sc_full.scale == sc_sh.scale
        for name in ("master", "m", "v", "half"):
            cat = np.concatenate([getattr(s, name) for s in shards])
            assert cat.tobytes() == getattr(full, name).tobytes(), name
    # padding stays zero
    assert (full.master[psi:] == 0).all() and (full.half[psi:] == 0).all()


def test_bucket_invariance():
    rng = np.random.default_rng(5)
    count, n, g = 5000, 3, 2
    hp = oracle.make_hparams(1e-3, 0.9, 0.999, 1e-8, 0.1)
    master0 = (rng.standard_normal(count) * 0.02).astype(np.float32)
    grads = [_rand_slices(rng, n, count, 256.0) for _ in range(g)]
    whole = oracle.ShardState.from_master(master0, FP16)
    oracle.shard_step(grads, FP16, whole, hp, 0, oracle.make_scaler(256.0))
    for bucket in (1, 7, 64, 1000, 4999):
        parts = oracle.ShardState.from_master(master0, FP16)
        accs = np.zeros(count, np.float32)
        for b in range(0, count, bucket):
            e = min(count, b + bucket)
            acc = np.zeros(e - b, np.float32)
            for k in range(g):
                oracle.reduce_accumulate([np.ascontiguousarray(s[b:e]) for s in grads[k]], FP16,
                                         acc, first=(k == 0))
            accs[b:e] = acc
        for b in range(0, count, bucket):
            e = min(count, b + bucket)
            sl = [np.ascontiguousarray(a[b:e]) for a in (parts.master, parts.m, parts.v)]
            hh = np.ascontiguousarray(parts.half[b:e])
            oracle.adamw_apply(np.ascontiguousarray(accs[b:e]), n * g * 256.0, sl[0], sl[1], sl[2],
                               hh, FP16, hp, 1)
            parts.master[b:e], parts.m[b:e], parts.v[b:e], parts.half[b:e] = sl[0], sl[1], sl[2], hh
        for name in ("master", "m", "v", "half"):
            assert getattr(parts, name).tobytes() == getattr(whole, name).tobytes()


def test_flat_workload_scale_trajectory_small():
    """The 2-rank flat workload's schedule at a reduced size: +inf at step 5
    (rank 1, micro-step 1) -> that step skips, the scale ends at 2^15, t = 9."""
    import synth
    wl = synth.WORKLOADS["flat-1m-n2"]
    psi = 1 << 14
    idx_all = np.arange(psi, dtype=np.int64)
    E = psi // 2
    hp = oracle.make_hparams(wl.lr, wl.beta1, wl.beta2, wl.eps, wl.weight_decay)
    master0 = synth.host_master(wl, idx_all)
    states = [oracle.ShardState.from_master(master0[q * E:(q + 1) * E], FP16) for q in range(2)]
    sc = oracle.make_scaler(wl.scale0, wl.min_scale, wl.window, wl.hysteresis, wl.dynamic)
    t = 0
    flags = []
    for step in range(1, wl.steps + 1):
        full = [synth.host_grad_bits(wl, idx_all, step, 1, r, sc.scale) for r in range(2)]
        per = [[[np.ascontiguousarray(f[q * E:(q + 1) * E]) for f in full]] for q in range(2)]
        ovf, t, _ = oracle.multi_shard_step(per, FP16, states, hp, t, sc)
        flags.append(ovf)
    assert flags == [0, 0, 0, 0, 1, 0, 0, 0, 0, 0]
    assert sc.scale == 2.0 ** 15 and t == 9
    assert math.isfinite(float(np.abs(states[0].master).max()))


def test_bf16_sum_past_fp32_max_is_an_overflow():
    # two finite bf16 values near 3e38 sum past the fp32 maximum: the step skips
    hp = oracle.make_hparams(1e-4, 0.9, 0.999, 1e-8, 0.0)
    st = oracle.ShardState.from_master(np.array([0.5, 0.25], np.float32), BF16)
    before = st.copy()
    big = _h([3.0e38, 1.0], BF16)
    assert oracle.any_nonfinite([big, big], BF16, 2) == 0
    sc = oracle.make_scaler(1.0, dynamic=False)
    ovf, t, acc = oracle.shard_step([[big, big]], BF16, st, hp, 0, sc)
    assert ovf == 1 and t == 0 and np.isinf(acc[0])
    assert st.master.tobytes() == before.master.tobytes()


# ---------------------------------------------------------------- clipping

def test_clip_coefficient_closed_form():
    # n equal gradients c: norm = |c|·sqrt(n); coef = max_norm / (norm + 1e-6) when below 1
    n, c, div = 400, 0.0625, 2.0 ** 18
    acc = np.full(n, c * div, np.float32)
    sumsq = oracle.grad_sumsq(acc, div)
    assert abs(sumsq - n * c * c) <= 1e-12 * n * c * c
    norm = c * math.sqrt(n)  # 1.25
    assert abs(oracle.clip_coef(sumsq, 0.25) - 0.25 / (norm + 1e-6)) < 1e-15
    assert oracle.clip_coef(sumsq, 2.0) == 1.0        # under the limit: untouched
    assert oracle.clip_coef(sumsq, 0.0) == 1.0        # disabled


def test_clipped_first_step_moments():
    # t=1 from m=v=0: m1 = (1-β1)·ĝ·coef and v1 = (1-β2)·(ĝ·coef)², coef from the whole vector
    hp = oracle.make_hparams(1e-3, 0.9, 0.999, 1e-8, 0.0)
    rng = np.random.default_rng(12)
    ghat = rng.standard_normal(1000) * 0.1
    div = 1024.0
    acc = (ghat * div).astype(np.float32)
    ghat = acc.astype(np.float64) / div
    norm = math.sqrt(float((ghat ** 2).sum()))
    coef = 0.5 / (norm + 1e-6)
    assert coef < 1
    st = oracle.ShardState.from_master(np.zeros(1000, np.float32), FP16)
    sumsq = oracle.grad_sumsq(acc, div)
    oracle.adamw_apply_clipped(acc, div, oracle.clip_coef(sumsq, 0.5), st.master, st.m, st.v,
                               st.half, FP16, hp, 1)
    want_m = (1 - hp.beta1) * ghat * coef
    want_v = (1 - hp.beta2) * (ghat * coef) ** 2
    assert np.all(np.abs(st.m - want_m) <= 1e-6 * np.abs(want_m) + 1e-12)
    assert np.all(np.abs(st.v - want_v) <= 1e-6 * np.abs(want_v) + 1e-15)


def test_unclipped_step_is_bitwise_the_plain_step():
    rng = np.random.default_rng(13)
    n, g, count = 2, 2, 777
    hp = oracle.make_hparams(1e-4, 0.9, 0.999, 1e-8, 0.01)
    master0 = (rng.standard_normal(count) * 0.02).astype(np.float32)
    grads = [_rand_slices(rng, n, count, 512.0) for _ in range(g)]
    a = oracle.ShardState.from_master(master0, FP16)
    b = oracle.ShardState.from_master(master0, FP16)
    oracle.shard_step(grads, FP16, a, hp, 0, oracle.make_scaler(512.0))
    _, _, _, norm = oracle.shard_step(grads, FP16, b, hp, 0, oracle.make_scaler(512.0),
                                      max_norm=1e9, return_norm=True)
    assert norm > 0
    for k in ("master", "m", "v", "half"):
        assert getattr(a, k).tobytes() == getattr(b, k).tobytes()


def test_clipped_shard_union_uses_the_global_norm():
    rng = np.random.default_rng(14)
    psi, n = 2048, 4
    psi_pad, E = oracle.partition(psi, n, 64)
    hp = oracle.make_hparams(1e-3, 0.9, 0.999, 1e-8, 0.0)
    master0 = (rng.standard_normal(psi_pad) * 0.02).astype(np.float32)
    full_g = [[_lib_half((rng.standard_normal(psi_pad) * 0.5 * 256).astype(np.float32), FP16)
               for _ in range(n)]]
    whole = oracle.ShardState.from_master(master0, FP16)
    _, _, _, norm = oracle.shard_step(full_g, FP16, whole, hp, 0, oracle.make_scaler(256.0),
                                      max_norm=0.1, return_norm=True)
    assert norm > 0.1   # clipping active
    shards = [oracle.ShardState.from_master(master0[q * E:(q + 1) * E], FP16) for q in range(n)]
    per = [[[np.ascontiguousarray(s[q * E:(q + 1) * E]) for s in full_g[0]]] for q in range(n)]
    oracle.multi_shard_step(per, FP16, shards, hp, 0, oracle.make_scaler(256.0), max_norm=0.1)
    cat = np.concatenate([s.master for s in shards])
    # the global norm is a sum of per-shard sums (fp64 grouping may differ in the last bit)
    assert np.all(np.abs(cat - whole.master) <= np.spacing(np.abs(whole.master)))


# ---------------------------------------------------------------- LR schedules (§4.4)

def test_warmup_decay_schedule_of_the_pages():
    # §4.4's WarmupDecayLR example: min 0, max 3e-4, 2000 warmup steps, 100000 total, linear
    lr = lambda t: oracle.lr_at(oracle.LR_WARMUP_DECAY, 0.0, 3e-4, 2000, 100000, t)  # noqa: E731
    assert lr(0) == 0.0
    assert lr(1000) == pytest.approx(1.5e-4, rel=1e-15)       # half way up
    assert lr(2000) == pytest.approx(3e-4, rel=1e-15)         # peak at the end of warmup
    assert lr(51000) == pytest.approx(1.5e-4, rel=1e-15)      # half way down
    assert lr(100000) == 0.0 and lr(150000) == 0.0            # decayed to zero, stays there
    ts = np.arange(0, 100001, 97)
    vals = np.array([lr(int(t)) for t in ts])
    up = ts <= 2000
    assert np.all(np.diff(vals[up]) > 0) and np.all(np.diff(vals[~up]) <= 0)


def test_warmup_and_constant_schedules():
    w = lambda t: oracle.lr_at(oracle.LR_WARMUP, 1e-5, 1e-3, 100, 0, t)  # noqa: E731
    assert w(0) == 1e-5 and w(50) == pytest.approx(5.05e-4) and w(100) == 1e-3
    assert w(10 ** 6) == 1e-3                                  # flat after warmup
    assert oracle.lr_at(oracle.LR_CONSTANT, 0.0, 2e-4, 10, 20, 7) == 2e-4
    assert oracle.lr_at(oracle.LR_WARMUP, 0.0, 2e-4, 0, 0, 1) == 2e-4  # no warmup


# ---------------------------------------------------------------- half accumulator

def test_half_accumulator_rounds_each_micro_step():
    # fp16 spacing at 2048 is 2: a carried half accumulator loses the odd unit that an
    # fp32 accumulator keeps
    one, big = _h([1.0]), _h([2048.0])
    acc_h = np.zeros(1, np.uint16)
    oracle.reduce_accumulate_half([big], FP16, acc_h, True)
    oracle.reduce_accumulate_half([one], FP16, acc_h, False)   # 2049 -> ties to even: 2048
    assert oracle.half_to_double(acc_h, FP16)[0] == 2048.0
    acc_f = np.zeros(1, np.float32)
    oracle.reduce_accumulate([big], FP16, acc_f, True)
    oracle.reduce_accumulate([one], FP16, acc_f, False)
    assert acc_f[0] == 2049.0
    # within one micro-step the ranks still sum in fp32 before the single rounding
    acc_h[:] = 0
    oracle.reduce_accumulate_half([big, one, one], FP16, acc_h, True)   # 2050 exactly
    assert oracle.half_to_double(acc_h, FP16)[0] == 2050.0


def test_half_accumulator_overflow_skips():
    # 40000 + 30000 is finite in fp32 but rounds past 65504: the step skips
    hp = oracle.make_hparams(1e-3, 0.9, 0.999, 1e-8, 0.0)
    st = oracle.ShardState.from_master(np.array([0.1], np.float32), FP16)
    before = st.copy()
    sc = oracle.make_scaler(1024.0)
    ovf, t, acc = oracle.shard_step_halfacc([[_h([40000.0])], [_h([30000.0])]], FP16, st, hp,
                                            0, sc)
    assert ovf == 1 and t == 0 and acc[0] == 0x7C00 and sc.scale == 512.0
    assert st.master.tobytes() == before.master.tobytes()
    # the fp32 accumulator does not overflow on the same inputs
    st2 = oracle.ShardState.from_master(np.array([0.1], np.float32), FP16)
    ovf2, _, _ = oracle.shard_step([[_h([40000.0])], [_h([30000.0])]], FP16, st2, hp, 0,
                                   oracle.make_scaler(1024.0))
    assert ovf2 == 0


def test_half_accumulator_equals_fp32_when_sums_are_representable():
    # integer gradients with small sums are exact in both accumulators: same step, bitwise
    rng = np.random.default_rng(40)
    n, g, count = 3, 3, 500
    grads = [[_h(rng.integers(-20, 20, count).astype(np.float32)) for _ in range(n)]
             for _ in range(g)]
    hp = oracle.make_hparams(1e-3, 0.9, 0.999, 1e-8, 0.01)
    master0 = (rng.standard_normal(count) * 0.02).astype(np.float32)
    a = oracle.ShardState.from_master(master0, FP16)
    b = oracle.ShardState.from_master(master0, FP16)
    oracle.shard_step(grads, FP16, a, hp, 0, oracle.make_scaler(16.0))
    oracle.shard_step_halfacc(grads, FP16, b, hp, 0, oracle.make_scaler(16.0))
    for k in ("master", "m", "v", "half"):
        assert getattr(a, k).tobytes() == getattr(b, k).tobytes()


# ---------------------------------------------------------------- randomized invariants

@pytest.mark.parametrize("seed", range(12))
def test_random_union_and_bucket_invariance(seed):
    """Random layouts: the union of N shard steps (global flag, one scale) equals
    the unpartitioned step bit for bit, and so does any bucketing of one shard."""
    rng = np.random.default_rng(100 + seed)
    psi = int(rng.integers(1, 3000))
    n = int(rng.integers(1, 9))
    g = int(rng.integers(1, 4))
    align = int(rng.choice([1, 8, 64]))
    dtype = int(rng.integers(0, 2))
    psi_pad, E = oracle.partition(psi, n, align)
    hp = oracle.make_hparams(float(rng.choice([1e-4, 3e-4, 1e-3])), 0.9, 0.999, 1e-8,
                             float(rng.choice([0.0, 0.01, 0.1])))
    master0 = np.zeros(psi_pad, np.float32)
    master0[:psi] = rng.standard_normal(psi) * 0.02
    scale = 256.0 if dtype == FP16 else 1.0
    grads = []
    for _ in range(g):
        micro = []
        for _ in range(n):
            x = np.zeros(psi_pad, np.float32)
            x[:psi] = rng.standard_normal(psi) * 1e-2 * scale
            micro.append(_lib_half(x, dtype))
        grads.append(micro)
    if rng.random() < 0.3:
        grads[int(rng.integers(0, g))][int(rng.integers(0, n))][int(rng.integers(0, psi))] = \
            0x7C00 if dtype == FP16 else 0x7F80
    full = oracle.ShardState.from_master(master0, dtype)
    sc_a = oracle.make_scaler(scale, dynamic=(dtype == FP16))
    ovf_a, t_a, acc_full = oracle.shard_step(grads, dtype, full, hp, 0, sc_a)
    shards = [oracle.ShardState.from_master(master0[q * E:(q + 1) * E], dtype) for q in range(n)]
    per = [[[np.ascontiguousarray(s[q * E:(q + 1) * E]) for s in micro] for micro in grads]
           for q in range(n)]
    sc_b = oracle.make_scaler(scale, dynamic=(dtype == FP16))
    ovf_b, t_b, _ = oracle.multi_shard_step(per, dtype, shards, hp, 0, sc_b)
    assert (ovf_a, t_a, sc_a.scale) == (ovf_b, t_b, sc_b.scale)
    for name in ("master", "m", "v", "half"):
        cat = np.concatenate([getattr(s, name) for s in shards])
        assert cat.tobytes() == getattr(full, name).tobytes()
    # bucketing of shard 0's accumulation
    bucket = int(rng.integers(1, max(2, E)))
    acc_b = np.zeros(E, np.float32)
    for b in range(0, E, bucket):
        e = min(E, b + bucket)
        part = np.zeros(e - b, np.float32)
        for k in range(g):
            oracle.reduce_accumulate([np.ascontiguousarray(s[b:e]) for s in per[0][k]], dtype,
                                     part, first=(k == 0))
        acc_b[b:e] = part
    assert acc_b.tobytes() == acc_full[:E].tobytes()


# ------------------------------------------ multi-step against a library AdamW

def _f32_sequential_sum(grads, dtype):
    """Per element: +0.0, then every micro-step's ranks in order, each an IEEE
    fp32 add (numpy float32 arithmetic, independent of the oracle's C)."""
    a = np.zeros(grads[0][0].shape[0], np.float32)
    for micro in grads:
        for bits in micro:
            if dtype == FP16:
                x = bits.view(np.float16).astype(np.float32)
            else:
                x = (bits.astype(np.uint32) << 16).view(np.float32)
            a = (a + x).astype(np.float32)
    return a


@pytest.mark.parametrize("dtype,n,g,max_norm,wd", [(FP16, 3, 2, 0.0, 0.01), (BF16, 2, 3, 0.0, 0.1),
                                                    (FP16, 4, 1, 0.01, 0.01),
                                                    (BF16, 1, 2, 1e-3, 0.0)])
def test_ten_steps_match_torch_adamw(dtype, n, g, max_norm, wd):
    """Ten steps (one skipped on an injected inf/NaN, the scale halving for fp16)
    of the oracle against torch.optim.AdamW in fp64 (and clip_grad_norm_ when
    clipping), fed the unscaled mean gradient acc / (N·G·S) of an fp32 sum taken
    here, with master, m and v rounded to fp32 after every step on the torch side
    too.  The two differ only in fp64 rounding order, so the stored fp32 state
    must agree to one ulp (nearly everywhere bit for bit)."""
    rng = np.random.default_rng(1000 * n + 10 * g + dtype)
    count = 4099
    hp = oracle.make_hparams(1e-3, 0.9, 0.999, 1e-8, wd)
    lr, b1, b2, eps, wdf = (float(hp.lr), float(hp.beta1), float(hp.beta2), float(hp.eps),
                            float(hp.weight_decay))
    master0 = (rng.standard_normal(count) * 0.02).astype(np.float32)
    st = oracle.ShardState.from_master(master0, dtype)
    dyn = dtype == FP16
    sc = oracle.make_scaler(1024.0 if dyn else 1.0, 1.0, 1000, 1, dyn)
    p = torch.tensor(master0.astype(np.float64), requires_grad=True)
    opt = torch.optim.AdamW([p], lr=lr, betas=(b1, b2), eps=eps, weight_decay=wdf,
                            foreach=False)
    t = 0
    applied = 0
    for s in range(1, 11):
        S = sc.scale
        grads = [[_lib_half((rng.standard_normal(count) * 1e-3 * S).astype(np.float32), dtype)
                  for _ in range(n)] for _ in range(g)]
        if s == 4:
            grads[g - 1][n - 1][77] = 0x7C00 if dtype == FP16 else 0x7FC0
        acc = _f32_sequential_sum(grads, dtype)
        ovf, t, _ = oracle.shard_step(grads, dtype, st, hp, t, sc, max_norm=max_norm)
        assert ovf == (s == 4)
        if ovf:
            continue
        applied += 1
        p.grad = torch.from_numpy(acc.astype(np.float64) / (n * g * S))
        if max_norm > 0:
            torch.nn.utils.clip_grad_norm_([p], max_norm)
        opt.step()
        with torch.no_grad():   # the stored state is fp32
            p.copy_(p.float().double())
            for key in ("exp_avg", "exp_avg_sq"):
                buf = opt.state[p][key]
                buf.copy_(buf.float().double())
    assert t == applied == 9
    if dyn:
        assert sc.scale == 512.0
    _same_fp32_state(st, p, opt, dtype)


def _same_fp32_state(st, p, opt, dtype):
    for got, want in ((st.master, p.detach()), (st.m, opt.state[p]["exp_avg"]),
                      (st.v, opt.state[p]["exp_avg_sq"])):
        want = want.float().numpy()
        gi, wi = got.view(np.int32).astype(np.int64), want.view(np.int32).astype(np.int64)
        assert np.abs(gi - wi).max() <= 1
        assert (gi == wi).mean() > 0.999
    assert (st.half == _lib_half(st.master, dtype)).all()


def _half_sequential_sum(grads, dtype):
    """The half accumulator written out with numpy/torch: per micro-step an fp32
    sum from the rounded accumulator (or +0.0) over the ranks in order, rounded
    to the half format to nearest even."""
    a = np.zeros(grads[0][0].shape[0], np.uint16)
    for k, micro in enumerate(grads):
        x = np.zeros(a.shape[0], np.float32) if k == 0 else _decode(a, dtype)
        for bits in micro:
            x = (x + _decode(bits, dtype)).astype(np.float32)
        a = _lib_half(x, dtype)
    return a


def _decode(bits, dtype):
    if dtype == FP16:
        return bits.view(np.float16).astype(np.float32)
    return (bits.astype(np.uint32) << 16).view(np.float32)


@pytest.mark.parametrize("dtype,n,g", [(FP16, 2, 3), (BF16, 3, 2)])
def test_half_accumulator_steps_match_torch_adamw(dtype, n, g):
    """The half-accumulator step: ten steps of the oracle against torch's AdamW
    in fp64 fed the half sum (written out here) / (N·G·S), fp32 state on both
    sides."""
    rng = np.random.default_rng(77 + n + dtype)
    count = 3001
    hp = oracle.make_hparams(1e-3, 0.9, 0.999, 1e-8, 0.01)
    master0 = (rng.standard_normal(count) * 0.02).astype(np.float32)
    st = oracle.ShardState.from_master(master0, dtype)
    dyn = dtype == FP16
    sc = oracle.make_scaler(1024.0 if dyn else 1.0, 1.0, 1000, 1, dyn)
    p = torch.tensor(master0.astype(np.float64), requires_grad=True)
    opt = torch.optim.AdamW([p], lr=float(hp.lr), betas=(float(hp.beta1), float(hp.beta2)),
                            eps=float(hp.eps), weight_decay=float(hp.weight_decay), foreach=False)
    t = 0
    for s in range(1, 11):
        S = sc.scale
        grads = [[_lib_half((rng.standard_normal(count) * 1e-3 * S).astype(np.float32), dtype)
                  for _ in range(n)] for _ in range(g)]
        acc = _half_sequential_sum(grads, dtype)
        ovf, t, acc_o = oracle.shard_step_halfacc(grads, dtype, st, hp, t, sc)
        assert ovf == 0 and (acc_o == acc).all()
        p.grad = torch.from_numpy(_decode(acc, dtype).astype(np.float64) / (n * g * S))
        opt.step()
        with torch.no_grad():
            p.copy_(p.float().double())
            for key in ("exp_avg", "exp_avg_sq"):
                buf = opt.state[p][key]
                buf.copy_(buf.float().double())
    assert t == 10
    _same_fp32_state(st, p, opt, dtype)
