"""zs_check_last, the flag-only pass over a step's last micro-step for callers
that exchange the flag before the update: its flag against the oracle's
overflow rule, and reduce_check x (G-1) + check_last + apply + scaler update
equal to zs_shard_step bit for bit."""
import numpy as np
import pytest
import torch

import oracle
from _helpers import dev16, lib_half

pytestmark = pytest.mark.gpu

FP16, BF16 = 0, 1
BITS = {(FP16, "inf"): 0x7C00, (FP16, "nan"): 0x7E00, (BF16, "inf"): 0x7F80, (BF16, "nan"): 0x7FC0}


@pytest.fixture(scope="module")
def zs():
    import zero_mixed_precision_shard_gb300 as pkg
    torch.cuda.set_device(0)
    return pkg


@pytest.fixture(scope="module")
def ctx(zs):
    c = zs.Ctx()
    yield c
    c.close()


@pytest.mark.parametrize("dtype", [FP16, BF16])
@pytest.mark.parametrize("n", [1, 3])
@pytest.mark.parametrize("with_acc", [False, True])
@pytest.mark.parametrize("where", [None, 0, 4096, "tail"])
def test_flag_matches_the_oracle(zs, ctx, dtype, n, with_acc, where):
    rng = np.random.default_rng(n * 10 + dtype)
    count = 20_003
    g = [lib_half(rng.standard_normal(count).astype(np.float32), dtype) for _ in range(n)]
    kind = "nan" if n == 3 else "inf"
    if where is not None:
        i = count - 1 if where == "tail" else where
        g[n - 1][i] = BITS[(dtype, kind)]
    acc0 = (rng.standard_normal(count) * 10).astype(np.float32)
    final = acc0.copy() if with_acc else np.zeros(count, np.float32)
    oracle.reduce_accumulate(g, dtype, final, first=not with_acc)
    want = int(oracle.any_nonfinite(g, dtype, count) or oracle.any_nonfinite_f32(final))
    assert want == (where is not None)
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    acc = torch.from_numpy(acc0).cuda() if with_acc else None
    before = acc.clone() if with_acc else None
    zs.zs_check_last(ctx, [dev16(x) for x in g], dtype, count, acc, flag)
    assert int(flag.item()) == want
    if with_acc:
        assert torch.equal(acc, before)      # nothing written


def test_bf16_sum_past_fp32_max_on_top_of_acc(zs, ctx):
    # finite bf16 halves whose sum with a finite accumulator passes the fp32 maximum
    count = 24
    acc = torch.full((count,), 3.0e38, dtype=torch.float32, device="cuda")
    g = lib_half(np.full(count, 1.0, np.float32), BF16)
    g[13] = lib_half(np.array([1.0e38], np.float32), BF16)[0]
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    zs.zs_check_last(ctx, [dev16(g)], BF16, count, acc, flag)
    assert int(flag.item()) == 1
    flag.zero_()
    zs.zs_check_last(ctx, [dev16(g)], BF16, count, None, flag)   # the slices alone are finite
    assert int(flag.item()) == 0


@pytest.mark.parametrize("dtype,n,G", [(FP16, 1, 4), (FP16, 2, 1), (BF16, 3, 2), (BF16, 1, 3)])
def test_split_step_equals_shard_step_bitwise(zs, ctx, dtype, n, G):
    rng = np.random.default_rng(5 + n + G)
    count = 50_008
    S0 = 1024.0 if dtype == FP16 else 1.0
    dyn = dtype == FP16
    master0 = (rng.standard_normal(count) * 0.02).astype(np.float32)
    sides = []
    for _ in range(2):
        master = torch.from_numpy(master0.copy()).cuda()
        sides.append({"master": master, "m": torch.zeros_like(master),
                      "v": torch.zeros_like(master),
                      "half": torch.zeros(count, dtype=torch.int16, device="cuda"),
                      "acc": torch.zeros_like(master),
                      "sc": zs.zs_scaler_init(S0, 1.0, 3, 1, dyn), "t": 0, "flags": []})
    hp = zs.make_hparams(1e-3, 0.9, 0.999, 1e-8, 0.01)
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    for s in range(1, 7):
        S = sides[0]["sc"].scale
        grads = [[dev16(lib_half((rng.standard_normal(count) * 1e-3 * S).astype(np.float32),
                                 dtype)) for _ in range(n)] for _ in range(G)]
        if s == 3:
            grads[G - 1][n - 1][11] = BITS[(dtype, "inf")]
        a = sides[0]   # the fused call
        for k in range(G - 1):
            zs.zs_grad_accum(ctx, grads[k], dtype, count, a["acc"], k == 0)
        ovf, _ = zs.zs_shard_step(ctx, grads[G - 1], dtype, count, a["acc"] if G > 1 else None, G,
                                  a["master"], a["m"], a["v"], a["half"], hp, a["t"] + 1, a["sc"])
        a["flags"].append(ovf)
        if not ovf:
            a["t"] += 1
        b = sides[1]   # split at the flag, as a multi-rank caller does
        flag.zero_()
        for k in range(G - 1):
            zs.zs_reduce_check(ctx, grads[k], dtype, count, b["acc"], k == 0, flag)
        zs.zs_check_last(ctx, grads[G - 1], dtype, count, b["acc"] if G > 1 else None, flag)
        zs.zs_apply(ctx, flag, grads[G - 1], dtype, b["acc"] if G > 1 else None, count,
                    float(n * G * b["sc"].scale), b["master"], b["m"], b["v"], b["half"], hp,
                    b["t"] + 1)
        ovf = zs.zs_scaler_update(ctx, flag, b["sc"])
        b["flags"].append(ovf)
        if not ovf:
            b["t"] += 1
    assert sides[0]["flags"] == sides[1]["flags"] == [0, 0, 1, 0, 0, 0]
    assert sides[0]["t"] == sides[1]["t"] == 5
    assert sides[0]["sc"].scale == sides[1]["sc"].scale
    for k in ("master", "m", "v", "half"):
        assert torch.equal(sides[0][k], sides[1][k]), k


def test_argument_errors(zs, ctx):
    x = torch.zeros(64, dtype=torch.float32, device="cuda")
    h = torch.zeros(64, dtype=torch.int16, device="cuda")
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    for args, status in (
            (([h[1:]], FP16, 8, None, flag), zs.ZS_ERR_ALIGN),     # misaligned slice
            (([h], FP16, 8, x[1:], flag), zs.ZS_ERR_ALIGN),       # misaligned acc
            (([h], 7, 8, None, flag), zs.ZS_ERR_DTYPE),
            (([], FP16, 8, None, flag), zs.ZS_ERR_ARG),            # no ranks
            (([h] * 257, FP16, 8, None, flag), zs.ZS_ERR_ARG),     # more than 256 ranks
            (([h], FP16, -8, None, flag), zs.ZS_ERR_ARG),
            (([h], FP16, 8, None, None), zs.ZS_ERR_ARG)):          # no flag
        with pytest.raises(zs.ZsError) as e:
            zs.zs_check_last(ctx, *args)
        assert e.value.status == status, args[1:3]
    # an empty range checks nothing and leaves the flag alone
    flag.fill_(0)
    zs.zs_check_last(ctx, [h], FP16, 0, None, flag)
    assert int(flag.item()) == 0
