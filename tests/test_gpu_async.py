"""The capture-friendly step (zs_shard_step_async, device-resident scaler,
Adam step count and learning-rate schedule) against the oracle, eagerly and
replayed from a CUDA graph: exact flags, scales and step counts, state within
1e-6 relative + 1e-9 absolute, half copies within 1 ulp."""
import numpy as np
import pytest
import torch

import oracle
from _helpers import STRESS_LR, assert_close, lib_half, ulps

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
    """1e-6 relative + 1e-9 absolute (these tests run at lr 3e-4)."""
    assert_close(got, want, name)


# kind, min, max, warmup, total; the rates as the fp32 values the library receives
SCHED = (oracle.LR_WARMUP_DECAY, float(np.float32(1e-5)), float(np.float32(STRESS_LR)), 3, 9)


def _run(zs, ctx, dtype, n, G, count, steps, graph, inject, max_norm=0.0):
    rng = np.random.default_rng(n * 10 + G + (100 if graph else 0))
    master0 = (rng.standard_normal(count) * 0.02).astype(np.float32)
    st = oracle.ShardState.from_master(master0, dtype)
    dyn = dtype == FP16
    sc_o = oracle.make_scaler(512.0 if dyn else 1.0, 1.0, 2, 1, dyn)
    kind, mn, mx, wu, tot = SCHED
    sched = zs.make_schedule(kind, mn, mx, wu, tot)
    hp = zs.make_hparams(mx, 0.9, 0.999, 1e-8, 0.01)
    state = zs.DeviceState(zs.zs_scaler_init(sc_o.scale, 1.0, 2, 1, dyn))
    master = torch.from_numpy(master0.copy()).cuda()
    m, v = torch.zeros_like(master), torch.zeros_like(master)
    half = torch.zeros(count, dtype=torch.int16, device="cuda")
    acc = torch.zeros(count, dtype=torch.float32, device="cuda")
    pad = (count + 7) // 8 * 8   # keeps every rank's slice 16-byte aligned
    gbuf = torch.zeros((G, n, pad), dtype=torch.int16, device="cuda")
    ptrs = [zs.pointer_array(gbuf[k, r, :count] for r in range(n)) for k in range(G)]

    norm = torch.zeros(1, dtype=torch.float64, device="cuda")

    def step_calls():
        for k in range(G - 1):
            zs.zs_grad_accum(ctx, ptrs[k], dtype, count, acc, k == 0)
        if max_norm > 0:
            zs.zs_shard_step_async_clipped(ctx, ptrs[G - 1], dtype, count, acc, G, master, m, v,
                                           half, hp, sched, max_norm, state, norm)
        else:
            zs.zs_shard_step_async(ctx, ptrs[G - 1], dtype, count, acc, G, master, m, v, half,
                                   hp, sched, state)

    g = None
    t_o = 0
    for s in range(1, steps + 1):
        grads = [[lib_half((rng.standard_normal(count) * 1e-2 * sc_o.scale).astype(np.float32),
                           dtype) for _ in range(n)] for _ in range(G)]
        if s in inject:
            grads[G - 1][n - 1][count - 1] = 0x7C00 if dtype == FP16 else 0x7F80
        host = np.stack([np.stack(mc) for mc in grads]).view(np.int16)
        gbuf[:, :, :count].copy_(torch.from_numpy(host))
        lr_t = oracle.lr_at(kind, mn, mx, wu, tot, t_o + 1)
        hp_o = oracle.make_hparams(lr_t, 0.9, 0.999, 1e-8, 0.01)
        ovf_o, t_o, _, norm_o = oracle.shard_step(grads, dtype, st, hp_o, t_o, sc_o,
                                                  max_norm=max_norm, return_norm=True)
        if graph:
            if g is None:
                step_calls()               # uncaptured first call: caches launch shapes
                torch.cuda.synchronize()
                # undo nothing: that call was step s; capture the next steps
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g):
                    step_calls()
            else:
                g.replay()
        else:
            step_calls()
        d = state.read()
        assert d.overflow == ovf_o, f"step {s}"
        assert d.scaler.scale == sc_o.scale and d.scaler.clean_count == sc_o.clean_count
        assert d.step == t_o and d.iterations == s
        if not ovf_o:
            assert d.lr == np.float32(lr_t)
            if max_norm > 0:
                assert abs(norm.item() - norm_o) <= 1e-6 * norm_o, (s, norm.item(), norm_o)
    close(master.cpu().numpy(), st.master, "master")
    close(m.cpu().numpy(), st.m, "m")
    close(v.cpu().numpy(), st.v, "v")
    assert ulps(half.cpu().numpy().view(np.uint16), st.half).max() <= 1


@pytest.mark.parametrize("dtype", [FP16, BF16])
@pytest.mark.parametrize("n,G,count", [(1, 3, 20_011), (2, 1, 8_192), (8, 2, 40_003)])
def test_async_steps_match_oracle(zs, ctx, dtype, n, G, count):
    _run(zs, ctx, dtype, n, G, count, 10, graph=False, inject={4, 5})


@pytest.mark.parametrize("n,G,count", [(1, 3, 20_011), (8, 2, 40_003)])
def test_graph_replayed_steps_match_oracle(zs, ctx, n, G, count):
    _run(zs, ctx, FP16, n, G, count, 10, graph=True, inject={6})


@pytest.mark.parametrize("dtype", [FP16, BF16])
@pytest.mark.parametrize("n,G,count,max_norm", [(1, 3, 20_011, 0.02), (8, 2, 40_003, 0.05),
                                                (2, 1, 8_192, 1e6)])
def test_async_clipped_steps_match_oracle(zs, ctx, dtype, n, G, count, max_norm):
    """The device-resident step with global-norm clipping: the norm formed in
    the last micro-step's pass and divided by N*G*S on the device, the clipped
    update, against the oracle's clipped steps (re-read and materialised forms;
    a max_norm that never clips)."""
    _run(zs, ctx, dtype, n, G, count, 10, graph=False, inject={4}, max_norm=max_norm)


@pytest.mark.parametrize("n,G,count", [(1, 3, 20_011), (8, 2, 40_003)])
def test_graph_replayed_clipped_steps_match_oracle(zs, ctx, n, G, count):
    _run(zs, ctx, FP16, n, G, count, 10, graph=True, inject={6}, max_norm=0.03)
