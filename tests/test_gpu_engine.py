"""zs_engine (backward per micro-batch, step after each, §5.1) against the
oracle: the engine must reach the same state as the oracle's steps, run the
optimizer step only at accumulation boundaries, count global and applied steps,
follow the learning-rate schedule and clip when asked."""
import numpy as np
import pytest
import torch

import oracle
from _helpers import STRESS_LR, assert_close

pytestmark = pytest.mark.gpu

FP16 = 0


@pytest.fixture(scope="module")
def zs():
    import zero_mixed_precision_shard_gb300 as pkg
    torch.cuda.set_device(0)
    return pkg


def close(got, want, name):
    assert_close(got, want, name)


@pytest.mark.parametrize("n,G,clip,sched", [(2, 3, 0.0, False), (8, 1, 0.05, True),
                                            (1, 4, 0.0, True)])
def test_engine_loop_matches_oracle(zs, n, G, clip, sched):
    rng = np.random.default_rng(n + 10 * G)
    count = 30_016
    master0 = (rng.standard_normal(count) * 0.02).astype(np.float32)
    st = oracle.ShardState.from_master(master0, FP16)
    sc_o = oracle.make_scaler(512.0, 1.0, 3, 1, True)
    lr_max, lr_min, wu, tot = float(np.float32(STRESS_LR)), float(np.float32(1e-5)), 3, 12
    schedule = zs.make_schedule(zs.ZS_LR_WARMUP_DECAY, lr_min, lr_max, wu, tot) if sched else None
    ctx = zs.Ctx()
    master = torch.from_numpy(master0.copy()).cuda()
    m, v = torch.zeros_like(master), torch.zeros_like(master)
    half = torch.zeros(count, dtype=torch.int16, device="cuda")
    acc = torch.zeros(count, dtype=torch.float32, device="cuda")
    eng = zs.Engine(ctx, n, FP16, count, G, acc, master, m, v, half,
                    zs.make_hparams(lr_max, 0.9, 0.999, 1e-8, 0.01),
                    zs.zs_scaler_init(512.0, 1.0, 3, 1, True), schedule, clip)
    t_o = 0
    steps = 8
    for s in range(1, steps + 1):
        grads = [[(rng.standard_normal(count) * 1e-2 * sc_o.scale).astype(np.float16)
                  .view(np.uint16) for _ in range(n)] for _ in range(G)]
        if s == 3:
            grads[G - 1][0][11] = 0x7C00
        lr_t = oracle.lr_at(oracle.LR_WARMUP_DECAY, lr_min, lr_max, wu, tot, t_o + 1) if sched \
            else lr_max
        hp_o = oracle.make_hparams(lr_t, 0.9, 0.999, 1e-8, 0.01)
        ovf_o, t_o, _, norm_o = oracle.shard_step(grads, FP16, st, hp_o, t_o, sc_o,
                                                  max_norm=clip, return_norm=True)
        keep = []
        for k in range(G):
            dg = [torch.from_numpy(x.view(np.int16)).cuda() for x in grads[k]]
            keep.append(dg)
            eng.backward(dg)
            r = eng.step()
            if k < G - 1:
                assert r is None
        ovf, ns, norm = r
        assert ovf == ovf_o and ns == sc_o.scale, f"step {s}"
        if clip > 0 and not ovf:
            assert abs(norm - norm_o) <= 1e-6 * norm_o
    state = eng.state()
    assert state["global_steps"] == steps and state["applied_steps"] == t_o == steps - 1
    assert state["micro_steps"] == steps * G and state["scaler"].scale == sc_o.scale
    close(master.cpu().numpy(), st.master, "master")
    close(m.cpu().numpy(), st.m, "m")
    close(v.cpu().numpy(), st.v, "v")
    eng.close()
    ctx.close()


def test_engine_rejects_backward_past_the_boundary(zs):
    ctx = zs.Ctx()
    count = 64
    buf = [torch.zeros(count, device="cuda") for _ in range(3)]
    half = torch.zeros(count, dtype=torch.int16, device="cuda")
    eng = zs.Engine(ctx, 1, FP16, count, 1, None, buf[0], buf[1], buf[2], half,
                    zs.make_hparams(1e-3), zs.zs_scaler_init(1.0, 1.0, 10, 1, True))
    g = [torch.zeros(count, dtype=torch.int16, device="cuda")]
    eng.backward(g)
    with pytest.raises(zs.ZsError):
        eng.backward(g)
    assert eng.step() is not None
    eng.backward(g)
    eng.close()
    ctx.close()
