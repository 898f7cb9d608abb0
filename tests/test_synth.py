"""The seeded input generator: Philox4x64-10 against numpy's implementation,
the Irwin-Hall normal's moments and bounds, determinism, padding, injections
and the workload table's parameter counts.  No GPU."""
import numpy as np
import pytest

import synth


@pytest.mark.parametrize("ctr,key", [((0, 0, 0, 0), (0, 0)), ((5, 0, 0, 0), (7, 9)),
                                     ((2 ** 64 - 2, 3, 4, 5), (2 ** 63, 11)),
                                     ((123456789, 2 ** 40 + 17, 1, 0), (0, 5))])
def test_philox_matches_numpy(ctr, key):
    # numpy advances the counter by one before producing a block
    bg = np.random.Philox(counter=np.array(ctr, dtype=np.uint64), key=np.array(key, dtype=np.uint64))
    want = [int(x) for x in bg.random_raw(4)]
    c = list(ctr)
    c[0] = (c[0] + 1) % 2 ** 64
    if c[0] == 0:
        c[1] += 1
    assert synth.philox(c, key) == want


def test_normal_moments_and_bound():
    wl = synth.WORKLOADS["flat-1m-n2"]
    idx = np.arange(1 << 18)
    bits = synth.host_grad_bits(wl, idx, 1, 1, 0, 1.0 / wl.sigma)  # sigma*S = 1
    z = bits.view(np.float16).astype(np.float64)
    assert abs(z.mean()) < 0.01 and abs(z.std() - 1) < 0.01
    assert np.abs(z).max() <= 6.0
    m = synth.host_master(wl, idx)
    assert abs(m.std() - 0.02) < 2e-4 and np.abs(m).max() <= 6 * 0.02 + 1e-6


def test_deterministic_and_keyed():
    wl = synth.WORKLOADS["gpt2-small-n8"]
    idx = np.array([0, 1, 17, 10 ** 8, wl.psi - 1])
    a = synth.host_grad_bits(wl, idx, 3, 2, 5, 65536.0)
    assert (a == synth.host_grad_bits(wl, idx, 3, 2, 5, 65536.0)).all()
    for other in ((4, 2, 5), (3, 3, 5), (3, 2, 6)):
        assert (a != synth.host_grad_bits(wl, idx, *other, 65536.0)).any()


def test_padding_is_zero():
    wl = synth.WORKLOADS["gpt2-small-n8"]
    idx = np.array([wl.psi - 1, wl.psi, wl.psi + 255])
    bits = synth.host_grad_bits(wl, idx, 1, 1, 0, 65536.0)
    assert bits[1] == 0 and bits[2] == 0
    assert (synth.host_master(wl, idx)[1:] == 0).all()


def test_low_sigma_tensors_and_heavy_tail():
    wl = synth.WORKLOADS["gpt2-small-n8"]
    ranges = {n: (b, e) for n, b, e in wl.tensor_ranges()}
    assert len(wl.low_sigma_tensors) == 2
    name = wl.low_sigma_tensors[0][0]
    b, e = ranges[name]
    idx = np.arange(b, e)
    z = synth.host_grad_bits(wl, idx, 1, 1, 0, 65536.0).view(np.float16).astype(np.float64)
    # 1e-7 * 2^16 = 6.6e-3 stays a normal fp16 after scaling
    assert abs(z.std() - 1e-7 * 65536) < 0.05 * 1e-7 * 65536
    wl3 = synth.WORKLOADS["decoder-1.3b-n16"]
    idx = np.arange(1 << 18)
    import torch
    bits = synth.host_grad_bits(wl3, idx, 1, 1, 0, 1.0)
    x = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).double().numpy()
    frac_big = np.mean(np.abs(x) > 6.01 * wl3.sigma)
    # only Student-t(3) draws pass the Irwin-Hall bound: 1% x P(|t3| > 6) ~ 9e-5
    assert 3e-5 < frac_big < 3e-4


def test_injections():
    wl = synth.WORKLOADS["flat-1m-n2"]
    idx = np.array([12344, 12345, 12346])
    bits = synth.host_grad_bits(wl, idx, 5, 1, 1, 65536.0)
    assert bits[1] == synth.FP16_POS_INF and bits[0] != synth.FP16_POS_INF
    assert (synth.host_grad_bits(wl, idx, 5, 1, 0, 65536.0) != synth.FP16_POS_INF).all()
    assert (synth.host_grad_bits(wl, idx, 4, 1, 1, 65536.0) != synth.FP16_POS_INF).all()
    wl3 = synth.WORKLOADS["decoder-1.3b-n16"]
    assert [j.step for j in wl3.injections] == [7, 14]
    wl5 = synth.WORKLOADS["llama7b-n1"]
    assert [j.step for j in wl5.injections] == [100, 200]


def test_workload_parameter_counts():
    w = synth.WORKLOADS
    assert w["gpt2-small-n8"].psi == 124_439_808 and len(w["gpt2-small-n8"].tensors) == 148
    assert w["decoder-1.3b-n16"].psi == 1_315_723_264 and len(w["decoder-1.3b-n16"].tensors) == 292
    assert w["llama7b-n1"].psi == 6_738_415_616 and len(w["llama7b-n1"].tensors) == 291
    assert w["llama7b-zero3-n64"].psi == w["llama7b-n1"].psi
