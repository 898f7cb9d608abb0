"""The device side of the seeded input generator writes the same bits as the
host side (which feeds the oracle): contiguous ranges and sampled indices of
every workload's gradients (fp16, bf16 with Student-t tails, per-tensor sigma),
master initial values, padding, and injections."""
import numpy as np
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", ["flat-1m-n2", "gpt2-small-n8", "decoder-1.3b-n16",
                                  "llama7b-zero3-n64", "llama7b-n1"])
def test_device_generator_matches_host(name):
    torch.cuda.set_device(0)
    wl = synth.WORKLOADS[name]
    rng = np.random.default_rng(3)
    starts = [0, max(0, wl.psi - 5000), int(rng.integers(0, max(1, wl.psi - 5000)))]
    low = dict(wl.low_sigma_tensors)
    starts += [max(0, b - 100) for t, b, _ in wl.tensor_ranges() if t in low][:3]
    cases = [(b, s, k, r) for b in starts
             for s, k, r in ((1, 1, 0), (7, 1, min(1, wl.n - 1)), (100, wl.g, wl.n - 1))]
    cases += [(max(0, j.index - 7), j.step, j.micro, j.rank) for j in wl.injections]
    count = 5008   # runs past psi at the second start: padding must be zero
    for begin, step, micro, rank in cases:
        scale = 1024.0 if wl.dtype == "fp16" else 1.0
        buf = torch.zeros(count, dtype=torch.int16, device="cuda")

        def writer(off, bits, buf=buf):
            buf[off] = bits - 65536 if bits >= 32768 else bits

        synth.dev_fill_grads(buf.data_ptr(), count, begin, wl, step, micro, rank, scale,
                             torch.cuda.current_stream().cuda_stream, inject=True,
                             inject_writer=writer)
        idx = np.arange(begin, begin + count, dtype=np.int64)
        want = synth.host_grad_bits(wl, idx, step, micro, rank, scale)
        got = buf.cpu().numpy().view(np.uint16)
        assert (got == want).all(), (name, begin, step, micro, rank)
    m = torch.zeros(count, dtype=torch.float32, device="cuda")
    begin = max(0, wl.psi - 3000)
    synth.dev_fill_master(m.data_ptr(), count, begin, wl, torch.cuda.current_stream().cuda_stream)
    want = synth.host_master(wl, np.arange(begin, begin + count, dtype=np.int64))
    assert m.cpu().numpy().tobytes() == want.tobytes()
