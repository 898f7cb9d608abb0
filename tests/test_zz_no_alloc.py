"""The allocation-free norm entry point, zs_grad_sumsq_noalloc.

It serves callers that cannot call cudaMalloc: a framework that owns all
device memory through its own planner or arena, an out-of-memory handler
that still needs the gradient norm, or code that cannot create a context
(creating one allocates).  Its scratch is a fixed static device array.

Checked through the C ABI against the oracle's squared norm of the same final
sums (and against zs_grad_sumsq) on two calls in a row, the second smaller
than the first so that stale partial sums left in the shared array would
show; that device memory stays put across further calls once the first call
has done its set-up; and that a count past the array's capacity is refused.
Collected last so that a failure here never hides the other tests; it also
passes when run alone in a fresh process."""
import numpy as np
import pytest
import torch
from _helpers import dev16, lib_half

import oracle

pytestmark = pytest.mark.gpu

FP16, BF16 = 0, 1
REL = 1e-6


def oracle_sumsq(acc0, slices, dtype, div):
    """The oracle's squared norm of the final sums: acc (or +0) then every
    slice added in rank order in fp32, each sum divided by div, squared, summed."""
    final = np.zeros(slices[0].shape[0] if acc0 is None else acc0.shape[0], np.float32)
    if acc0 is not None:
        final[:] = acc0
    if slices:
        oracle.reduce_accumulate(slices, dtype, final, first=acc0 is None)
    return oracle.grad_sumsq(final, div)


@pytest.mark.parametrize("dtype", [FP16, BF16])
def test_noalloc_sumsq_matches_oracle_twice(dtype):
    import zero_mixed_precision_shard_gb300 as zs
    torch.cuda.set_device(0)
    ctx = zs.Ctx()
    rng = np.random.default_rng(31)
    n, div = 3, 3 * 2 * 1024.0
    for count in (1_000_003, 50_001):  # two calls in a row, the second smaller
        acc0 = (rng.standard_normal(count) * 0.3 * div).astype(np.float32)
        sl = [lib_half((rng.standard_normal(count) * 0.2 * 1024).astype(np.float32), dtype)
              for _ in range(n)]
        acc = torch.from_numpy(acc0).cuda()
        grads = [dev16(s) for s in sl]
        for form_grads, form_acc, a0, s in ((grads, acc, acc0, sl), (None, acc, acc0, []),
                                            (grads, None, None, sl)):
            want = oracle_sumsq(a0, s, dtype, div)
            got = torch.full((1,), -1.0, dtype=torch.float64, device="cuda")
            zs.zs_grad_sumsq_noalloc(form_grads, dtype, form_acc, count, div, got)
            g = got.item()
            assert want > 0 and abs(g - want) <= REL * want, (count, g, want)
            # and the context form gives the same value (same kernels, other scratch)
            ref = torch.zeros(1, dtype=torch.float64, device="cuda")
            zs.zs_grad_sumsq(ctx, form_grads, dtype, form_acc, count, div, ref)
            assert abs(ref.item() - g) <= REL * want
    ctx.close()


def test_noalloc_calls_leave_device_memory_unchanged():
    import zero_mixed_precision_shard_gb300 as zs
    torch.cuda.set_device(0)
    rng = np.random.default_rng(5)
    count, div = 300_017, 2048.0
    acc = torch.from_numpy((rng.standard_normal(count) * div).astype(np.float32)).cuda()
    grads = [dev16(lib_half(rng.standard_normal(count).astype(np.float32), d)) for d in (0, 0)]
    out = torch.zeros(1, dtype=torch.float64, device="cuda")
    zs.zs_grad_sumsq_noalloc(None, FP16, acc, 0, div, out)     # start-up call: the set-up
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    for dtype in (FP16, BF16):
        for g, a in ((grads, acc), (None, acc), (grads, None)):
            for _ in range(3):
                zs.zs_grad_sumsq_noalloc(g, dtype, a, count, div, out)
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0


def test_noalloc_rejects_counts_beyond_its_scratch():
    import zero_mixed_precision_shard_gb300 as zs
    torch.cuda.set_device(0)
    acc = torch.zeros(16, dtype=torch.float32, device="cuda")
    out = torch.zeros(1, dtype=torch.float64, device="cuda")
    # rejected before any work: nothing beyond these 16 elements is touched
    rc = zs.lib.zs_grad_sumsq_noalloc(None, 0, FP16, acc.data_ptr(), zs.ZS_NOALLOC_MAX_COUNT + 1,
                                      1.0, out.data_ptr(), None)
    assert rc == zs.ZS_ERR_LIMIT
    zs.zs_grad_sumsq_noalloc(None, FP16, acc, 16, 1.0, out)
    assert out.item() == 0.0
