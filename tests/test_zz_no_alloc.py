"""The allocation-free norm entry point, zs_grad_sumsq_noalloc.

It serves callers that cannot call cudaMalloc (a framework that owns all
device memory through its own planner or arena, an out-of-memory handler, or
code that cannot create a context, since creating one allocates), so its
scratch lives in a fixed static device array.  Checked through the C ABI
against zs_grad_sumsq on two calls in a row (the second smaller than the
first, so stale partial sums in the shared array would show), and against
its size limit.  Collected last so that a failure here never hides the other
tests; it also passes when run alone in a fresh process."""
import numpy as np
import pytest
import torch
from _helpers import dev16, lib_half

pytestmark = pytest.mark.gpu

FP16, BF16 = 0, 1
REL = 1e-6


@pytest.mark.parametrize("dtype", [FP16, BF16])
def test_noalloc_sumsq_matches_context_version_twice(dtype):
    import zero_mixed_precision_shard_gb300 as zs
    torch.cuda.set_device(0)
    ctx = zs.Ctx()
    rng = np.random.default_rng(31)
    n, div = 3, 3 * 2 * 1024.0
    for count in (1_000_003, 50_001):  # two calls in a row, the second smaller
        acc = torch.from_numpy((rng.standard_normal(count) * 0.3 * div).astype(np.float32)).cuda()
        grads = [dev16(lib_half((rng.standard_normal(count) * 0.2 * 1024).astype(np.float32),
                                dtype)) for _ in range(n)]
        want = torch.zeros(1, dtype=torch.float64, device="cuda")
        zs.zs_grad_sumsq(ctx, grads, dtype, acc, count, div, want)
        got = torch.full((1,), -1.0, dtype=torch.float64, device="cuda")
        zs.zs_grad_sumsq_noalloc(grads, dtype, acc, count, div, got)
        w, g = want.item(), got.item()
        assert w > 0 and abs(g - w) <= REL * w, (count, g, w)
        # accumulator-only form too
        zs.zs_grad_sumsq(ctx, None, dtype, acc, count, div, want)
        zs.zs_grad_sumsq_noalloc(None, dtype, acc, count, div, got)
        assert abs(got.item() - want.item()) <= REL * want.item()
    ctx.close()


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
