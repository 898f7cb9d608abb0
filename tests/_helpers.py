"""Small helpers shared by the tests: half bit patterns from fp32 values (the
libraries' round to nearest even), device/host transfers of 16-bit patterns,
and distances in units in the last place between half bit patterns."""
import numpy as np
import torch

FP16, BF16 = 0, 1


def lib_half(x, dtype):
    """fp32 values -> half bit patterns, rounded by numpy (fp16) or torch (bf16);
    values past the format's range round to infinity, as IEEE rounding does."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    if dtype == FP16:
        with np.errstate(over="ignore"):
            return x.astype(np.float16).view(np.uint16)
    return torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def dev16(bits):
    """uint16 patterns -> an int16 tensor on the current CUDA device."""
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda()


def host16(t):
    """An int16 tensor -> its uint16 patterns on the host."""
    return t.cpu().numpy().view(np.uint16)


def half_ulps(a, b):
    """Distance in units in the last place between two half bit-pattern arrays."""
    def ordered(x):
        x = x.astype(np.int32)
        return np.where(x & 0x8000, -(x & 0x7FFF), x & 0x7FFF)
    return np.abs(ordered(a) - ordered(b))


ulps = half_ulps

# The parity bar for the fp32 state after at most 10 steps: 1e-6 relative plus
# 1e-9 absolute, the same at every learning rate.  The stress tests run at the
# highest learning rate of the workloads (the 1.3B decoder's 3e-4).
REL, ABS = 1e-6, 1e-9
STRESS_LR = 3e-4


def tol_ratio(got, want):
    """Worst |got - want| over the bound (1.0 = at the bound), over finite want."""
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    f = np.isfinite(want)
    err = np.abs(got[f] - want[f])
    tol = REL * np.abs(want[f]) + ABS
    return float((err / tol).max()) if err.size else 0.0


def assert_close(got, want, name):
    r = tol_ratio(got, want)
    assert r <= 1.0, f"{name}: worst error {r:.3g}x the bound (1e-6 rel + 1e-9 abs)"


def assert_half_close(got_half, got_master, want_half, want_master, dtype, name="half"):
    """The half copy is the round-to-nearest-even of the library's own fp32
    master, every element; and within 1 ulp of the oracle's half copy wherever
    the oracle's master is at least 1e-6 in magnitude.  Below that the master's
    1e-9 absolute bound spans more than a bf16 ulp (bf16 keeps fp32's exponent
    range), so two masters within the bar may round 2 ulps apart there."""
    got_half = np.asarray(got_half).view(np.uint16)
    assert (got_half == lib_half(np.asarray(got_master, np.float32), dtype)).all(), name
    u = half_ulps(got_half, want_half)
    big = np.abs(np.asarray(want_master)) >= 1e-6
    assert u[big].max(initial=0) <= 1, name
