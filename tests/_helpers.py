"""Small helpers shared by the tests: half bit patterns from fp32 values (the
libraries' round to nearest even), device/host transfers of 16-bit patterns,
and distances in units in the last place between half bit patterns."""
import numpy as np
import torch

FP16, BF16 = 0, 1


def lib_half(x, dtype):
    """fp32 values -> half bit patterns, rounded by numpy (fp16) or torch (bf16)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    if dtype == FP16:
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
