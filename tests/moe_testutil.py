"""Helpers shared by the tests: host<->device conversion of bf16 bit
patterns and ulp distances.  No path arithmetic lives here."""
import numpy as np


def to_dev(a, device="cuda"):
    import torch
    if a.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(device)
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def to_host(t):
    import torch
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


def bf16_ordinal(bits):
    """Map bf16 bit patterns to integers whose differences count ulps
    (+0 and -0 both map to 0)."""
    b = np.asarray(bits, np.uint16).astype(np.int64)
    mag = b & 0x7FFF
    return np.where(b & 0x8000, -mag, mag)


def bf16_ulp_diff(a, b):
    return np.abs(bf16_ordinal(a) - bf16_ordinal(b))


def f32_ordinal(v):
    u = np.asarray(v, np.float32).view(np.int32).astype(np.int64)
    mag = u & 0x7FFFFFFF
    return np.where(u < 0, -mag, mag)


def f32_ulp_diff(a, b):
    return np.abs(f32_ordinal(a) - f32_ordinal(b))


def bf16_ulp_of(x64):
    """Size of one bf16 ulp at each value of a float64 array."""
    ax = np.maximum(np.abs(np.asarray(x64, np.float64)), 2.0 ** -126)
    return np.exp2(np.floor(np.log2(ax)) - 7)


def within_one_bf16_ulp(got, ref64):
    return np.abs(np.asarray(got, np.float64) - ref64) <= bf16_ulp_of(ref64)
