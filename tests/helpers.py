"""Host/device marshalling shared by the GPU tests (no arithmetic of the layer)."""
import numpy as np
import torch

import moe_inputs as mi


def dev(a, dtype=None):
    """numpy -> CUDA tensor; uint16 arrays become bf16, the rest keep their type."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).cuda().view(torch.bfloat16)
    t = torch.from_numpy(a).cuda()
    return t if dtype is None else t.view(dtype)


def host_bits(t):
    """bf16 CUDA tensor -> uint16 numpy bits."""
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def host(t):
    return t.contiguous().cpu().numpy()


def layer_tolerance(got_bits, ref_bits):
    """The layer-output bar: max|err| <= 2e-2 * max|ref| and sum|err| / sum|ref| <= 5e-3,
    no NaN/Inf. Returns (max_err_ratio, l1_ratio)."""
    g = mi.bf16_to_f32(got_bits).astype(np.float64)
    r = mi.bf16_to_f32(ref_bits).astype(np.float64)
    assert np.isfinite(g).all(), "non-finite output"
    err = np.abs(g - r)
    mx = err.max() / max(np.abs(r).max(), 1e-30)
    l1 = err.sum() / max(np.abs(r).sum(), 1e-30)
    assert mx <= 2e-2, f"max abs err ratio {mx:.3g} > 2e-2"
    assert l1 <= 5e-3, f"normalised L1 err {l1:.3g} > 5e-3"
    return mx, l1


def e4m3_ulp_diff(a, b):
    """Distance in representable steps between two arrays of e4m3 codes (same sign)."""
    def ordinal(c):
        c = c.astype(np.int32)
        mag = c & 0x7F
        return np.where(c & 0x80, -mag, mag)
    return np.abs(ordinal(a) - ordinal(b))
