"""Shared helpers of the GPU parity tests (no arithmetic of the method)."""

import numpy as np


def u16(t):
    """Device int16/bfloat16 tensor -> host numpy uint16 bit patterns."""
    import torch
    if t.dtype == torch.bfloat16:
        t = t.view(torch.int16)
    return t.detach().cpu().numpy().view(np.uint16)


def rel_fro(a, b):
    den = np.linalg.norm(b)
    if den == 0.0:
        return float(np.linalg.norm(a))
    return float(np.linalg.norm(a - b) / den)


def ulp_close(gpu32, ref32, ulps=1):
    """|gpu - ref| <= ulps * spacing(|ref|) elementwise (FP32)."""
    gpu32 = np.asarray(gpu32, dtype=np.float32)
    ref32 = np.asarray(ref32, dtype=np.float32)
    tol = ulps * np.spacing(np.abs(ref32)).astype(np.float64)
    return np.abs(gpu32.astype(np.float64) - ref32.astype(np.float64)) <= tol


def to_wide(x):
    """Transpose the last two axes when the matrix is tall."""
    return np.swapaxes(x, -1, -2) if x.shape[-2] > x.shape[-1] else x
