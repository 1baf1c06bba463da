"""Helpers shared by the GPU parity tests."""
import numpy as np
import torch


def rel_err(gpu, ref):
    """max_i |g_i - r_i| / max(|r_i|, rms(r)) — relative error per element,
    with elements near zero measured against the vector's RMS."""
    g = np.asarray(gpu, dtype=np.float64).ravel()
    r = np.asarray(ref, dtype=np.float64).ravel()
    assert g.shape == r.shape
    rms = np.sqrt(np.mean(r * r)) if r.size else 0.0
    den = np.maximum(np.abs(r), rms if rms > 0 else 1e-30)
    return float(np.max(np.abs(g - r) / den)) if r.size else 0.0


def host(t):
    """Device tensor -> numpy: float32 values or uint16 bf16 bits."""
    t = t.detach().contiguous().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16).copy()
    return t.numpy().copy()


def top2_gap(logits):
    s = np.sort(np.asarray(logits, dtype=np.float64).ravel())
    return float(s[-1] - s[-2])


FP32_TOL = 1e-4   # fp32 paths: max relative error
BF16_TOL = 2e-2   # bf16-weight paths: relative error on logits
TIE_GAP = 1e-3    # ids must match wherever the oracle's top-2 gap exceeds this
