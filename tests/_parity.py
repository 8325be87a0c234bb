"""Helpers shared by the GPU parity tests (comparison metric, canaries)."""

from __future__ import annotations

import numpy as np
import torch

# Tolerances of the comparison against the float64 oracle: float32 io with
# float32 arithmetic, and bf16 io with float32 accumulation.
TOL_F32 = 1e-5
TOL_BF16 = 2e-2


def rel_err(gpu: np.ndarray, ref: np.ndarray, slice_axes: int = 2) -> float:
    """max over (b, h) slices of ||gpu - ref||_inf / ||ref||_inf (reading R12)."""
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    assert gpu.shape == ref.shape, (gpu.shape, ref.shape)
    lead = int(np.prod(gpu.shape[:slice_axes]))
    g = gpu.reshape(lead, -1)
    r = ref.reshape(lead, -1)
    den = np.maximum(np.abs(r).max(axis=1), 1e-30)
    return float((np.abs(g - r).max(axis=1) / den).max())


class Guarded:
    """A CUDA buffer with canary bands on both sides of the usable view."""

    BAND = 4096  # bytes on each side

    def __init__(self, shape, dtype, device="cuda", fill=None):
        n = int(np.prod(shape)) if len(shape) else 1
        esz = torch.empty(0, dtype=dtype).element_size()
        band = self.BAND // esz
        self.raw = torch.empty(n + 2 * band, dtype=dtype, device=device)
        self.raw.view(torch.uint8).fill_(0xA5)
        self.band = band
        self.view = self.raw[band:band + n].view(shape)
        if fill is not None:
            self.view.copy_(fill)

    def intact(self) -> bool:
        b = self.band
        pat = torch.full((b * self.raw.element_size(),), 0xA5, dtype=torch.uint8, device=self.raw.device)
        lo = self.raw[:b].contiguous().view(torch.uint8)
        hi = self.raw[-b:].contiguous().view(torch.uint8)
        return bool(torch.equal(lo, pat) and torch.equal(hi, pat))
