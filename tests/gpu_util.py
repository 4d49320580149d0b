"""Helpers for the GPU parity tests: build/load the library, move logical inputs to the device."""
from __future__ import annotations

import numpy as np
import torch

_built = False


def qlib():
    """Build (if stale) and load the C library; returns the binding module."""
    global _built
    import prefill_dequant_gemv_gb300 as q
    from prefill_dequant_gemv_gb300 import build as b
    if not _built:
        b.build()
        _built = True
    q.lib()
    return q


def dev_bf16(bits: np.ndarray, device="cuda"):
    """bf16 bit patterns [r, c] -> device bf16 tensor view [r, c] whose row stride is a multiple of 8."""
    r, c = bits.shape
    cp = (c + 7) // 8 * 8
    host = np.zeros((r, cp), dtype=np.uint16)
    host[:, :c] = bits
    t = torch.from_numpy(host.view(np.int16)).view(torch.bfloat16).to(device)
    return t[:, :c]


def to_f64(t) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)
