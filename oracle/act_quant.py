"""NVFP4 activation quantisation and the W4A4 GEMM (oracle; test infrastructure only).

Source: TurboEXL3 article, §2.2 "NVFP4 with 4-bit and with 16-bit activations": the
W4A4 mode quantises the activations to NVFP4 too, during the forward pass, with one
scale per 16 values, so that both operands of the multiply are FP4 (W4A16, in
``oracle.gemv``, keeps them in 16 bits).  §2.1 gives NVFP4's structure: E2M1 values,
an E4M3 scale per block of 16, and one fp32 scale per tensor.

Readings where the pages are silent (each listed in the design notes):
* The activation tensor scale ``act_scale`` (fp32, finite, > 0) is an input of the call
  (a calibrated constant).  Each block of 16 consecutive values of a row along K gets the
  E4M3 scale S that maps the block's largest magnitude onto E2M1's largest, 6.
* Each step is one fp32 operation rounded to nearest even, in this order:
  d6 = fp32(6 * act_scale); r = fp32(amax / d6); S = the E4M3 value nearest r (ties to
  the even code, saturating at 448); den = fp32(E4M3(S) * act_scale);
  q = fp32(x / den), or x * 0 when den is 0; code = the E2M1 value nearest q (ties to
  the even code, saturating at 6), with x's sign bit (so -0 and tiny negatives give
  code 8).
* The quantised activation is act_scale * E4M3(S) * E2M1(code) (exact in fp64), and the
  W4A4 GEMM is the W4A16 definition with it in place of x:
  y[m, n] = RN_bf16( sum_k w[n, k] * xq[m, k]  (+ res[m, n]) ).
* Activations are finite; K is a multiple of 16 (whole blocks, as for NVFP4 weights).
"""
from __future__ import annotations

import numpy as np

from .formats import bf16_value, dequant_rows, e2m1_value, e4m3fn_value, round_to_bf16

_E2M1_GRID = e2m1_value(np.arange(8))      # 0, 0.5, 1, 1.5, 2, 3, 4, 6 (codes 0..7)
_E4M3_GRID = e4m3fn_value(np.arange(0x7F))  # the finite non-negative E4M3 values, codes 0..0x7E
_ROW_CHUNK = 4096


def _nearest_even_index(v, grid) -> np.ndarray:
    """Index of the value of the ascending `grid` nearest each |v|; of two equally near
    values the one with the even index.  Past the grid's end the last index (saturation)."""
    a = np.minimum(np.abs(np.asarray(v, dtype=np.float64)), grid[-1])  # saturate first: huge |v| are
    d = np.abs(a[..., None] - grid)                                     # not equidistant from the grid
    near = d == d.min(axis=-1, keepdims=True)
    even = near & (np.arange(grid.size) % 2 == 0)
    return np.where(even.any(axis=-1), np.argmax(even, axis=-1), np.argmax(near, axis=-1)).astype(np.uint8)


def e2m1_encode(q) -> np.ndarray:
    """E2M1 code (uint8, 0..15) of each fp32 value: the nearest of 0, 0.5, 1, 1.5, 2, 3,
    4, 6 to |q| (ties to the even code, saturating at 6), sign bit 3 from q's sign bit
    (TurboEXL3 article §2.1, the E2M1 magnitudes)."""
    q = np.asarray(q, dtype=np.float32)
    mag = _nearest_even_index(q, _E2M1_GRID)
    return (mag | (np.signbit(q).astype(np.uint8) << 3)).astype(np.uint8)


def e4m3_encode(r) -> np.ndarray:
    """E4M3FN byte of each non-negative fp32 value: the nearest finite E4M3 value (ties to
    the even code, saturating at 448).  TurboEXL3 article §2.1: NVFP4's block scale is E4M3."""
    r = np.asarray(r, dtype=np.float32)
    if np.any(r < 0) or not np.all(np.isfinite(r)):
        raise ValueError("block scales are encoded from finite non-negative values")
    return _nearest_even_index(r, _E4M3_GRID)


def quantize_act_nvfp4(x_bits, act_scale: float):
    """Quantise bf16 activations [M, K] to NVFP4 (TurboEXL3 article §2.2, W4A4: one scale
    per 16 values) in the steps of the module docstring.

    Returns (codes uint8 [M, K] one E2M1 code per value, scales uint8 [M, K/16] E4M3
    bytes, xe fp64 [M, K] = E4M3(S) * E2M1(code), xq fp64 [M, K] = act_scale * xe)."""
    x32 = bf16_value(x_bits).astype(np.float32)
    m, k = x32.shape
    if k % 16:
        raise ValueError("K must be a multiple of 16")
    a = np.float32(act_scale)
    if not (np.isfinite(a) and a > 0):
        raise ValueError("act_scale must be finite and positive")
    codes = np.empty((m, k), dtype=np.uint8)
    scales = np.empty((m, k // 16), dtype=np.uint8)
    xe = np.empty((m, k), dtype=np.float64)
    d6 = np.float32(np.float32(6.0) * a)
    for i in range(m):  # one row at a time keeps the nearest-value search small
        blk = x32[i].reshape(k // 16, 16)
        amax = np.abs(blk).max(axis=1)
        r = (amax / d6).astype(np.float32)
        s = e4m3_encode(r)
        sf = e4m3fn_value(s).astype(np.float32)
        den = (sf * a).astype(np.float32)
        with np.errstate(divide="ignore", invalid="ignore"):
            q = np.where(den[:, None] > 0, blk / den[:, None], blk * np.float32(0.0)).astype(np.float32)
        c = e2m1_encode(q)
        codes[i] = c.reshape(k)
        scales[i] = s
        xe[i] = (sf.astype(np.float64)[:, None] * e2m1_value(c)).reshape(k)
    return codes, scales, xe, float(a) * xe


def gemm_w4a4(w, x_bits, act_scale: float, res_bits=None, rows=None):
    """W4A4 GEMM (TurboEXL3 article §2.2): y[m, n] = RN_bf16( sum_k w[n, k] * xq[m, k]
    (+ res[m, n]) ) with w the fp32 dequantised weight (as in ``oracle.gemv``), xq the
    NVFP4-quantised activation, the sum in fp64 and one bf16 rounding.

    Returns (y, v, xq): bf16-exact outputs and fp64 pre-rounding sums [M, len(rows)], and
    the quantised activations."""
    rows = np.arange(w.n) if rows is None else np.asarray(rows, dtype=np.int64)
    xq = quantize_act_nvfp4(x_bits, act_scale)[3]
    v = np.empty((xq.shape[0], rows.size), dtype=np.float64)
    for i in range(0, rows.size, _ROW_CHUNK):
        r = rows[i:i + _ROW_CHUNK]
        v[:, i:i + r.size] = xq @ dequant_rows(w, r).astype(np.float64).T
    if res_bits is not None:
        v = v + bf16_value(np.asarray(res_bits)[:, rows])
    return round_to_bf16(v), v, xq
