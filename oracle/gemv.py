"""Reference GEMV / GEMM (oracle; test infrastructure only).

Definition followed (TurboEXL3 article §2.2: W4A16 expands each weight and
multiplies with 16-bit activations; §4.4: 32-bit accumulation, one rounding
where the reference rounds):

    y[m, n] = RN_bf16( sum_k w[n, k] * x[m, k]  (+ res[m, n]) )

with w the fp32 dequantised weight (one rounding of its exact value), x the bf16
activation, the sum taken in fp64 and the bf16 rounding applied once.  The same
definition serves the M = 1..4 GEMV and the prefill GEMM at any token count.
"""
from __future__ import annotations

import numpy as np

from .formats import bf16_value, dequant_rows, round_to_bf16

_ROW_CHUNK = 4096


def _accumulate(wrows_f32: np.ndarray, x64: np.ndarray) -> np.ndarray:
    return x64 @ wrows_f32.astype(np.float64).T  # [M, rows], fp64


def gemv_rows(w, x_bits, rows, res_bits=None):
    """Outputs of the selected rows only.

    Returns (y, v): y = bf16-exact fp64 values [M, len(rows)], v = the fp64
    pre-rounding sums (residual included)."""
    rows = np.asarray(rows, dtype=np.int64)
    x64 = bf16_value(x_bits)
    v = np.empty((x64.shape[0], rows.size), dtype=np.float64)
    for i in range(0, rows.size, _ROW_CHUNK):
        r = rows[i:i + _ROW_CHUNK]
        v[:, i:i + r.size] = _accumulate(dequant_rows(w, r), x64)
    if res_bits is not None:
        v += bf16_value(np.asarray(res_bits)[:, rows])
    return round_to_bf16(v), v


def gemv(w, x_bits, res_bits=None):
    """All N outputs: (y, v) as in ``gemv_rows``; y has shape [M, N]."""
    return gemv_rows(w, x_bits, np.arange(w.n), res_bits)


def row_norms(w, rows=None) -> np.ndarray:
    """||w_n||_2 of the fp32 dequantised rows (all rows, or the selected ones)."""
    rows = np.arange(w.n) if rows is None else np.asarray(rows, dtype=np.int64)
    out = np.empty(rows.size, dtype=np.float64)
    for i in range(0, rows.size, _ROW_CHUNK):
        r = rows[i:i + _ROW_CHUNK]
        out[i:i + r.size] = np.linalg.norm(dequant_rows(w, r).astype(np.float64), axis=1)
    return out


def tolerance(w, x_bits, res_bits=None, rows=None, max_row_norm=None, ref=None) -> np.ndarray:
    """Per-element error bound [M, len(rows)] for a GEMV / GEMM output.

    Base bound (the stated contract): 2e-3 * ||x_m||_2 * max_n ||w_n||_2 on the value
    before the output's single bf16 rounding.  After that rounding the two sides may
    land on neighbouring bf16 numbers when the exact value is near a rounding boundary,
    so one bf16 ulp of the output is added: max(2**-7 * |ref|, 2**-133) (an upper bound on
    the spacing next to ref; below bf16's smallest normal number, 2**-126, the spacing is
    the subnormal quantum 2**-133) when the reference outputs `ref` are given.  Without
    `ref`, with a residual, 2**-7 * |res| stands in for it (the residual dominates the
    magnitude)."""
    x64 = bf16_value(x_bits)
    xn = np.linalg.norm(x64, axis=1)
    wmax = float(np.max(row_norms(w))) if max_row_norm is None else float(max_row_norm)
    ncols = w.n if rows is None else len(rows)
    tol = np.repeat((2e-3 * xn * wmax)[:, None], ncols, axis=1)
    if ref is not None:
        tol = tol + np.maximum(2.0 ** -7 * np.abs(np.asarray(ref, dtype=np.float64)), 2.0 ** -133)
    elif res_bits is not None:
        r = bf16_value(res_bits) if rows is None else bf16_value(np.asarray(res_bits)[:, rows])
        tol = tol + 2.0 ** -7 * np.abs(r)
    return tol
