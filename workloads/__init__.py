"""Seeded synthetic inputs for the quantized GEMV / GEMM workloads.

This module is shared by the tests, the oracle checks and ``bench.py``.  It only
draws random numbers and stores them in the *logical* form of each weight format
(one code per byte, raw scale bytes, fp16 scale/bias values, bf16 activation
bits).  It holds none of the method's arithmetic: no dequantisation, no packing,
no dot products.  Encodings of drawn values into storage types (fp32 -> bf16,
fp32 -> E4M3, fp32 -> fp16) use PyTorch / numpy casts.

Recipe (every tensor of a workload comes from its own child stream of
``numpy.random.SeedSequence(seed).spawn(6)``, in this fixed order of purpose:
codes, scales, aux, x, residual, logits).  The value distributions follow the
workload definitions of the quantized-GEMV benchmark:

* MLX affine 4-bit, group 64: codes uniform in [0, 15]; per-64 fp16 scale
  s = fp16(0.02 * U(0.5, 1.5)); fp16 bias b = fp16(-8 * s).
* MXFP4: E2M1 codes uniform over the 16 bit patterns; per-32 E8M0 scale with
  exponent uniform in [-8, -4] (bytes 119..123).
* NVFP4: E2M1 codes uniform over 16; per-16 E4M3 scale = RN_E4M3(|N(0,1)| * 0.05);
  fp32 tensor scale 1/448.
* Q6_K-style: 6-bit codes uniform in [0, 63]; int8 scale per 16 uniform in
  [-64, 63]; fp16 super-scale d per 256 = fp16(|N(0,1)| * 1e-3).
* 5-bit formats (codes uniform in [0, 31], 32-weight blocks):
  Q5_0: fp16 d = fp16(0.02 * U(0.5, 1.5));
  Q5_1: the same d and fp16 m = fp16(-d * U(12, 20)) (a block minimum near -16 d);
  Q5_K: 6-bit sc and mn uniform in [0, 63] per block, fp16 d and dmin per 256 =
  fp16(|N(0,1)| * 1e-3) each.
* Activations and residuals: fp32 N(0,1) draws rounded to bf16 (round to
  nearest even).  Router logits: fp32 N(0,1).
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional

import numpy as np
import torch

# Format identifiers (same numbering as the C ABI enum).
MLX_AFFINE4_G64 = 1
MXFP4 = 2
NVFP4 = 3
Q6K = 4
Q5_0 = 5
Q5_1 = 6
Q5_K = 7

FORMAT_NAMES = {MLX_AFFINE4_G64: "mlx_affine4_g64", MXFP4: "mxfp4", NVFP4: "nvfp4", Q6K: "q6k", Q5_0: "q5_0",
                Q5_1: "q5_1", Q5_K: "q5_k"}
BLOCK = {MLX_AFFINE4_G64: 64, MXFP4: 32, NVFP4: 16, Q6K: 16, Q5_0: 32, Q5_1: 32, Q5_K: 32}
SUPER_BLOCK = {Q6K: 256, Q5_K: 256}

_STREAMS = ("codes", "scales", "aux", "x", "residual", "logits")


def streams(seed: int) -> dict:
    """One numpy Generator per purpose, spawned from ``seed`` in fixed order."""
    children = np.random.SeedSequence(seed).spawn(len(_STREAMS))
    return {name: np.random.default_rng(c) for name, c in zip(_STREAMS, children)}


def bf16_bits_from_f32(a: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (RNE, via torch) and return the uint16 bit patterns."""
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def e4m3_bytes_from_f32(a: np.ndarray) -> np.ndarray:
    """Round fp32 values to E4M3FN (RNE, saturating, via torch) and return the bytes."""
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.float8_e4m3fn)
    return t.view(torch.uint8).numpy().copy()


@dataclass
class QWeight:
    """A quantized N x K weight matrix in logical (unpacked) form.

    codes:  uint8 [N, K], one code per byte (4-bit formats: 0..15, Q6_K: 0..63,
            5-bit formats: 0..31).
    scales: MLX: float16 [N, K/64] scale s; MXFP4: uint8 [N, K/32] E8M0 bytes;
            NVFP4: uint8 [N, K/16] E4M3 bytes; Q6_K: int8 [N, K/16];
            Q5_0, Q5_1: float16 [N, K/32] d; Q5_K: uint8 [N, K/32, 2] (sc, mn).
    aux:    MLX: float16 [N, K/64] bias b; Q6_K: float16 [N, K/256] d;
            Q5_1: float16 [N, K/32] m; Q5_K: float16 [N, K/256, 2] (d, dmin);
            else None.
    tensor_scale: NVFP4 fp32 tensor scale (1.0 for the other formats).
    """

    fmt: int
    n: int
    k: int
    codes: np.ndarray
    scales: np.ndarray
    aux: Optional[np.ndarray] = None
    tensor_scale: float = 1.0
    meta: dict = field(default_factory=dict)


def _draw_weight(fmt: int, n: int, k: int, rs: dict) -> QWeight:
    if k % (SUPER_BLOCK.get(fmt, BLOCK[fmt])) != 0:
        raise ValueError(f"K={k} is not a multiple of the {FORMAT_NAMES[fmt]} block")
    if fmt == MLX_AFFINE4_G64:
        codes = rs["codes"].integers(0, 16, size=(n, k), dtype=np.uint8)
        s = (0.02 * rs["scales"].uniform(0.5, 1.5, size=(n, k // 64))).astype(np.float16)
        b = (-8.0 * s.astype(np.float32)).astype(np.float16)
        return QWeight(fmt, n, k, codes, s, b, 1.0)
    if fmt == MXFP4:
        codes = rs["codes"].integers(0, 16, size=(n, k), dtype=np.uint8)
        e = (127 + rs["scales"].integers(-8, -3, size=(n, k // 32))).astype(np.uint8)
        return QWeight(fmt, n, k, codes, e, None, 1.0)
    if fmt == NVFP4:
        codes = rs["codes"].integers(0, 16, size=(n, k), dtype=np.uint8)
        raw = np.abs(rs["scales"].standard_normal(size=(n, k // 16), dtype=np.float32)) * np.float32(0.05)
        return QWeight(fmt, n, k, codes, e4m3_bytes_from_f32(raw), None, float(np.float32(1.0 / 448.0)))
    if fmt == Q6K:
        codes = rs["codes"].integers(0, 64, size=(n, k), dtype=np.uint8)
        sc = rs["scales"].integers(-64, 64, size=(n, k // 16), dtype=np.int8)
        d = (np.abs(rs["aux"].standard_normal(size=(n, k // 256), dtype=np.float32)) * np.float32(1e-3)).astype(np.float16)
        return QWeight(fmt, n, k, codes, sc, d, 1.0)
    if fmt in (Q5_0, Q5_1):
        codes = rs["codes"].integers(0, 32, size=(n, k), dtype=np.uint8)
        d = (0.02 * rs["scales"].uniform(0.5, 1.5, size=(n, k // 32))).astype(np.float16)
        if fmt == Q5_0:
            return QWeight(fmt, n, k, codes, d, None, 1.0)
        m = (-d.astype(np.float64) * rs["aux"].uniform(12.0, 20.0, size=(n, k // 32))).astype(np.float16)
        return QWeight(fmt, n, k, codes, d, m, 1.0)
    if fmt == Q5_K:
        codes = rs["codes"].integers(0, 32, size=(n, k), dtype=np.uint8)
        sm = rs["scales"].integers(0, 64, size=(n, k // 32, 2), dtype=np.uint8)
        dd = (np.abs(rs["aux"].standard_normal(size=(n, k // 256, 2), dtype=np.float32)) * np.float32(1e-3)).astype(np.float16)
        return QWeight(fmt, n, k, codes, sm, dd, 1.0)
    raise ValueError(f"unknown format {fmt}")


def weight(fmt: int, n: int, k: int, seed: int = 0) -> QWeight:
    """One N x K weight of ``fmt`` drawn from ``seed``."""
    return _draw_weight(fmt, n, k, streams(seed))


def activations(m: int, k: int, seed: int = 0, stream: str = "x") -> np.ndarray:
    """bf16 bit patterns [m, k] of fp32 N(0,1) draws."""
    rs = streams(seed)[stream]
    return bf16_bits_from_f32(rs.standard_normal(size=(m, k), dtype=np.float32))


EDGE_KINDS = ("spread", "zero_next_to_huge", "subnormal", "near_max", "nonfinite")


def activations_edge(m: int, k: int, kind: str, seed: int = 0) -> np.ndarray:
    """bf16 bit patterns [m, k] of activations with the magnitude structure ``kind``, drawn
    as fp32 N(0,1) values times powers of two (exact in fp32), rounded to bf16 once:

    * "spread": inside every 16-input quarter the values take magnitudes 2^0, 2^-20, 2^-27
      and 2^-30 (a quarter's largest and smallest value are up to 2^30 apart); every fourth
      quarter also holds one value 2^20 times larger.
    * "zero_next_to_huge": quarters cycle through all zero, values near 2^100, and N(0,1).
    * "subnormal": row 0 only bf16 subnormals (|x| < 2^-126); the other rows subnormal
      quarters next to N(0,1) ones.
    * "near_max": N(0,1) values plus, per row, one value of magnitude 1.5 * 2^127 (bf16's
      largest finite numbers are just below 2^128).
    * "nonfinite": N(0,1) rows; row 1 (when present) holds one +inf, row 2 one NaN and row 3
      one -inf.
    """
    rs = streams(seed)["x"]
    v = rs.standard_normal(size=(m, k), dtype=np.float32)
    q = np.arange(k) // 16  # quarter index of each input
    if kind == "spread":
        e = rs.choice(np.array([0, -20, -27, -30]), size=(m, k))
        e[:, ::16] = 0  # every quarter keeps values at full magnitude
        v = v * np.exp2(e).astype(np.float32)
        big = (q % 4 == 1) & (np.arange(k) % 16 == 5)
        v[:, big] = v[:, big] * np.float32(2.0 ** 20)
    elif kind == "zero_next_to_huge":
        v[:, q % 3 == 0] = 0.0
        v[:, q % 3 == 1] *= np.float32(2.0 ** 100)
    elif kind == "subnormal":
        sub = np.full((m, k), True) if m == 1 else np.broadcast_to(q % 2 == 0, (m, k)).copy()
        sub[0] = True
        v = np.where(sub, v * np.float32(2.0 ** -130), v).astype(np.float32)
    elif kind == "near_max":
        j = rs.integers(0, k, size=m)
        v[np.arange(m), j] = np.sign(v[np.arange(m), j]) * np.float32(1.5 * 2.0 ** 127)
    elif kind == "nonfinite":
        for row, val in ((1, np.inf), (2, np.nan), (3, -np.inf)):
            if row < m:
                v[row, rs.integers(0, k)] = val
    else:
        raise ValueError(kind)
    return bf16_bits_from_f32(v)


def gemv_case(fmt: int, n: int, k: int, m: int, seed: int = 0, residual: bool = False):
    """(weight, x bits [m,k], residual bits [m,n] or None) for one GEMV workload."""
    rs = streams(seed)
    w = _draw_weight(fmt, n, k, rs)
    x = bf16_bits_from_f32(rs["x"].standard_normal(size=(m, k), dtype=np.float32))
    res = None
    if residual:
        res = bf16_bits_from_f32(rs["residual"].standard_normal(size=(m, n), dtype=np.float32))
    return w, x, res


@dataclass
class MoELayer:
    """A mixture-of-experts FFN layer in logical form.

    gate_up[e]: QWeight 2F x H (rows 0..F-1 gate, rows F..2F-1 up); down[e]: QWeight H x F.
    shared_gate_up / shared_down: the shared expert, same shapes, or None.
    """

    fmt: int
    n_experts: int
    hidden: int
    ffn: int
    gate_up: list
    down: list
    shared_gate_up: Optional[QWeight]
    shared_down: Optional[QWeight]


def moe_layer(fmt: int, n_experts: int, hidden: int, ffn: int, seed: int = 0, shared: bool = True) -> MoELayer:
    """All experts' weights from one seed: gate/up codes of every expert are drawn first,
    then down codes, then the shared expert (same order for scales and aux)."""
    rs = streams(seed)
    gu = [_draw_weight(fmt, 2 * ffn, hidden, rs) for _ in range(n_experts)]
    dn = [_draw_weight(fmt, hidden, ffn, rs) for _ in range(n_experts)]
    sgu = _draw_weight(fmt, 2 * ffn, hidden, rs) if shared else None
    sdn = _draw_weight(fmt, hidden, ffn, rs) if shared else None
    return MoELayer(fmt, n_experts, hidden, ffn, gu, dn, sgu, sdn)


def router_logits(t: int, n_experts: int, seed: int = 0, sets: int = 1) -> np.ndarray:
    """fp32 N(0,1) router logits, shape [sets, t, n_experts] (or [t, n_experts] if sets == 1)."""
    rs = streams(seed)["logits"]
    a = rs.standard_normal(size=(sets, t, n_experts), dtype=np.float32)
    return a[0] if sets == 1 else a


def shared_gate_logits(t: int, seed: int = 0) -> np.ndarray:
    """fp32 N(0, 2^2) gate logits [t] of the shared expert (one per token); the first is 0
    and, from four tokens on, the fourth is +30 (a saturated gate) when t allows."""
    a = (streams(seed)["logits"].standard_normal(size=t, dtype=np.float32) * np.float32(2.0)).astype(np.float32)
    if t > 0:
        a[0] = 0.0
    if t > 3:
        a[3] = 30.0
    return a


def moe_tokens(t: int, hidden: int, seed: int = 0) -> np.ndarray:
    """bf16 bits [t, hidden] of the MoE layer input."""
    return activations(t, hidden, seed, stream="x")


# Named workloads (sizes of the quantized-GEMV benchmark suite).
WORKLOADS = {
    "mlx_affine4_g64_5120x5120": dict(fmt=MLX_AFFINE4_G64, n=5120, k=5120, ms=(1,), residual=False),
    "nvfp4_gate_up_17408x5120": dict(fmt=NVFP4, n=17408, k=5120, ms=(1, 2, 3, 4), residual=False),
    "nvfp4_down_5120x17408": dict(fmt=NVFP4, n=5120, k=17408, ms=(1, 2, 3, 4), residual=True),
    "q6k_output_248320x5120": dict(fmt=Q6K, n=248320, k=5120, ms=(1, 2, 3, 4), residual=False),
    "q6k_5120x6144": dict(fmt=Q6K, n=5120, k=6144, ms=(1, 2, 3, 4), residual=False),
}
# The 5-bit GEMVs of the Q6_K operand PR's 5-bit commit (its q5k / q50 / q51 rows).
WORKLOADS_Q5 = {
    "q5_k_gate_up_17408x5120": dict(fmt=Q5_K, n=17408, k=5120, ms=(1, 2, 3, 4), residual=False),
    "q5_k_down_5120x17408": dict(fmt=Q5_K, n=5120, k=17408, ms=(1, 2, 3, 4), residual=True),
    "q5_k_out_5120x6144": dict(fmt=Q5_K, n=5120, k=6144, ms=(1, 2, 3, 4), residual=False),
    "q5_0_gate_up_17408x5120": dict(fmt=Q5_0, n=17408, k=5120, ms=(1, 2, 3, 4), residual=False),
    "q5_1_gate_up_17408x5120": dict(fmt=Q5_1, n=17408, k=5120, ms=(1, 2, 3, 4), residual=False),
}
MOE_DECODE = dict(fmt=MXFP4, n_experts=512, hidden=2048, ffn=512, topk=10, tokens=4, shared=True)
PREFILL = dict(fmt=NVFP4, n=17408, k=5120, tokens=8192, tile=128)
MOE_PREFILL = dict(fmt=MXFP4, n_experts=512, hidden=2048, ffn=512, topk=10, tokens=8192, shared=True)
