"""Element decoders and the one-rounding dequantiser (oracle; test infrastructure only).

Sources:
* TurboEXL3 article, §2.1 "Block-scaled 4-bit formats": a block-scaled format
  stores each weight as a 4-bit code with one shared scale per block;
  dequantising is one multiply, plus one add for affine formats.  MLX affine
  4-bit: 16-bit scale and 16-bit bias per 64 weights (4.5 bpw).  MXFP4: E2M1
  values with an E8M0 power-of-two scale per 32 (4.25 bpw); the E2M1
  magnitudes are 0, 0.5, 1, 1.5, 2, 3, 4, 6, each with a sign.  NVFP4: E2M1
  with an E4M3 scale per 16 plus one fp32 scale per tensor (4.5 bpw).
* Q6_K operand PR, "What changed": 6-bit codes with zero point 32, a scale per
  16 weights, and the half-precision operand 1 + code/64 whose value minus 1.5
  is exactly (code - 32)/64.
* Q6_K operand PR, commit "5-bit nibble operand": the 5-bit formats Q5_K, Q5_1
  and Q5_0 (the last taken "as ZeroAsMin": its zero point as a block minimum);
  the five-bit operand is the nibble with the fifth bit at bit 8 of the
  halfword, the half 1 + code/64, exact for codes up to 31.

Readings where the pages are silent (each listed in the design notes):
* E2M1 bit layout: bit 3 sign, bits 2..1 exponent with bias 1, bit 0 mantissa;
  exponent 0 is subnormal (0 or 0.5).
* E8M0: value 2**(E - 127); E = 255 is NaN.
* E4M3 is the FN variant: bias 7, no infinities, 0x7F / 0xFF are NaN,
  subnormals kept, largest finite 448.
* MLX scale and bias are fp16 and w = s * code + b.
* Q6_K: w = d * sc * (code - 32) with fp16 d per 256 weights and int8 sc per 16.
* NVFP4: w = RN_fp32(tensor_scale * (E4M3(S) * E2M1(code))), the tensor scale last.
* The 5-bit formats, which the PR names but does not define, follow the public
  GGML block definitions: codes 0..31 and 32-weight blocks;
  Q5_0: w = d * (code - 16), fp16 d per block (5.5 bpw);
  Q5_1: w = d * code + m, fp16 d and fp16 m per block (6 bpw);
  Q5_K: w = (d * sc) * code - dmin * mn, a 6-bit scale sc and 6-bit minimum mn per
  32-weight block and fp16 d, dmin per 256 (5 + 12/32 + 32/256 = 5.5 bpw).
"""
from __future__ import annotations

import numpy as np

MLX_AFFINE4_G64, MXFP4, NVFP4, Q6K, Q5_0, Q5_1, Q5_K = 1, 2, 3, 4, 5, 6, 7
BLOCK = {MLX_AFFINE4_G64: 64, MXFP4: 32, NVFP4: 16, Q6K: 16, Q5_0: 32, Q5_1: 32, Q5_K: 32}


# ---------------------------------------------------------------- element decoders
def e2m1_value(code) -> np.ndarray:
    """fp64 value of 4-bit E2M1 codes (TurboEXL3 article §2.1: magnitudes
    0, 0.5, 1, 1.5, 2, 3, 4, 6 with a sign)."""
    c = np.asarray(code).astype(np.int64) & 0xF
    sign = (c >> 3) & 1
    exp = (c >> 1) & 3
    man = c & 1
    mag = np.where(exp == 0, 0.5 * man, np.ldexp(1.0 + 0.5 * man, exp - 1))
    return np.where(sign == 1, -mag, mag)


def e8m0_value(byte) -> np.ndarray:
    """fp64 value of E8M0 scale bytes: 2**(E-127), NaN for 0xFF (TurboEXL3 article
    §2.1: an 8-bit power-of-two scale)."""
    e = np.asarray(byte).astype(np.int64) & 0xFF
    v = np.ldexp(1.0, e - 127)
    return np.where(e == 255, np.nan, v)


def e4m3fn_value(byte) -> np.ndarray:
    """fp64 value of E4M3FN bytes (TurboEXL3 article §2.1: an 8-bit floating-point
    block scale; the FN variant, largest finite 448)."""
    b = np.asarray(byte).astype(np.int64) & 0xFF
    sign = (b >> 7) & 1
    exp = (b >> 3) & 0xF
    man = b & 7
    mag = np.where(exp == 0, np.ldexp(man / 8.0, -6), np.ldexp(1.0 + man / 8.0, exp - 7))
    mag = np.where((exp == 15) & (man == 7), np.nan, mag)
    return np.where(sign == 1, -mag, mag)


def bf16_value(bits) -> np.ndarray:
    """fp64 value of bf16 bit patterns (the top half of an fp32)."""
    u = np.asarray(bits).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32).astype(np.float64)


def round_to_bf16(v) -> np.ndarray:
    """Round fp64 values to the nearest bf16 value, ties to even, in one step
    (no intermediate fp32 rounding).  Returns fp64 values that are bf16-exact;
    magnitudes that round past the largest finite bf16 become +-inf."""
    v = np.asarray(v, dtype=np.float64)
    out = v.copy()
    fin = np.isfinite(v) & (v != 0)
    x = v[fin]
    _, e = np.frexp(x)  # x = m * 2**e with 0.5 <= |m| < 1
    q = np.maximum(e - 8, -133)  # 8 significant bits; subnormal quantum 2**-133
    r = np.ldexp(np.round(np.ldexp(x, -q)), q)  # np.round: half to even
    r = np.where(np.abs(r) >= 2.0 ** 128, np.copysign(np.inf, r), r)
    out[fin] = r
    return out


def bf16_bits_of(v) -> np.ndarray:
    """uint16 bit patterns of fp64 values that are already bf16-exact."""
    f = np.asarray(v, dtype=np.float64).astype(np.float32)
    return (f.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


# ---------------------------------------------------------------- dequantisation
def _exact_values(fmt: int, codes, scales, aux, tensor_scale: float) -> np.ndarray:
    """Exact real value of every weight (fp64 holds it exactly for all four formats)."""
    codes = np.asarray(codes)
    n, k = codes.shape
    blk = BLOCK[fmt]
    if fmt == MLX_AFFINE4_G64:
        s = np.repeat(np.asarray(scales, dtype=np.float16).astype(np.float64), blk, axis=1)
        b = np.repeat(np.asarray(aux, dtype=np.float16).astype(np.float64), blk, axis=1)
        return s * codes.astype(np.float64) + b
    if fmt == MXFP4:
        s = np.repeat(e8m0_value(scales), blk, axis=1)
        return e2m1_value(codes) * s
    if fmt == NVFP4:
        s = np.repeat(e4m3fn_value(scales), blk, axis=1)
        ts = float(np.float32(tensor_scale))
        return ts * (s * e2m1_value(codes))
    if fmt == Q6K:
        sc = np.repeat(np.asarray(scales, dtype=np.int8).astype(np.float64), blk, axis=1)
        d = np.repeat(np.asarray(aux, dtype=np.float16).astype(np.float64), 256, axis=1)
        return d * sc * (codes.astype(np.float64) - 32.0)
    if fmt == Q5_0:
        d = np.repeat(np.asarray(scales, dtype=np.float16).astype(np.float64), blk, axis=1)
        return d * (codes.astype(np.float64) - 16.0)
    if fmt == Q5_1:
        d = np.repeat(np.asarray(scales, dtype=np.float16).astype(np.float64), blk, axis=1)
        m = np.repeat(np.asarray(aux, dtype=np.float16).astype(np.float64), blk, axis=1)
        return d * codes.astype(np.float64) + m
    if fmt == Q5_K:
        sm = np.asarray(scales, dtype=np.uint8).astype(np.float64)  # [N, K/32, 2]: (sc, mn)
        dd = np.asarray(aux, dtype=np.float16).astype(np.float64)   # [N, K/256, 2]: (d, dmin)
        sc = np.repeat(sm[:, :, 0], blk, axis=1)
        mn = np.repeat(sm[:, :, 1], blk, axis=1)
        d = np.repeat(dd[:, :, 0], 256, axis=1)
        dmin = np.repeat(dd[:, :, 1], 256, axis=1)
        return d * sc * codes.astype(np.float64) - dmin * mn
    raise ValueError(f"unknown format {fmt}")


def dequant(w) -> np.ndarray:
    """fp32 [N, K] dequantised weights of a logical QWeight, each the exact value
    rounded once to fp32 (TurboEXL3 article §2.1; Q6_K operand PR "What changed")."""
    return _exact_values(w.fmt, w.codes, w.scales, w.aux, w.tensor_scale).astype(np.float32)


def dequant_rows(w, rows) -> np.ndarray:
    """fp32 dequantised weights of the selected rows only."""
    rows = np.asarray(rows, dtype=np.int64)
    aux = None if w.aux is None else np.asarray(w.aux)[rows]
    return _exact_values(w.fmt, np.asarray(w.codes)[rows], np.asarray(w.scales)[rows], aux,
                         w.tensor_scale).astype(np.float32)


def dequant_operand_bf16(w) -> np.ndarray:
    """bf16-exact fp64 values [N, K] of the 16-bit operand a prefill GEMM multiplies
    (TurboEXL3 article §2.2: W4A16 expands each weight to 16 bits).  MXFP4 and NVFP4:
    the E2M1 value times its block scale, without the NVFP4 tensor scale (exact in
    bf16: at most 6 significant bits); MLX affine, Q6_K and the 5-bit formats: the fp32
    weight rounded to bf16 (a second rounding, since these weights carry up to 24
    bits)."""
    if w.fmt == MXFP4:
        v = e2m1_value(w.codes) * np.repeat(e8m0_value(w.scales), BLOCK[MXFP4], axis=1)
    elif w.fmt == NVFP4:
        v = e2m1_value(w.codes) * np.repeat(e4m3fn_value(w.scales), BLOCK[NVFP4], axis=1)
    else:
        v = dequant(w).astype(np.float64)
    return round_to_bf16(v)


def bits_per_weight(fmt: int) -> float:
    """Storage bits per weight of the logical format: code bits plus the per-block
    scale data spread over the block (TurboEXL3 article §2.1)."""
    if fmt == MLX_AFFINE4_G64:
        return 4 + (16 + 16) / 64
    if fmt == MXFP4:
        return 4 + 8 / 32
    if fmt == NVFP4:
        return 4 + 8 / 16  # the single fp32 tensor scale is not per weight
    if fmt == Q6K:
        return 6 + 8 / 16 + 16 / 256
    if fmt == Q5_0:
        return 5 + 16 / 32
    if fmt == Q5_1:
        return 5 + (16 + 16) / 32
    if fmt == Q5_K:
        return 5 + (6 + 6) / 32 + (16 + 16) / 256
    raise ValueError(fmt)


def q6k_half_operand_bits(code) -> np.ndarray:
    """fp16 bit pattern of the Q6_K operand of the Q6_K operand PR ("What changed"):
    the code's low nibble in mantissa bits 4..7 and its two high bits in bits 8..9
    of a half whose exponent encodes 1.0, i.e. the half 1 + code/64."""
    c = np.asarray(code).astype(np.uint16) & 0x3F
    return (np.uint16(0x3C00) | ((c & 0xF) << 4) | ((c >> 4) << 8)).astype(np.uint16)


def q5_half_operand_bits(code) -> np.ndarray:
    """fp16 bit pattern of the 5-bit operand of the Q6_K operand PR (commit "5-bit
    nibble operand"): the low nibble in mantissa bits 4..7 and the fifth bit at bit 8
    of a half whose exponent encodes 1.0, i.e. the half 1 + code/64."""
    c = np.asarray(code).astype(np.uint16) & 0x1F
    return (np.uint16(0x3C00) | ((c & 0xF) << 4) | ((c >> 4) << 8)).astype(np.uint16)
