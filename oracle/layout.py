"""Independent reader of the packed device layout (oracle; test infrastructure only).

Written from the layout specification alone, so that a packer bug cannot hide
behind a shared helper.  The specification ("T128x64"):

* Rows are padded to NP = 128 * ceil(N / 128), the reduction dimension to KP =
  ceil(K / KB) * KB with KB = 64 for the 4-bit formats and 256 for Q6_K.  The
  matrix is cut into tiles of 128 rows x 64 columns; tile (q, g) has index
  t = q * KG + g with KG = KP / 64.  Padding holds zero codes and zero scales.
* codes: TB bytes per tile (4096 for 4-bit formats, 6144 for Q6_K) at offset
  t * TB.  Row r of the tile (rt = r // 32, lane = r % 32) owns the 16-byte
  chunks at ((rt * CH + c) * 32 + lane) * 16, CH = 2 (4-bit) or 3 (Q6_K).
  - 4-bit formats, chunk c in {0, 1}: byte b holds code (g*64 + c*32 + 2b) in
    its low nibble and code (g*64 + c*32 + 2b + 1) in its high nibble.
  - Q6_K: chunks 0 and 1 hold the low nibbles (code & 15) as above; chunk 2 is
    four little-endian 32-bit words, word w in 0..3 holding in its nibble j
    (bits 4j..4j+3) hi(g*64 + 16w + j) | hi(g*64 + 16w + 8 + j) << 2, with
    hi(code) = code >> 4.
* scales: 128 * SB bytes per tile at offset t * 128 * SB, SB bytes per row:
  - NVFP4 (SB = 4): byte i = E4M3 scale of columns g*64 + 16i .. +15;
  - MXFP4 (SB = 2): byte i = E8M0 scale of columns g*64 + 32i .. +31;
  - MLX affine (SB = 4): little-endian fp16 scale s, then fp16 bias b, of the
    64-column group;
  - Q6_K (SB = 4): byte i = int8 scale of columns g*64 + 16i .. +15.
* aux (Q6_K only): fp16 d of columns u*256 .. +255 for row r of row tile q at
  byte offset (q * (KG / 4) + u) * 256 + 2 r.
"""
from __future__ import annotations

import numpy as np

MLX_AFFINE4_G64, MXFP4, NVFP4, Q6K = 1, 2, 3, 4
_SB = {MLX_AFFINE4_G64: 4, MXFP4: 2, NVFP4: 4, Q6K: 4}


def _geometry(fmt: int, n: int, k: int):
    kb = 256 if fmt == Q6K else 64
    np_ = -(-n // 128) * 128
    kp = -(-k // kb) * kb
    return np_, kp, np_ // 128, kp // 64


def packed_sizes(fmt: int, n: int, k: int):
    """(codes, scales, aux) byte counts of the packed layout."""
    np_, kp, nt, kg = _geometry(fmt, n, k)
    tb = 6144 if fmt == Q6K else 4096
    codes = nt * kg * tb
    scales = nt * kg * 128 * _SB[fmt]
    aux = nt * (kg // 4) * 256 if fmt == Q6K else 0
    return codes, scales, aux


def unpack(fmt: int, n: int, k: int, codes: np.ndarray, scales: np.ndarray, aux=None, full: bool = False):
    """Logical arrays from packed bytes.

    Returns (codes u8 [n, k], scales, aux) in the logical form of each format;
    with ``full=True`` the padded [NP, KP] arrays are returned instead."""
    np_, kp, nt, kg = _geometry(fmt, n, k)
    codes = np.frombuffer(np.ascontiguousarray(codes).tobytes(), dtype=np.uint8)
    scales = np.frombuffer(np.ascontiguousarray(scales).tobytes(), dtype=np.uint8)
    ch = 3 if fmt == Q6K else 2
    # chunk bytes indexed [q, g, rt, c, lane, b]
    cb = codes.reshape(nt, kg, 4, ch, 32, 16)
    lo = cb[:, :, :, :2] & 0x0F
    hi = cb[:, :, :, :2] >> 4
    nib = np.stack([lo, hi], axis=-1)  # [q, g, rt, c, lane, b, 2]
    # -> [q, rt, lane, g, c, b, 2] -> rows x columns
    logical = nib.transpose(0, 2, 4, 1, 3, 5, 6).reshape(np_, kp).astype(np.uint8)
    if fmt == Q6K:
        words = cb[:, :, :, 2].reshape(nt, kg, 4, 32, 4, 4)  # [q, g, rt, lane, w, byte]
        words = words.astype(np.uint32)
        w32 = words[..., 0] | (words[..., 1] << 8) | (words[..., 2] << 16) | (words[..., 3] << 24)
        j = np.arange(8, dtype=np.uint32)
        nibs = (w32[..., None] >> (4 * j)) & 0xF  # [q, g, rt, lane, w, j]
        h_first = nibs & 3  # code 16w + j
        h_second = nibs >> 2  # code 16w + 8 + j
        hsel = np.concatenate([h_first, h_second], axis=-1)  # [q, g, rt, lane, w, 16]
        hrow = hsel.transpose(0, 2, 3, 1, 4, 5).reshape(np_, kp).astype(np.uint8)
        logical = (logical | (hrow << 4)).astype(np.uint8)
    sb = _SB[fmt]
    sc = scales.reshape(nt, kg, 128, sb).transpose(0, 2, 1, 3).reshape(np_, kg * sb)
    aux_out = None
    if fmt == NVFP4:
        sc_out = sc.copy()
    elif fmt == MXFP4:
        sc_out = sc.copy()
    elif fmt == Q6K:
        sc_out = sc.view(np.int8).copy()
        a = np.frombuffer(np.ascontiguousarray(aux).tobytes(), dtype=np.uint8)
        a = a.reshape(nt, kg // 4, 128, 2).transpose(0, 2, 1, 3).reshape(np_, (kg // 4) * 2)
        aux_out = a.copy().view(np.float16)
    else:  # MLX: (s, b) fp16 pairs
        pairs = sc.reshape(np_, kg, 2, 2).copy()
        sc_out = pairs[:, :, 0, :].copy().view(np.float16).reshape(np_, kg)
        aux_out = pairs[:, :, 1, :].copy().view(np.float16).reshape(np_, kg)
    if full:
        return logical, sc_out, aux_out
    blk = {MLX_AFFINE4_G64: 64, MXFP4: 32, NVFP4: 16, Q6K: 16}[fmt]
    sc_cut = sc_out[:n, :k // blk]
    if fmt == Q6K:
        aux_cut = aux_out[:n, :k // 256]
    elif fmt == MLX_AFFINE4_G64:
        aux_cut = aux_out[:n, :k // 64]
    else:
        aux_cut = None
    return logical[:n, :k], sc_cut, aux_cut
