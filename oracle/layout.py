"""Independent reader of the packed device layout (oracle; test infrastructure only).

Written from the layout specification alone, so that a packer bug cannot hide
behind a shared helper.  The specification ("T128x64"):

* Rows are padded to NP = 128 * ceil(N / 128), the reduction dimension to KP =
  ceil(K / KB) * KB with KB = 64 for the 4-bit formats and 256 for Q6_K.  The
  matrix is cut into tiles of 128 rows x 64 columns; tile (q, g) has index
  t = q * KG + g with KG = KP / 64.  Padding holds zero codes and zero scales.
* codes: TB bytes per tile (4096 for 4-bit formats, 6144 for Q6_K) at offset
  t * TB.  Row r of the tile (rt = r // 32, lane = r % 32) owns the 16-byte
  chunks at ((rt * 2 + c) * 32 + lane) * 16 (4-bit and 5-bit formats).
  - 4-bit formats, chunk c in {0, 1}: byte b holds code (g*64 + c*32 + 2b) in
    its low nibble and code (g*64 + c*32 + 2b + 1) in its high nibble.
  - Q6_K (TB = 6144): row r's 16-column quarter kq (columns g*64 + 16 kq ..)
    is three little-endian 32-bit words, word c in 0..2 at byte offset
    ((rt * 4 + kq) * 3 + c) * 128 + lane * 4; byte j of word c holds in bits
    2..7 the code of column 16 kq + 4c + j and in bits 0..1 bits 2c..2c+1 of the
    code of column 16 kq + 12 + j.
* scales: 128 * SB bytes per tile at offset t * 128 * SB, SB bytes per row:
  - NVFP4 (SB = 4): byte i = E4M3 scale of columns g*64 + 16i .. +15;
  - MXFP4 (SB = 2): byte i = E8M0 scale of columns g*64 + 32i .. +31;
  - MLX affine (SB = 4): little-endian fp16 scale s, then fp16 bias b, of the
    64-column group;
  - Q6_K (SB = 4): byte i = int8 scale of columns g*64 + 16i .. +15.
* aux (Q6_K only): fp16 d of columns u*256 .. +255 for row r of row tile q at
  byte offset (q * (KG / 4) + u) * 256 + 2 r.
* 5-bit formats (Q5_0, Q5_1, Q5_K): TB = 5120.  Bytes 0..4095 hold the low nibbles
  (code & 15) exactly as the 4-bit formats' chunks (CH = 2); bytes 4096..5119 hold
  the fifth bits: two little-endian 32-bit words per row, word j in {0, 1} of row r
  at byte 4096 + 512 j + 4 r, holding bit (code >> 4) of column g*64 + 32j + 8u + i
  (u in 0..3, i in 0..7) at bit (4i + 4 + u) mod 32.  KB = 256 for Q5_K, 64
  otherwise.
  - Q5_0 (SB = 4): fp16 d of columns g*64 + 32i .. +31 at bytes 2i..2i+1;
  - Q5_1 (SB = 8): fp16 d then fp16 m of columns g*64 + 32i .. +31 at bytes
    4i..4i+3;
  - Q5_K (SB = 3): a little-endian 24-bit value holding the 6-bit sc of columns
    g*64 .. +31 in bits 0..5, its mn in 6..11, and sc, mn of g*64+32 .. +63 in
    12..17 and 18..23;
  - aux (Q5_K): fp16 d then fp16 dmin of columns u*256 .. +255 for row r of row
    tile q at byte offset (q * (KG / 4) + u) * 512 + 4 r.
"""
from __future__ import annotations

import numpy as np

MLX_AFFINE4_G64, MXFP4, NVFP4, Q6K, Q5_0, Q5_1, Q5_K = 1, 2, 3, 4, 5, 6, 7
_SB = {MLX_AFFINE4_G64: 4, MXFP4: 2, NVFP4: 4, Q6K: 4, Q5_0: 4, Q5_1: 8, Q5_K: 3}
_Q5 = (Q5_0, Q5_1, Q5_K)


def _geometry(fmt: int, n: int, k: int):
    kb = 256 if fmt in (Q6K, Q5_K) else 64
    np_ = -(-n // 128) * 128
    kp = -(-k // kb) * kb
    return np_, kp, np_ // 128, kp // 64


def packed_sizes(fmt: int, n: int, k: int):
    """(codes, scales, aux) byte counts of the packed layout."""
    np_, kp, nt, kg = _geometry(fmt, n, k)
    tb = 6144 if fmt == Q6K else 5120 if fmt in _Q5 else 4096
    codes = nt * kg * tb
    scales = nt * kg * 128 * _SB[fmt]
    aux = nt * (kg // 4) * 256 if fmt == Q6K else nt * (kg // 4) * 512 if fmt == Q5_K else 0
    return codes, scales, aux


def unpack(fmt: int, n: int, k: int, codes: np.ndarray, scales: np.ndarray, aux=None, full: bool = False):
    """Logical arrays from packed bytes.

    Returns (codes u8 [n, k], scales, aux) in the logical form of each format;
    with ``full=True`` the padded [NP, KP] arrays are returned instead."""
    np_, kp, nt, kg = _geometry(fmt, n, k)
    codes = np.frombuffer(np.ascontiguousarray(codes).tobytes(), dtype=np.uint8)
    scales = np.frombuffer(np.ascontiguousarray(scales).tobytes(), dtype=np.uint8)
    tb = 6144 if fmt == Q6K else 5120 if fmt in _Q5 else 4096
    tiles = codes.reshape(nt, kg, tb)
    if fmt == Q6K:
        # bytes indexed [q, g, rt, kq, c, lane, j]
        qb = tiles.reshape(nt, kg, 4, 4, 3, 32, 4)
        main = qb >> 2  # codes of columns 16 kq + 4c + j
        low = (qb[..., 0, :, :] & 3) | ((qb[..., 1, :, :] & 3) << 2) | ((qb[..., 2, :, :] & 3) << 4)  # 12 + j
        cols = np.concatenate([main.transpose(0, 1, 2, 3, 5, 4, 6).reshape(nt, kg, 4, 4, 32, 12),
                               low.reshape(nt, kg, 4, 4, 32, 4)], axis=-1)  # [q, g, rt, kq, lane, 16]
        logical = cols.transpose(0, 2, 4, 1, 3, 5).reshape(np_, kp).astype(np.uint8)
    else:
        # chunk bytes indexed [q, g, rt, c, lane, b]
        cb = tiles[:, :, :4096].reshape(nt, kg, 4, 2, 32, 16)
        lo = cb & 0x0F
        hi = cb >> 4
        nib = np.stack([lo, hi], axis=-1)  # [q, g, rt, c, lane, b, 2]
        # -> [q, rt, lane, g, c, b, 2] -> rows x columns
        logical = nib.transpose(0, 2, 4, 1, 3, 5, 6).reshape(np_, kp).astype(np.uint8)
    if fmt in _Q5:
        fb = tiles[:, :, 4096:].reshape(nt, kg, 2, 128, 4).transpose(0, 1, 3, 2, 4).astype(np.uint32)  # [q, g, row, j, byte]
        w32 = fb[..., 0] | (fb[..., 1] << 8) | (fb[..., 2] << 16) | (fb[..., 3] << 24)
        u = np.arange(4, dtype=np.uint32)[:, None]
        i = np.arange(8, dtype=np.uint32)[None, :]
        pos = (4 * i + 4 + u) % 32  # [u, i]: column 32j + 8u + i
        bits = (w32[..., None, None] >> pos) & 1  # [q, g, row, j, u, i]
        frow = bits.reshape(nt, kg, 128, 64).transpose(0, 2, 1, 3).reshape(np_, kp).astype(np.uint8)
        logical = (logical | (frow << 4)).astype(np.uint8)
    sb = _SB[fmt]
    sc = scales.reshape(nt, kg, 128, sb).transpose(0, 2, 1, 3).reshape(np_, kg * sb)
    aux_out = None
    if fmt == NVFP4:
        sc_out = sc.copy()
    elif fmt == MXFP4:
        sc_out = sc.copy()
    elif fmt == Q5_0:
        sc_out = sc.copy().view(np.float16).reshape(np_, kg * 2)
    elif fmt == Q5_1:
        pairs = sc.reshape(np_, kg * 2, 2, 2).copy()  # [row, block, (d, m), byte]
        sc_out = pairs[:, :, 0, :].copy().view(np.float16).reshape(np_, kg * 2)
        aux_out = pairs[:, :, 1, :].copy().view(np.float16).reshape(np_, kg * 2)
    elif fmt == Q5_K:
        b = sc.reshape(np_, kg, 3).astype(np.uint32)
        v = b[..., 0] | (b[..., 1] << 8) | (b[..., 2] << 16)
        f = np.stack([(v >> s) & 63 for s in (0, 6, 12, 18)], axis=-1)  # sc0, mn0, sc1, mn1
        sc_out = f.reshape(np_, kg * 2, 2).astype(np.uint8)
        a = np.frombuffer(np.ascontiguousarray(aux).tobytes(), dtype=np.uint8)
        a = a.reshape(nt, kg // 4, 128, 2, 2).transpose(0, 2, 1, 3, 4).reshape(np_, (kg // 4) * 4)
        aux_out = a.copy().view(np.float16).reshape(np_, kg // 4, 2)
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
    blk = {MLX_AFFINE4_G64: 64, MXFP4: 32, NVFP4: 16, Q6K: 16, Q5_0: 32, Q5_1: 32, Q5_K: 32}[fmt]
    sc_cut = sc_out[:n, :k // blk]
    if fmt in (Q6K, Q5_K):
        aux_cut = aux_out[:n, :k // 256]
    elif fmt == MLX_AFFINE4_G64:
        aux_cut = aux_out[:n, :k // 64]
    elif fmt == Q5_1:
        aux_cut = aux_out[:n, :k // 32]
    else:
        aux_cut = None
    return logical[:n, :k], sc_cut, aux_cut
