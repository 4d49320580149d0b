// Host-side packer: logical block-scaled weights -> packed "T128x64" layout.
//
// Formats (TurboEXL3 article §2.1; Q6_K operand PR #19): MLX affine 4-bit with fp16
// scale and bias per 64, MXFP4 (E2M1 + E8M0 per 32), NVFP4 (E2M1 + E4M3 per 16),
// Q6_K-style 6-bit codes with int8 scale per 16 and fp16 d per 256, and the 5-bit
// formats of the PR's 5-bit nibble operand as the GGML blocks define them (Q5_0: fp16 d
// per 32; Q5_1: fp16 d and m per 32; Q5_K: 6-bit sc and mn per 32, fp16 d and dmin per
// 256).  The layout is
// documented in include/qgemv.h; it groups each 128-row x 64-input tile's bytes
// contiguously so one bulk copy moves a whole tile, and interleaves rows so that
// 32 consecutive rows share every 512-byte chunk.
#include <string.h>

#include "qg_internal.h"

namespace qg {

int format_block(int fmt) {
  switch (fmt) {
    case QG_FMT_MLX_AFFINE4_G64: return 64;
    case QG_FMT_MXFP4: return 32;
    case QG_FMT_NVFP4: return 16;
    case QG_FMT_Q6K: return 256;
    case QG_FMT_Q5_0: return 32;
    case QG_FMT_Q5_1: return 32;
    case QG_FMT_Q5_K: return 256;
    default: return 0;
  }
}

bool is_q5(int fmt) { return fmt == QG_FMT_Q5_0 || fmt == QG_FMT_Q5_1 || fmt == QG_FMT_Q5_K; }

// Aux bytes per row tile and 256-input group (4 tiles): Q6_K d, Q5_K (d, dmin).
int aux_group_bytes(int fmt) { return fmt == QG_FMT_Q6K ? 256 : fmt == QG_FMT_Q5_K ? 512 : 0; }

bool geometry(int fmt, int64_t n, int64_t k, Geometry* g) {
  const int blk = format_block(fmt);
  if (blk == 0 || n <= 0 || k <= 0 || k % blk != 0) return false;
  if (n > (int64_t(1) << 40) || k > (int64_t(1) << 30)) return false;
  const int64_t kb = (fmt == QG_FMT_Q6K || fmt == QG_FMT_Q5_K) ? 256 : 64;
  g->fmt = fmt;
  g->n = n;
  g->k = k;
  g->np = (n + 127) / 128 * 128;
  g->kp = (k + kb - 1) / kb * kb;
  g->nt = g->np / 128;
  g->kg = g->kp / 64;
  g->tile_bytes = (fmt == QG_FMT_Q6K) ? 6144 : is_q5(fmt) ? 5120 : 4096;
  g->sb = (fmt == QG_FMT_MXFP4) ? 2 : (fmt == QG_FMT_Q5_1) ? 8 : (fmt == QG_FMT_Q5_K) ? 3 : 4;
  return true;
}

}  // namespace qg

using qg::Geometry;

extern "C" qg_status qg_packed_sizes(int fmt, int64_t n, int64_t k, size_t* codes_bytes, size_t* scales_bytes,
                                     size_t* aux_bytes) {
  Geometry g;
  if (!qg::geometry(fmt, n, k, &g)) return QG_ERR_INVALID_ARG;
  const size_t tiles = (size_t)(g.nt * g.kg);
  if (codes_bytes) *codes_bytes = tiles * (size_t)g.tile_bytes;
  if (scales_bytes) *scales_bytes = tiles * 128 * (size_t)g.sb;
  if (aux_bytes) *aux_bytes = (size_t)(g.nt * (g.kg / 4)) * (size_t)qg::aux_group_bytes(fmt);
  return QG_OK;
}

extern "C" qg_status qg_pack_host(int fmt, int64_t n, int64_t k, const uint8_t* lc, const void* ls, const void* la,
                                  void* codes, void* scales, void* aux) {
  Geometry g;
  if (!qg::geometry(fmt, n, k, &g)) return QG_ERR_INVALID_ARG;
  if (!lc || !ls || !codes || !scales) return QG_ERR_INVALID_ARG;
  const bool q6k = fmt == QG_FMT_Q6K;
  const bool mlx = fmt == QG_FMT_MLX_AFFINE4_G64;
  const bool q5 = qg::is_q5(fmt);
  if ((q6k || mlx || fmt == QG_FMT_Q5_1 || fmt == QG_FMT_Q5_K) && !la) return QG_ERR_INVALID_ARG;
  if ((q6k || fmt == QG_FMT_Q5_K) && !aux) return QG_ERR_INVALID_ARG;
  const uint8_t maxcode = q6k ? 63 : q5 ? 31 : 15;
  for (int64_t i = 0; i < n * k; ++i)
    if (lc[i] > maxcode) return QG_ERR_INVALID_ARG;
  if (fmt == QG_FMT_Q5_K) {
    const uint8_t* sm = static_cast<const uint8_t*>(ls);
    for (int64_t i = 0; i < n * (k / 32) * 2; ++i)
      if (sm[i] > 63) return QG_ERR_INVALID_ARG;
  }

  size_t cb = 0, sb = 0, ab = 0;
  qg_packed_sizes(fmt, n, k, &cb, &sb, &ab);
  uint8_t* co = static_cast<uint8_t*>(codes);
  uint8_t* so = static_cast<uint8_t*>(scales);
  uint8_t* ao = static_cast<uint8_t*>(aux);
  memset(co, 0, cb);
  memset(so, 0, sb);
  if (ab) memset(ao, 0, ab);

  for (int64_t r = 0; r < n; ++r) {
    const int64_t q = r / 128;
    const int row = (int)(r % 128), rt = row / 32, lane = row % 32;
    const uint8_t* src = lc + r * k;
    for (int64_t c = 0; c < k; ++c) {
      const int64_t gi = c / 64;
      const int kk = (int)(c % 64);
      uint8_t* tile = co + (size_t)(q * g.kg + gi) * g.tile_bytes;
      const uint8_t code = src[c];
      if (q6k) {  // quarter kq, words of ((rt*4 + kq)*3 + w)*128 + lane*4
        const int kq = kk / 16, i = kk % 16;
        uint8_t* qw = tile + ((rt * 4 + kq) * 3) * 128 + lane * 4;
        if (i < 12) {
          qw[(i / 4) * 128 + i % 4] |= (uint8_t)(code << 2);  // bits 2..7 of byte i%4 of word i/4
        } else {
          for (int w = 0; w < 3; ++w) qw[w * 128 + (i - 12)] |= (uint8_t)((code >> (2 * w)) & 3);
        }
        continue;
      }
      const int chunk = kk / 32, byte = (kk % 32) / 2, high = kk & 1;
      tile[((rt * 2 + chunk) * 32 + lane) * 16 + byte] |= (uint8_t)((code & 15) << (4 * high));
      if (q5) {  // fifth bit of input 32j + 8u + i at bit (4i + 4 + u) mod 32 of word j
        const int j = kk / 32, u = (kk % 32) / 8, i = kk % 8;
        const int bit = (4 * i + 4 + u) % 32;
        tile[4096 + j * 512 + row * 4 + bit / 8] |= (uint8_t)((code >> 4) << (bit % 8));
      }
    }
  }

  const int64_t kg = g.kg;
  for (int64_t r = 0; r < n; ++r) {
    const int64_t q = r / 128;
    const int row = (int)(r % 128);
    switch (fmt) {
      case QG_FMT_NVFP4: {
        const uint8_t* s = static_cast<const uint8_t*>(ls) + r * (k / 16);
        for (int64_t b = 0; b < k / 16; ++b) so[(size_t)(q * kg + b / 4) * 128 * 4 + row * 4 + b % 4] = s[b];
        break;
      }
      case QG_FMT_MXFP4: {
        const uint8_t* s = static_cast<const uint8_t*>(ls) + r * (k / 32);
        for (int64_t b = 0; b < k / 32; ++b) so[(size_t)(q * kg + b / 2) * 128 * 2 + row * 2 + b % 2] = s[b];
        break;
      }
      case QG_FMT_MLX_AFFINE4_G64: {
        const uint16_t* s = static_cast<const uint16_t*>(ls) + r * (k / 64);
        const uint16_t* bi = static_cast<const uint16_t*>(la) + r * (k / 64);
        for (int64_t b = 0; b < k / 64; ++b) {
          uint8_t* d = so + (size_t)(q * kg + b) * 128 * 4 + row * 4;
          d[0] = (uint8_t)(s[b] & 0xFF);
          d[1] = (uint8_t)(s[b] >> 8);
          d[2] = (uint8_t)(bi[b] & 0xFF);
          d[3] = (uint8_t)(bi[b] >> 8);
        }
        break;
      }
      case QG_FMT_Q5_0:
      case QG_FMT_Q5_1: {  // fp16 d (and m) per 32 inputs
        const uint16_t* d = static_cast<const uint16_t*>(ls) + r * (k / 32);
        const uint16_t* m = static_cast<const uint16_t*>(la) + r * (k / 32);
        const int per = fmt == QG_FMT_Q5_1 ? 4 : 2;
        for (int64_t b = 0; b < k / 32; ++b) {
          uint8_t* o = so + (size_t)(q * kg + b / 2) * 128 * g.sb + row * g.sb + (b % 2) * per;
          o[0] = (uint8_t)(d[b] & 0xFF);
          o[1] = (uint8_t)(d[b] >> 8);
          if (fmt == QG_FMT_Q5_1) {
            o[2] = (uint8_t)(m[b] & 0xFF);
            o[3] = (uint8_t)(m[b] >> 8);
          }
        }
        break;
      }
      case QG_FMT_Q5_K: {  // 6-bit (sc, mn) pairs per 32 inputs, fp16 (d, dmin) per 256
        const uint8_t* sm = static_cast<const uint8_t*>(ls) + r * (k / 32) * 2;
        for (int64_t gi = 0; gi < k / 64; ++gi) {
          const uint32_t v = (uint32_t)sm[4 * gi] | ((uint32_t)sm[4 * gi + 1] << 6) |
                             ((uint32_t)sm[4 * gi + 2] << 12) | ((uint32_t)sm[4 * gi + 3] << 18);
          uint8_t* o = so + (size_t)(q * kg + gi) * 128 * 3 + row * 3;
          o[0] = (uint8_t)(v & 0xFF);
          o[1] = (uint8_t)((v >> 8) & 0xFF);
          o[2] = (uint8_t)(v >> 16);
        }
        const uint16_t* dd = static_cast<const uint16_t*>(la) + r * (k / 256) * 2;
        for (int64_t u = 0; u < k / 256; ++u) {
          uint8_t* o = ao + (size_t)(q * (kg / 4) + u) * 512 + row * 4;
          o[0] = (uint8_t)(dd[2 * u] & 0xFF);
          o[1] = (uint8_t)(dd[2 * u] >> 8);
          o[2] = (uint8_t)(dd[2 * u + 1] & 0xFF);
          o[3] = (uint8_t)(dd[2 * u + 1] >> 8);
        }
        break;
      }
      default: {  // Q6_K
        const uint8_t* s = static_cast<const uint8_t*>(ls) + r * (k / 16);
        for (int64_t b = 0; b < k / 16; ++b) so[(size_t)(q * kg + b / 4) * 128 * 4 + row * 4 + b % 4] = s[b];
        const uint16_t* d = static_cast<const uint16_t*>(la) + r * (k / 256);
        for (int64_t u = 0; u < k / 256; ++u) {
          uint8_t* o = ao + (size_t)(q * (kg / 4) + u) * 256 + row * 2;
          o[0] = (uint8_t)(d[u] & 0xFF);
          o[1] = (uint8_t)(d[u] >> 8);
        }
        break;
      }
    }
  }
  return QG_OK;
}
