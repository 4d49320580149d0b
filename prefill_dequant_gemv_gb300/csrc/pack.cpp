// Host-side packer: logical block-scaled weights -> packed "T128x64" layout.
//
// Formats (TurboEXL3 article §2.1; Q6_K operand PR #19): MLX affine 4-bit with fp16
// scale and bias per 64, MXFP4 (E2M1 + E8M0 per 32), NVFP4 (E2M1 + E4M3 per 16),
// Q6_K-style 6-bit codes with int8 scale per 16 and fp16 d per 256.  The layout is
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
    default: return 0;
  }
}

bool geometry(int fmt, int64_t n, int64_t k, Geometry* g) {
  const int blk = format_block(fmt);
  if (blk == 0 || n <= 0 || k <= 0 || k % blk != 0) return false;
  if (n > (int64_t(1) << 40) || k > (int64_t(1) << 30)) return false;
  const int64_t kb = (fmt == QG_FMT_Q6K) ? 256 : 64;
  g->fmt = fmt;
  g->n = n;
  g->k = k;
  g->np = (n + 127) / 128 * 128;
  g->kp = (k + kb - 1) / kb * kb;
  g->nt = g->np / 128;
  g->kg = g->kp / 64;
  g->tile_bytes = (fmt == QG_FMT_Q6K) ? 6144 : 4096;
  g->sb = (fmt == QG_FMT_MXFP4) ? 2 : 4;
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
  if (aux_bytes) *aux_bytes = (fmt == QG_FMT_Q6K) ? (size_t)(g.nt * (g.kg / 4)) * 256 : 0;
  return QG_OK;
}

extern "C" qg_status qg_pack_host(int fmt, int64_t n, int64_t k, const uint8_t* lc, const void* ls, const void* la,
                                  void* codes, void* scales, void* aux) {
  Geometry g;
  if (!qg::geometry(fmt, n, k, &g)) return QG_ERR_INVALID_ARG;
  if (!lc || !ls || !codes || !scales) return QG_ERR_INVALID_ARG;
  const bool q6k = fmt == QG_FMT_Q6K;
  const bool mlx = fmt == QG_FMT_MLX_AFFINE4_G64;
  if ((q6k || mlx) && !la) return QG_ERR_INVALID_ARG;
  if (q6k && !aux) return QG_ERR_INVALID_ARG;
  const uint8_t maxcode = q6k ? 63 : 15;
  for (int64_t i = 0; i < n * k; ++i)
    if (lc[i] > maxcode) return QG_ERR_INVALID_ARG;

  size_t cb = 0, sb = 0, ab = 0;
  qg_packed_sizes(fmt, n, k, &cb, &sb, &ab);
  uint8_t* co = static_cast<uint8_t*>(codes);
  uint8_t* so = static_cast<uint8_t*>(scales);
  uint8_t* ao = static_cast<uint8_t*>(aux);
  memset(co, 0, cb);
  memset(so, 0, sb);
  if (ab) memset(ao, 0, ab);

  const int ch = q6k ? 3 : 2;
  for (int64_t r = 0; r < n; ++r) {
    const int64_t q = r / 128;
    const int row = (int)(r % 128), rt = row / 32, lane = row % 32;
    const uint8_t* src = lc + r * k;
    for (int64_t c = 0; c < k; ++c) {
      const int64_t gi = c / 64;
      const int kk = (int)(c % 64);
      uint8_t* tile = co + (size_t)(q * g.kg + gi) * g.tile_bytes;
      const int chunk = kk / 32, byte = (kk % 32) / 2, high = kk & 1;
      const uint8_t code = src[c];
      tile[((rt * ch + chunk) * 32 + lane) * 16 + byte] |= (uint8_t)((code & 15) << (4 * high));
      if (q6k) {
        const int w = kk / 16, j = kk % 16;
        const int bit = 4 * (j % 8) + (j < 8 ? 0 : 2);  // nibble j%8, low or high bit pair
        tile[((rt * ch + 2) * 32 + lane) * 16 + w * 4 + bit / 8] |= (uint8_t)((code >> 4) << (bit % 8));
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
