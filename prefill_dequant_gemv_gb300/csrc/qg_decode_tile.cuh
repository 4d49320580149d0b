// Decode of one packed 128 x 64 weight tile into bf16 tensor-core operands, shared by the
// dense and grouped prefill GEMMs (each thread's words go to its TMEM lane).  Every
// decoded value is exact in bf16: E2M1 x a power-of-two or E4M3 block scale, and integer
// codes times the fp16/fp32 scale products, rounded once (TurboEXL3 article §4.1: the
// stage's weights are decoded into on-chip memory in the multiplier's fragment order).
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "qg_common.cuh"

namespace qg {

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Decode one code word of row r: word wg (0..7) of the row's 64-input stage holds inputs
// 8wg..8wg+7 (4-bit formats; 5-bit low nibbles, with the fifth bits from the tile's
// fifth-bit plane); the result is four bf16x2 words in input order (low half = lower
// input).  Raw stage layout: codes, then 128 rows' scales, then the rows' aux records
// (Q6_K, Q5_K).  Q6_K decodes by quarters (decode_q6k_quarter).
template <int FMT>
__device__ __forceinline__ void decode_word(const uint8_t* raw, int r, int wg, uint32_t w, uint32_t* o) {
  using F = Fmt<FMT>;
  const uint8_t* sp = raw + F::TB + r * F::SB;
  float v[8];
  if constexpr (FMT == FMT_NVFP4 || FMT == FMT_MXFP4) {
    float S;
    if (FMT == FMT_NVFP4) {
      const int blk = wg >> 1;  // 16-input blocks
      const uint32_t sw = *reinterpret_cast<const uint32_t*>(sp);
      const float2 s01 = (blk >> 1) ? e4m3x2_f32<1>(sw) : e4m3x2_f32<0>(sw);
      S = (blk & 1) ? s01.y : s01.x;
    } else {
      S = e8m0_f32(sp[wg >> 2]);  // 32-input blocks
    }
    const uint32_t hb[4] = {e2m1x2_h2<0>(w), e2m1x2_h2<1>(w), e2m1x2_h2<2>(w), e2m1x2_h2<3>(w)};
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const float2 e = __half22float2(*reinterpret_cast<const __half2*>(&hb[b]));
      v[2 * b] = S * e.x;  // exact
      v[2 * b + 1] = S * e.y;
    }
  } else {
    static_assert(FMT != FMT_Q6K, "Q6_K decodes by quarters");
    uint32_t op[4];
    uint32_t hh = 0;
    if (fmt_q5(FMT)) {
      hh = q5_hi_for(*reinterpret_cast<const uint32_t*>(raw + kQ5Plane + (wg >> 2) * 512 + r * 4), wg & 3);
    }
    int_ops<FMT>(w, hh, op);
    float code[8];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 e = __half22float2(*reinterpret_cast<const __half2*>(&op[j]));
      const float mul = (j & 1) ? 64.0f : 1024.0f;
      code[j] = (e.x - 1.0f) * mul;  // exact integer code
      code[j + 4] = (e.y - 1.0f) * mul;
    }
    if (FMT == FMT_MLX) {
      const uint32_t sw = *reinterpret_cast<const uint32_t*>(sp);
      const float s = __half2float(__ushort_as_half((unsigned short)(sw & 0xFFFFu)));
      const float bias = __half2float(__ushort_as_half((unsigned short)(sw >> 16)));
#pragma unroll
      for (int j = 0; j < 8; ++j) v[j] = fmaf(s, code[j], bias);
    } else {  // 5-bit: the fp32 weight, one rounding: fma of the exact s * code and bias
      const float2 sb = q5_affine<FMT>(sp, raw + F::TB + 128 * F::SB + r * fmt_aux_row(FMT), wg >> 2);
#pragma unroll
      for (int j = 0; j < 8; ++j) v[j] = fmaf(sb.x, code[j], sb.y);
    }
  }
  o[0] = pack_bf16x2(v[0], v[1]);
  o[1] = pack_bf16x2(v[2], v[3]);
  o[2] = pack_bf16x2(v[4], v[5]);
  o[3] = pack_bf16x2(v[6], v[7]);
}

// Q6_K: one 16-input quarter kq of row r as 8 bf16x2 words in input order, w = d*sc*(code - 32)
// (exact in fp32, rounded once to bf16).
__device__ __forceinline__ void decode_q6k_quarter(const uint8_t* raw, int r, int kq, uint32_t* o) {
  using F = Fmt<FMT_Q6K>;
  const uint8_t* qb = raw + q6k_word_offset(r >> 5, kq, 0, r & 31);
  uint32_t op[8];
  q6k_ops(*reinterpret_cast<const uint32_t*>(qb), *reinterpret_cast<const uint32_t*>(qb + 128),
          *reinterpret_cast<const uint32_t*>(qb + 256), op);
  float code[16];  // input order
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const float2 e = __half22float2(*reinterpret_cast<const __half2*>(&op[j]));
    const float mul = j < 6 ? 256.0f : 1024.0f;
    // op 2c holds inputs (4c, 4c+2), op 2c+1 holds (4c+1, 4c+3)
    const int base = (j >> 1) * 4 + (j & 1);
    code[base] = (e.x - 1.0f) * mul;  // exact integer code
    code[base + 2] = (e.y - 1.0f) * mul;
  }
  const float sc = (float)(int8_t)raw[F::TB + r * F::SB + kq];
  const float d = __half2float(*reinterpret_cast<const __half*>(raw + F::TB + 128 * F::SB + r * 2));
  const float ds = d * sc;
#pragma unroll
  for (int i = 0; i < 8; ++i) o[i] = pack_bf16x2(ds * (code[2 * i] - 32.0f), ds * (code[2 * i + 1] - 32.0f));
}

// Decode one thread's share of a stage: row r, inputs 32h..32h+31, as 16 bf16x2 words in
// input order (word i holds inputs 32h+2i (low half) and 32h+2i+1).
template <int FMT>
__device__ __forceinline__ void decode_regs(const uint8_t* raw, int r, int h, uint32_t (&o)[16]) {
  using F = Fmt<FMT>;
  if constexpr (FMT == FMT_Q6K) {
    decode_q6k_quarter(raw, r, 2 * h, o);
    decode_q6k_quarter(raw, r, 2 * h + 1, o + 8);
  } else {
    const int rt = r >> 5, lane = r & 31;
    const uint4 cw = *reinterpret_cast<const uint4*>(raw + ((rt * F::CH + h) * 32 + lane) * 16);
    decode_word<FMT>(raw, r, 4 * h, cw.x, o);
    decode_word<FMT>(raw, r, 4 * h + 1, cw.y, o + 4);
    decode_word<FMT>(raw, r, 4 * h + 2, cw.z, o + 8);
    decode_word<FMT>(raw, r, 4 * h + 3, cw.w, o + 12);
  }
}

}  // namespace qg
