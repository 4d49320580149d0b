// Decode of one packed 128 x 64 weight tile into the tensor cores' bf16 operand layout
// (128-byte swizzled, K-major), shared by the dense and grouped prefill GEMMs.  Every
// decoded value is exact in bf16: E2M1 x a power-of-two or E4M3 block scale, and integer
// codes times the fp16/fp32 scale products, rounded once (TurboEXL3 article §4.1: the
// stage's weights are decoded into on-chip memory in the multiplier's fragment order).
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "qg_common.cuh"

namespace qg {

constexpr int kATileBytes = 128 * 128;  // 128 rows x 64 bf16

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Decode one thread's share of a stage: row r, inputs 32h..32h+31, as 16 bf16x2 words in
// input order (word i holds inputs 32h+2i (low half) and 32h+2i+1).
template <int FMT>
__device__ __forceinline__ void decode_regs(const uint8_t* raw, int r, int h, uint32_t (&o)[16]) {
  using F = Fmt<FMT>;
  const int rt = r >> 5, lane = r & 31;
  const uint4 cw = *reinterpret_cast<const uint4*>(raw + ((rt * F::CH + h) * 32 + lane) * 16);
  const uint32_t words[4] = {cw.x, cw.y, cw.z, cw.w};
  const uint8_t* sp = raw + F::TB + r * F::SB;
#pragma unroll
  for (int wi = 0; wi < 4; ++wi) {
    const uint32_t w = words[wi];
    float v[8];
    if (FMT == FMT_NVFP4 || FMT == FMT_MXFP4) {
      float S;
      if (FMT == FMT_NVFP4) {
        const int blk = 2 * h + (wi >> 1);
        const uint32_t sw = *reinterpret_cast<const uint32_t*>(sp);
        const float2 s01 = (blk >> 1) ? e4m3x2_f32<1>(sw) : e4m3x2_f32<0>(sw);
        S = (blk & 1) ? s01.y : s01.x;
      } else {
        S = e8m0_f32(sp[h]);
      }
      const uint32_t hb[4] = {e2m1x2_h2<0>(w), e2m1x2_h2<1>(w), e2m1x2_h2<2>(w), e2m1x2_h2<3>(w)};
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const float2 e = __half22float2(*reinterpret_cast<const __half2*>(&hb[b]));
        v[2 * b] = S * e.x;  // exact
        v[2 * b + 1] = S * e.y;
      }
    } else {
      uint32_t op[4];
      const uint32_t rw = rot8(w);
      if (FMT == FMT_MLX) {
        op[0] = i4_op_lo(w);
        op[1] = i4_op_hi(w);
        op[2] = i4_op_lo(rw);
        op[3] = i4_op_hi(rw);
      } else {
        const int quarter = 2 * h + (wi >> 1);
        const uint32_t hw = *reinterpret_cast<const uint32_t*>(raw + ((rt * 3 + 2) * 32 + lane) * 16 + quarter * 4);
        const uint32_t hh = q6k_hi_for(hw, wi & 1), hr = rot8(hh);
        op[0] = i6_op_lo(w, hh);
        op[1] = i6_op_hi(w, hh);
        op[2] = i6_op_lo(rw, hr);
        op[3] = i6_op_hi(rw, hr);
      }
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
      } else {
        const float sc = (float)(int8_t)sp[2 * h + (wi >> 1)];
        const float d = __half2float(*reinterpret_cast<const __half*>(raw + F::TB + 128 * F::SB + r * 2));
        const float ds = d * sc;
#pragma unroll
        for (int j = 0; j < 8; ++j) v[j] = ds * (code[j] - 32.0f);
      }
    }
    o[4 * wi] = pack_bf16x2(v[0], v[1]);
    o[4 * wi + 1] = pack_bf16x2(v[2], v[3]);
    o[4 * wi + 2] = pack_bf16x2(v[4], v[5]);
    o[4 * wi + 3] = pack_bf16x2(v[6], v[7]);
  }
}

// The same share written as four 16-byte chunks of the 128-byte swizzled K-major shared
// memory tile (chunk j of row r lives at (r/8)*1024 + (r%8)*128 + ((j ^ (r%8)) * 16)).
template <int FMT>
__device__ __forceinline__ void decode_stage(const uint8_t* raw, uint8_t* A, int r, int h) {
  uint32_t o[16];
  decode_regs<FMT>(raw, r, h, o);
#pragma unroll
  for (int wi = 0; wi < 4; ++wi) {
    const int j = 4 * h + wi;
    *reinterpret_cast<uint4*>(A + (r >> 3) * 1024 + (r & 7) * 128 + ((j ^ (r & 7)) << 4)) =
        make_uint4(o[4 * wi], o[4 * wi + 1], o[4 * wi + 2], o[4 * wi + 3]);
  }
}

}  // namespace qg
