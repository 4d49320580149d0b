// Device-side building blocks shared by the kernels of the quantized GEMV / GEMM
// library: format traits of the packed "T128x64" layout, streaming loads, and the
// in-register decoders that turn packed codes into fp32 operands.
//
// Decoders (TurboEXL3 article §2.1 formats; Q6_K operand PR #19, "What changed"):
//  * E2M1 (MXFP4, NVFP4): the hardware e2m1x2 -> f16x2 conversion, then f16 -> f32;
//    every E2M1 value is exact in f16 and f32.
//  * Integer codes (MLX affine, Q6_K): the zero point and the integer-to-float
//    conversion live in the operand's bit pattern.  The code is placed in the
//    mantissa of 1.0f, giving the exact operand 1 + code * 2^-11 (code in bits
//    12..) or 1 + code * 2^-7 (code in bits 16..); the constant 1 is removed once
//    per block with the block's input sums.  This is the fp32 form of the PR's
//    half operand 1 + code/64, whose offset is removed by subtracting 1.5.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace qg {

enum : int { FMT_MLX = 1, FMT_MXFP4 = 2, FMT_NVFP4 = 3, FMT_Q6K = 4 };

template <int FMT> struct Fmt;
template <> struct Fmt<FMT_MLX>   { static constexpr int TB = 4096, CH = 2, SB = 4; };
template <> struct Fmt<FMT_MXFP4> { static constexpr int TB = 4096, CH = 2, SB = 2; };
template <> struct Fmt<FMT_NVFP4> { static constexpr int TB = 4096, CH = 2, SB = 4; };
template <> struct Fmt<FMT_Q6K>   { static constexpr int TB = 6144, CH = 3, SB = 4; };

// ------------------------------------------------------------------ loads
// Weight stream: read once, never reused by this SM -> no L1 allocation.
__device__ __forceinline__ uint4 ld_stream16(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}
__device__ __forceinline__ uint32_t ld_stream4(const void* p) {
  uint32_t v;
  asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}
__device__ __forceinline__ uint32_t ld_stream2(const void* p) {
  unsigned short v;
  asm volatile("ld.global.nc.L1::no_allocate.u16 %0, [%1];" : "=h"(v) : "l"(p));
  return v;
}

// ------------------------------------------------------------------ decoders
// Two E2M1 codes (low nibble, high nibble of byte `b` of `wd`) -> fp32 pair (lo, hi).
template <int b>
__device__ __forceinline__ float2 e2m1x2_f32(uint32_t wd) {
  uint32_t h2;
  asm("{\n\t.reg .b8 t;\n\tcvt.u8.u32 t, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, t;\n\t}"
      : "=r"(h2) : "r"(wd >> (8 * b)));
  __half2 h = *reinterpret_cast<__half2*>(&h2);
  return __half22float2(h);
}

// Two E4M3FN bytes (bytes 2i, 2i+1 of `wd`) -> fp32 pair; exact (E4M3 fits f16).
template <int i>
__device__ __forceinline__ float2 e4m3x2_f32(uint32_t wd) {
  uint32_t h2;
  asm("{\n\t.reg .b16 t;\n\tcvt.u16.u32 t, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, t;\n\t}"
      : "=r"(h2) : "r"(wd >> (16 * i)));
  __half2 h = *reinterpret_cast<__half2*>(&h2);
  return __half22float2(h);
}

// E8M0 byte -> 2^(E-127) as fp32 (E = 0 is the subnormal 2^-127, E = 255 is NaN).
__device__ __forceinline__ float e8m0_f32(uint32_t e) {
  e &= 0xFFu;
  uint32_t bits = e ? (e << 23) : 0x00400000u;
  if (e == 0xFFu) bits = 0x7FC00000u;
  return __uint_as_float(bits);
}

// Byte rotations of a 32-bit word (one PRMT each).
__device__ __forceinline__ uint32_t rot8(uint32_t w)  { return __byte_perm(w, w, 0x0321); }
__device__ __forceinline__ uint32_t rot16(uint32_t w) { return __byte_perm(w, w, 0x1032); }
__device__ __forceinline__ uint32_t rot24(uint32_t w) { return __byte_perm(w, w, 0x2103); }

// Integer-code operands.  For a word holding eight 4-bit codes n0..n7 (nibble i at
// bits 4i..4i+3), rotation by 8r bits brings nibbles (3+2r)%8 to bits 12..15 and
// (4+2r)%8 to bits 16..19.  The operand pair is
//   x: 1 + n_odd  * 2^-11   (odd nibble, "class 12")
//   y: 1 + n_even * 2^-7    (even nibble, "class 16")
// Pair order over r = 0..3: (n3,n4) (n5,n6) (n7,n0) (n1,n2); the activations are
// staged in the matching order [3,4,5,6,7,0,1,2] within each group of eight.
// For Q6_K the two high bits of each code sit just above the nibble (bits 16..17
// for class 12, 20..21 for class 16) and `hi` supplies them after the same rotation.
__device__ __forceinline__ float2 int4_pair(uint32_t rotated) {
  return make_float2(__uint_as_float((rotated & 0x0000F000u) | 0x3F800000u),
                     __uint_as_float((rotated & 0x000F0000u) | 0x3F800000u));
}
__device__ __forceinline__ float2 int6_pair(uint32_t rot_lo, uint32_t rot_hi) {
  return make_float2(__uint_as_float((rot_lo & 0x0000F000u) | (rot_hi & 0x00030000u) | 0x3F800000u),
                     __uint_as_float((rot_lo & 0x000F0000u) | (rot_hi & 0x00300000u) | 0x3F800000u));
}
// Scale factors that turn (operand - 1) back into the integer code.
constexpr float kClass12 = 2048.0f;  // 2^11
constexpr float kClass16 = 128.0f;   // 2^7

// Q6_K high-bit word for the low-nibble word `half` (0: codes 16w..16w+7, 1: codes
// 16w+8..16w+15) of the layout's chunk-2 word: after this shift, the high bits of
// the code in nibble i of the low word sit at bits 4i+4..4i+5 (mod 32), so the same
// byte rotations align them above the rotated nibble.
__device__ __forceinline__ uint32_t q6k_hi_for(uint32_t hw, int half) {
  return half ? __funnelshift_l(hw, hw, 2) : __funnelshift_l(hw, hw, 4);
}

__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }

}  // namespace qg
