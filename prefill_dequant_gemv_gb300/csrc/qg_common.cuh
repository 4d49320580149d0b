// Device-side building blocks shared by the kernels of the quantized GEMV / GEMM
// library: format traits of the packed "T128x64" layout, streaming loads, and the
// in-register decoders that turn packed codes into exact f16 operands.
//
// Decoders (TurboEXL3 article §2.1 formats; Q6_K operand PR #19, "What changed"):
//  * E2M1 (MXFP4, NVFP4): the hardware e2m1x2 -> f16x2 conversion; every E2M1 value
//    is exact in f16.
//  * Integer codes (MLX affine, Q6_K): the zero point and the integer-to-float
//    conversion live in the operand's bit pattern.  The code is placed in the
//    mantissa of 1.0 (f16), giving the exact operand 1 + code/1024, 1 + code/256 or
//    1 + code/64; the constant 1 (and Q6_K's zero point 32) is removed once per block
//    with the block's input sums instead of once per weight.  This is the PR's half
//    operand 1 + code/64, whose offset the PR removes by subtracting 1.5; Q6_K keeps
//    its 6-bit codes byte-aligned so that most operands take one mask.
//  * 5-bit codes (Q5_0, Q5_1, Q5_K; the PR's 5-bit nibble operand): the nibble with
//    the fifth bit just above it, 1 + code/1024 or 1 + code/64 (exact for codes to 31);
//    zero points and minimums are a per-block affine term, as for MLX.
// Products are formed with the mixed-precision FMA f32 += f16 * f16 (exact
// products, fp32 accumulation).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace qg {

enum : int { FMT_MLX = 1, FMT_MXFP4 = 2, FMT_NVFP4 = 3, FMT_Q6K = 4, FMT_Q50 = 5, FMT_Q51 = 6, FMT_Q5K = 7 };

// TB: code bytes per 128 x 64 tile; CH: 512-byte chunks per 32 rows (the 5-bit formats'
// fifth-bit plane follows the two nibble chunks at byte kQ5Plane); SB: scale bytes per row.
template <int FMT> struct Fmt;
template <> struct Fmt<FMT_MLX>   { static constexpr int TB = 4096, CH = 2, SB = 4; };
template <> struct Fmt<FMT_MXFP4> { static constexpr int TB = 4096, CH = 2, SB = 2; };
template <> struct Fmt<FMT_NVFP4> { static constexpr int TB = 4096, CH = 2, SB = 4; };
template <> struct Fmt<FMT_Q6K>   { static constexpr int TB = 6144, CH = 3, SB = 4; };
template <> struct Fmt<FMT_Q50>   { static constexpr int TB = 5120, CH = 2, SB = 4; };
template <> struct Fmt<FMT_Q51>   { static constexpr int TB = 5120, CH = 2, SB = 8; };
template <> struct Fmt<FMT_Q5K>   { static constexpr int TB = 5120, CH = 2, SB = 3; };
constexpr int kQ5Plane = 4096;  // 5-bit formats: word j of row r at kQ5Plane + 512 j + 4 r

__host__ __device__ constexpr bool fmt_q5(int f) { return f == FMT_Q50 || f == FMT_Q51 || f == FMT_Q5K; }
// Integer codes (decoded through the operand classes below) rather than E2M1.
__host__ __device__ constexpr bool fmt_int(int f) { return f == FMT_MLX || f == FMT_Q6K || fmt_q5(f); }
// Aux bytes per row tile and 256 inputs (four tiles): Q6_K fp16 d, Q5_K fp16 (d, dmin).
__host__ __device__ constexpr int fmt_aux(int f) { return f == FMT_Q6K ? 256 : f == FMT_Q5K ? 512 : 0; }
// Aux bytes of one row inside that record.
__host__ __device__ constexpr int fmt_aux_row(int f) { return f == FMT_Q6K ? 2 : f == FMT_Q5K ? 4 : 0; }

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


// ---------------------------------------------------------------- f16 operands
// Mixed-precision FMA: c + a.half * b.half in fp32 (the f16 x f16 product is exact
// in fp32, so this equals an fp32 FMA of the two exact operands).
__device__ __forceinline__ float hfma_lo(uint32_t a, uint32_t b, float c) {
  float d;
  asm("{\n\t.reg .b16 al, ah, bl, bh;\n\tmov.b32 {al, ah}, %1;\n\tmov.b32 {bl, bh}, %2;\n\t"
      "fma.rn.f32.f16 %0, al, bl, %3;\n\t}" : "=f"(d) : "r"(a), "r"(b), "f"(c));
  return d;
}
__device__ __forceinline__ float hfma_hi(uint32_t a, uint32_t b, float c) {
  float d;
  asm("{\n\t.reg .b16 al, ah, bl, bh;\n\tmov.b32 {al, ah}, %1;\n\tmov.b32 {bl, bh}, %2;\n\t"
      "fma.rn.f32.f16 %0, ah, bh, %3;\n\t}" : "=f"(d) : "r"(a), "r"(b), "f"(c));
  return d;
}

// Two E2M1 codes (byte b of wd) -> f16x2 (low nibble in the low half); exact.  The word is
// split into its four bytes with one vector move, which the conversion reads in place
// (measured on this GPU: 85 against 57 weights per clock per SM for shifting each byte
// down to bit 0 first, the same results bit for bit).
template <int b>
__device__ __forceinline__ uint32_t e2m1x2_h2(uint32_t wd) {
  static_assert(b >= 0 && b < 4, "byte index");
  uint32_t h2;
  if (b == 0)
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, b0;\n\t}"
        : "=r"(h2) : "r"(wd));
  else if (b == 1)
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, b1;\n\t}"
        : "=r"(h2) : "r"(wd));
  else if (b == 2)
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, b2;\n\t}"
        : "=r"(h2) : "r"(wd));
  else
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, b3;\n\t}"
        : "=r"(h2) : "r"(wd));
  return h2;
}

// Integer codes as exact f16 operands (the Q6_K operand PR's zero-point-in-the-
// operand idea: the code sits in the mantissa of 1.0).  For a word of eight 4-bit
// codes n0..n7 (nibble i at bits 4i..4i+3) and r = the word rotated right by 8:
//   op0 = halves (n0, n4) = 1 + n/1024   (mantissa bits 0..3,  "class 1024")
//   op1 = halves (n1, n5) = 1 + n/64     (mantissa bits 4..7,  "class 64")
//   op2 = halves (n2, n6) from r, class 1024;  op3 = halves (n3, n7) from r, class 64.
// Activations of class-1024 positions are staged multiplied by 16, so every
// product is 16*x + code*x/64 (class 1024) or x + code*x/64 (class 64): one
// accumulator, and the constants are removed per block with precomputed sums.
__device__ __forceinline__ uint32_t i4_op_lo(uint32_t w) { return (w & 0x000F000Fu) | 0x3C003C00u; }
__device__ __forceinline__ uint32_t i4_op_hi(uint32_t w) { return (w & 0x00F000F0u) | 0x3C003C00u; }
// Q6_K (zero point 32 in the operand, as the PR does, with byte-aligned codes): a tile row's
// 16-input quarter is three 32-bit words; byte j of word c holds the code of input 4c + j in
// bits 2..7 and bits 2c..2c+1 of the code of input 12 + j in bits 0..1.  Word c of quarter
// kq of row (rt, lane) sits at q6k_word_offset(rt, kq, c, lane): a warp reads 128 bytes.
__host__ __device__ constexpr int q6k_word_offset(int rt, int kq, int c, int lane) {
  return ((rt * 4 + kq) * 3 + c) * 128 + lane * 4;
}
// The quarter's eight operands: (x0,x2) (x1,x3) (x4,x6) (x5,x7) (x8,x10) (x9,x11) are
// 1 + code/256 (the code in mantissa bits 2..7, straight from the word or its byte
// rotation), (x12,x14) (x13,x15) are 1 + code/1024 (the code gathered from the three words'
// low bit pairs into mantissa bits 0..5).
__device__ __forceinline__ void q6k_ops(uint32_t w0, uint32_t w1, uint32_t w2, uint32_t (&op)[8]) {
  constexpr uint32_t K = 0x3C003C00u, M6 = 0x00FC00FCu, M2 = 0x03030303u;
  op[0] = (w0 & M6) | K;
  op[1] = (rot8(w0) & M6) | K;
  op[2] = (w1 & M6) | K;
  op[3] = (rot8(w1) & M6) | K;
  op[4] = (w2 & M6) | K;
  op[5] = (rot8(w2) & M6) | K;
  const uint32_t t = (w0 & M2) + (w1 & M2) * 4u + (w2 & M2) * 16u;  // disjoint fields: + is |
  op[6] = (t & 0x003F003Fu) | K;
  op[7] = (rot8(t) & 0x003F003Fu) | K;
}

// 5-bit codes: the fifth bit sits just above its nibble (bit 4 for class 1024, bit 8 for
// class 64: the PR's "fifth bit at bit 8 of each halfword").  The layout stores the fifth
// bit of input 8u + i of a 32-input half at bit (4i + 4 + u) mod 32 of the row's word, so
// rotating that word right by u (one funnel shift) puts code i's bit at 4i + 4.
__device__ __forceinline__ uint32_t q5_hi_for(uint32_t hw, int u) { return __funnelshift_r(hw, hw, u & 3); }
__device__ __forceinline__ uint32_t i5_op_lo(uint32_t w, uint32_t h) {
  return (w & 0x000F000Fu) | (h & 0x00100010u) | 0x3C003C00u;
}
__device__ __forceinline__ uint32_t i5_op_hi(uint32_t w, uint32_t h) {
  return (w & 0x00F000F0u) | (h & 0x01000100u) | 0x3C003C00u;
}

// The four operands of one code word of MLX affine or a 5-bit format: op0 = (n0, n4) and
// op2 = (n2, n6) of class 1024, op1 = (n1, n5) and op3 = (n3, n7) of class 64.  `h`: the
// fifth-bit word aligned for this code word (q5_hi_for); unused for MLX.
template <int FMT>
__device__ __forceinline__ void int_ops(uint32_t w, uint32_t h, uint32_t (&op)[4]) {
  static_assert(FMT == FMT_MLX || fmt_q5(FMT), "nibble-word formats only");
  const uint32_t r = rot8(w);
  if (FMT == FMT_MLX) {
    op[0] = i4_op_lo(w);
    op[1] = i4_op_hi(w);
    op[2] = i4_op_lo(r);
    op[3] = i4_op_hi(r);
  } else {
    const uint32_t hr = rot8(h);
    op[0] = i5_op_lo(w, h);
    op[1] = i5_op_hi(w, h);
    op[2] = i5_op_lo(r, hr);
    op[3] = i5_op_hi(r, hr);
  }
}

// Per-block affine map of the 5-bit formats, w = s * code + bias (GGML blocks):
//   Q5_0: s = d, bias = -16 d (the zero point as a minimum, "ZeroAsMin");
//   Q5_1: s = d, bias = m;  Q5_K: s = d * sc, bias = -(dmin * mn).
// sp: the row's SB scale bytes of the tile; ap: the row's aux record (Q5_K d, dmin);
// blk: the 32-input block of the tile (0, 1).  s and bias are exact in fp32.
template <int FMT>
__device__ __forceinline__ float2 q5_affine(const uint8_t* sp, const uint8_t* ap, int blk) {
  if (FMT == FMT_Q50) {
    const float d = __half2float(*reinterpret_cast<const __half*>(sp + 2 * blk));
    return make_float2(d, -16.0f * d);
  } else if (FMT == FMT_Q51) {
    const uint32_t v = *reinterpret_cast<const uint32_t*>(sp + 4 * blk);
    return make_float2(__half2float(__ushort_as_half((unsigned short)(v & 0xFFFFu))),
                       __half2float(__ushort_as_half((unsigned short)(v >> 16))));
  } else {
    const uint32_t v = ((uint32_t)sp[0] | ((uint32_t)sp[1] << 8) | ((uint32_t)sp[2] << 16)) >> (12 * blk);
    // 6-bit integers to float exactly: (2^23 + i) - 2^23, cheaper than an integer conversion
    const float sc = __uint_as_float(0x4B000000u | (v & 63u)) - 8388608.0f;
    const float mn = __uint_as_float(0x4B000000u | ((v >> 6) & 63u)) - 8388608.0f;
    const uint32_t dd = *reinterpret_cast<const uint32_t*>(ap);
    const float d = __half2float(__ushort_as_half((unsigned short)(dd & 0xFFFFu)));
    const float dmin = __half2float(__ushort_as_half((unsigned short)(dd >> 16)));
    return make_float2(d * sc, -(dmin * mn));
  }
}

// ---------------------------------------------------------------- MoE finish
// Weight of the shared expert's output for one token: its sigmoid gate
// 1 / (1 + e^-l) in fp32 from the gate logit l (TurboEXL3 article §4.2), or 1 when the
// caller passes no gate logits.
__device__ __forceinline__ float shared_gate_weight(const float* gate_logits, int t) {
  if (!gate_logits) return 1.0f;
  return 1.0f / (1.0f + expf(-gate_logits[t]));
}

}  // namespace qg
