// NVFP4 activation quantisation for the W4A4 mode (TurboEXL3 article §2.2: the
// activations are quantised to NVFP4 during the forward pass, one E4M3 scale per 16
// values, so both operands of the multiply are FP4).
//
// One thread per block of 16 consecutive values of a row: two 16-byte loads of bf16,
// the block's largest magnitude, its E4M3 scale, sixteen E2M1 codes (one 8-byte store),
// the scale byte, and the exact bf16 expansion E4M3(S) * E2M1(code) (two 16-byte stores)
// that a bf16 tensor-core or CUDA-core GEMM multiplies; the activation tensor scale is
// left for that GEMM's epilogue.  Consecutive threads take consecutive blocks of a row,
// so every warp reads one contiguous 1 KB span.  Memory traffic: 32 bytes in and
// 32 + 8 + 1 bytes out per block; the arithmetic below, not HBM, sets the pace.
//
// Every rounding decision is one fp32 operation rounded to nearest even, in this order:
// d6 = 6 * act_scale; r = amax / d6; S = E4M3(r) (nearest even, saturating at 448);
// den = E4M3(S) * act_scale; q = x / den (x * 0 when den is 0); code = E2M1(q) (nearest
// even, saturating at 6, with x's sign bit).
//
// The ALU pipe bounds the kernel, so the sixteen divisions of a block are
// replaced by one reciprocal and sixteen products, without changing a single code:
// q' = RN(x * RN(1/den)) lies within 2 ulps of x/den (two roundings), and every value at
// which E2M1's nearest-even rounding changes its code -- 0.25, 0.75, 1.25, 1.75, 2.5,
// 3.5, 5 -- has at most 3 significant bits, so the low 21 mantissa bits of each are zero.
// Unless q' lies within 8 ulps of such a value, q' and the correctly rounded quotient
// are on the same side of every decision point and give the same code; the few that do
// (exact ties and their neighbours among them) are divided exactly, as are an infinite or
// NaN q' (a reciprocal that overflowed: low mantissa bits zero).  When den is a normal
// power of two (or 0, where q' = x * 0 as q), q' is already the correctly rounded quotient.
// The codes themselves come from the hardware's nearest-even E2M1 conversion, four
// instructions for eight values; the bf16 expansion is computed only when it is asked for.
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <stdint.h>

#include <algorithm>

#include "qg_internal.h"
#include "qg_sync.cuh"

namespace qg {
namespace {

constexpr int kQThreads = 256;

struct QuantArgs {
  const uint16_t* x;
  int64_t ldx, m, kb;
  float act_scale;
  uint8_t* codes;
  int64_t ldc;
  uint8_t* scales;
  int64_t lds;
  uint16_t* xe;
  int64_t lde;
};

// Value of a non-negative E4M3FN byte (bias 7; exponent field 0 is subnormal, 2^-9 steps).
__device__ __forceinline__ float e4m3_pos_value(uint32_t b) {
  const uint32_t e = (b >> 3) & 15u, mt = b & 7u;
  return e ? __uint_as_float(((e + 120u) << 23) | (mt << 20)) : (float)mt * 0x1p-9f;
}

// E2M1 code of q: the magnitude nearest |q| among 0, 0.5, 1, 1.5, 2, 3, 4, 6 with ties to
// the even code, saturating at 6; bit 3 is q's sign bit.  Below 1 the grid has step 1/2:
// 2^23 + 2|q| rounded once to fp32 is 2^23 + the nearest-even integer to 2|q| (0, 1 or 2
// = codes 0, 0.5, 1.0).  From 1 up the grid keeps one mantissa bit: adding 2^21 - 1 plus
// that bit to the fp32 bits rounds the mantissa to it, nearest even, and bits 22..30
// (exponent, kept bit) then count codes from 252 up, clamped at 7.
__device__ __forceinline__ uint32_t e2m1_code(float q) {
  const float a = fabsf(q);
  const uint32_t ua = __float_as_uint(a);
  const uint32_t lo = __float_as_uint(__fmaf_rn(a, 2.0f, 0x1p23f)) & 3u;
  const uint32_t hi = min(7u, ((ua + 0x1FFFFFu + ((ua >> 22) & 1u)) >> 22) - 252u);
  return (a < 1.0f ? lo : hi) | ((__float_as_uint(q) >> 31) << 3);
}

// True when the fp32 value q lies within 8 ulps of a number whose low 21 mantissa bits are
// zero -- among them every E2M1 decision point.
__device__ __forceinline__ bool near_decision(float q) {
  return ((__float_as_uint(q) + 8u) & 0x1FFFFFu) <= 16u;
}

// E2M1 codes of eight values q[0..7] as one word (value i in bits 4i..4i+3), by the
// hardware conversion: round to nearest even on the E2M1 grid, saturating at 6, the sign
// kept -- the same decision e2m1_code takes for every number (NaN excepted: the caller
// takes e2m1_code for a block with a NaN quotient).
__device__ __forceinline__ uint32_t e2m1x8_cvt(const float* q) {
  uint32_t w;
  asm("{\n\t.reg .b8 c0, c1, c2, c3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 c0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 c1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 c2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 c3, %8, %7;\n\t"
      "mov.b32 %0, {c0, c1, c2, c3};\n\t}"
      : "=r"(w)
      : "f"(q[0]), "f"(q[1]), "f"(q[2]), "f"(q[3]), "f"(q[4]), "f"(q[5]), "f"(q[6]), "f"(q[7]));
  return w;
}

// fp32 bits of the E2M1 magnitude of code c (0..7): 0, 0.5, then (1 + m/2) * 2^(e-1).
__device__ __forceinline__ uint32_t e2m1_mag_bits(uint32_t c) {
  return c < 2 ? (c ? 0x3F000000u : 0u) : (((126u + (c >> 1)) << 23) | ((c & 1u) << 22));
}

template <bool XE>  // XE: also write the bf16 expansion
__global__ void __launch_bounds__(kQThreads) quant_act_nvfp4_kernel(QuantArgs a) {
  // A GEMV launched next (programmatic serialisation) may start streaming its weights now;
  // it waits for this grid to complete before it reads the expansion.
  if (threadIdx.x == 0) pdl_launch_dependents();
  const float d6 = __fmul_rn(6.0f, a.act_scale);
  const uint32_t total = (uint32_t)(a.m * a.kb), kb = (uint32_t)a.kb;  // the host keeps it below 2^31
  for (uint32_t i = blockIdx.x * kQThreads + threadIdx.x; i < total; i += gridDim.x * kQThreads) {
    const int64_t row = i / kb, b = i - (uint32_t)row * kb;
    const uint4* src = reinterpret_cast<const uint4*>(a.x + row * a.ldx + b * 16);
    const uint4 v0 = __ldcs(src), v1 = __ldcs(src + 1);  // read once: do not keep in L2
    const uint32_t u[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
    float f[16];
    float amax = 0.0f;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      f[2 * j] = __uint_as_float(u[j] << 16);
      f[2 * j + 1] = __uint_as_float(u[j] & 0xFFFF0000u);
      amax = fmaxf(amax, fmaxf(fabsf(f[2 * j]), fabsf(f[2 * j + 1])));
    }
    const uint32_t s = (uint32_t)__nv_cvt_float_to_fp8(__fdiv_rn(amax, d6), __NV_SATFINITE, __NV_E4M3);
    const float sf = e4m3_pos_value(s);
    const float den = __fmul_rn(sf, a.act_scale);
    const float rcp = den > 0.0f ? __frcp_rn(den) : 0.0f;  // den == 0: q' = x * 0, as q
    // a normal power of two has an exact reciprocal: then q' is x / den rounded once
    const bool exact = (__float_as_uint(den) & 0x7FFFFFu) == 0u;
    float q[16];
    bool nan = false;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      q[j] = __fmul_rn(f[j], rcp);
      if (!exact && near_decision(q[j])) q[j] = __fdiv_rn(f[j], den);
      nan |= q[j] != q[j];
    }
    uint32_t cw[2] = {e2m1x8_cvt(q), e2m1x8_cvt(q + 8)};
    if (nan) {  // a NaN input: the software encoder's saturating code
      cw[0] = cw[1] = 0u;
#pragma unroll
      for (int j = 0; j < 16; ++j) cw[j >> 3] |= e2m1_code(q[j]) << (4 * (j & 7));
    }
    uint32_t ew[8];
    if (XE) {
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const uint32_t c = (cw[j >> 3] >> (4 * (j & 7))) & 15u;
        // sf * magnitude has at most 6 significant bits: exact in fp32, and its low 16 bits
        // are zero, so the top half is the bf16 value itself
        const uint32_t e = __float_as_uint(__fmul_rn(sf, __uint_as_float(e2m1_mag_bits(c & 7u)))) | ((c >> 3) << 31);
        if (j & 1)
          ew[j >> 1] |= e & 0xFFFF0000u;
        else
          ew[j >> 1] = e >> 16;
      }
    }
    if (a.codes) *reinterpret_cast<uint2*>(a.codes + row * a.ldc + b * 8) = make_uint2(cw[0], cw[1]);
    if (a.scales) a.scales[row * a.lds + b] = (uint8_t)s;
    if (XE) {
      uint4* dst = reinterpret_cast<uint4*>(a.xe + row * a.lde + b * 16);
      dst[0] = make_uint4(ew[0], ew[1], ew[2], ew[3]);
      dst[1] = make_uint4(ew[4], ew[5], ew[6], ew[7]);
    }
  }
}

}  // namespace

int launch_quant_act_nvfp4(const void* x, int64_t m, int64_t k, int64_t ldx, float act_scale, uint8_t* codes,
                           int64_t ldc, uint8_t* scales, int64_t lds, void* xe, int64_t lde, void* stream) {
  QuantArgs a;
  a.x = static_cast<const uint16_t*>(x);
  a.ldx = ldx;
  a.m = m;
  a.kb = k / 16;
  a.act_scale = act_scale;
  a.codes = codes;
  a.ldc = ldc;
  a.scales = scales;
  a.lds = lds;
  a.xe = static_cast<uint16_t*>(xe);
  a.lde = lde;
  const int64_t blocks = std::min<int64_t>((m * a.kb + kQThreads - 1) / kQThreads, (int64_t)1 << 20);
  if (xe)
    quant_act_nvfp4_kernel<true><<<(unsigned)blocks, kQThreads, 0, static_cast<cudaStream_t>(stream)>>>(a);
  else
    quant_act_nvfp4_kernel<false><<<(unsigned)blocks, kQThreads, 0, static_cast<cudaStream_t>(stream)>>>(a);
  return cudaGetLastError() == cudaSuccess ? QG_OK : QG_ERR_CUDA;
}

}  // namespace qg
