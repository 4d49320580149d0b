// NVFP4 activation quantisation for the W4A4 mode (TurboEXL3 article §2.2: the
// activations are quantised to NVFP4 during the forward pass, one E4M3 scale per 16
// values, so both operands of the multiply are FP4).
//
// One thread per block of 16 consecutive values of a row: two 16-byte loads of bf16,
// the block's largest magnitude, its E4M3 scale, sixteen E2M1 codes (one 8-byte store),
// the scale byte, and the exact bf16 expansion E4M3(S) * E2M1(code) (two 16-byte stores)
// that a bf16 tensor-core or CUDA-core GEMM multiplies; the activation tensor scale is
// left for that GEMM's epilogue.  Consecutive threads take consecutive blocks of a row,
// so every warp reads one contiguous 1 KB span.  HBM-bound: 32 bytes in and 32 + 8 + 1
// bytes out per block.
//
// Every rounding decision is one fp32 operation rounded to nearest even, in this order:
// d6 = 6 * act_scale; r = amax / d6; S = E4M3(r) (nearest even, saturating at 448);
// den = E4M3(S) * act_scale; q = x / den (x * 0 when den is 0); code = E2M1(q) (nearest
// even, saturating at 6, with x's sign bit).
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
// the even code -- at each midpoint the comparison is strict where the lower neighbour's
// code is even (0.25, 1.25, 2.5, 5) and inclusive where the upper one's is (0.75, 1.75,
// 3.5) -- and 7 (6) above 5; bit 3 is q's sign bit.
__device__ __forceinline__ uint32_t e2m1_code(float q) {
  const float a = fabsf(q);
  const uint32_t c = (uint32_t)(a > 0.25f) + (uint32_t)(a >= 0.75f) + (uint32_t)(a > 1.25f) +
                     (uint32_t)(a >= 1.75f) + (uint32_t)(a > 2.5f) + (uint32_t)(a >= 3.5f) + (uint32_t)(a > 5.0f);
  return c | ((__float_as_uint(q) >> 31) << 3);
}

// fp32 bits of the E2M1 magnitude of code c (0..7): 0, 0.5, then (1 + m/2) * 2^(e-1).
__device__ __forceinline__ uint32_t e2m1_mag_bits(uint32_t c) {
  return c < 2 ? (c ? 0x3F000000u : 0u) : (((126u + (c >> 1)) << 23) | ((c & 1u) << 22));
}

__global__ void __launch_bounds__(kQThreads) quant_act_nvfp4_kernel(QuantArgs a) {
  // A GEMV launched next (programmatic serialisation) may start streaming its weights now;
  // it waits for this grid to complete before it reads the expansion.
  if (threadIdx.x == 0) pdl_launch_dependents();
  const float d6 = __fmul_rn(6.0f, a.act_scale);
  const int64_t total = a.m * a.kb;
  for (int64_t i = (int64_t)blockIdx.x * kQThreads + threadIdx.x; i < total; i += (int64_t)gridDim.x * kQThreads) {
    const int64_t row = i / a.kb, b = i - row * a.kb;
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
    uint32_t cw[2] = {0u, 0u};
    uint32_t ew[8];
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const float q = den > 0.0f ? __fdiv_rn(f[j], den) : f[j] * 0.0f;
      const uint32_t c = e2m1_code(q);
      cw[j >> 3] |= c << (4 * (j & 7));
      // sf * magnitude has at most 6 significant bits: exact in fp32, and its low 16 bits
      // are zero, so the top half is the bf16 value itself
      const uint32_t e = __float_as_uint(__fmul_rn(sf, __uint_as_float(e2m1_mag_bits(c & 7u)))) | ((c >> 3) << 31);
      if (j & 1)
        ew[j >> 1] |= e & 0xFFFF0000u;
      else
        ew[j >> 1] = e >> 16;
    }
    if (a.codes) *reinterpret_cast<uint2*>(a.codes + row * a.ldc + b * 8) = make_uint2(cw[0], cw[1]);
    if (a.scales) a.scales[row * a.lds + b] = (uint8_t)s;
    if (a.xe) {
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
  quant_act_nvfp4_kernel<<<(unsigned)blocks, kQThreads, 0, static_cast<cudaStream_t>(stream)>>>(a);
  return cudaGetLastError() == cudaSuccess ? QG_OK : QG_ERR_CUDA;
}

}  // namespace qg
