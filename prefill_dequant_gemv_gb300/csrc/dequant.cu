// Debug / test dequantisation: packed "T128x64" weights -> dense fp32 or bf16.
//
// It runs the same in-register decoders as the GEMV (qg_common.cuh) and then turns
// each operand back into the weight, so a bit-exact comparison of its output with
// the CPU oracle checks the layout reader and every decoder of the fast path.
//   fp32: the exact weight rounded once (TurboEXL3 article §2.1 formats; Q6_K
//         operand PR #19 zero point 32 and its 5-bit formats).
//   bf16: the prefill tensor-core operand: e2m1 * block scale (without the NVFP4
//         tensor scale; exact in bf16) or the fp32 weight rounded to bf16.
#include <cuda_runtime.h>

#include "qg_common.cuh"
#include "qg_internal.h"

namespace qg {

struct DequantArgs {
  const uint8_t* codes;
  const uint8_t* scales;
  const uint8_t* aux;
  int64_t n, k, kg, items;
  float ts;
  void* out;
  int64_t ldo;
  int bf16;
};

template <int FMT>
__global__ void __launch_bounds__(256) dequant_kernel(const DequantArgs a) {
  using F = Fmt<FMT>;
  const int64_t it = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (it >= a.items) return;
  // item = (row n, group g, quarter kq)
  const int kq = (int)(it & 3);
  const int64_t g = (it >> 2) % a.kg;
  const int64_t n = (it >> 2) / a.kg;
  const int64_t q = n / 128;
  const int row = (int)(n % 128), rt = row / 32, lane = row % 32;
  const int64_t t = q * a.kg + g;
  const uint8_t* tc = a.codes + t * F::TB;
  const uint8_t* sp = a.scales + t * 128 * F::SB + row * F::SB;
  float w[16];
  if constexpr (FMT == FMT_Q6K) {  // one quarter: three words, eight operands (input pairs (4c, 4c+2), (4c+1, 4c+3))
    const uint8_t* qb = tc + q6k_word_offset(rt, kq, 0, lane);
    uint32_t op[8];
    q6k_ops(*reinterpret_cast<const uint32_t*>(qb), *reinterpret_cast<const uint32_t*>(qb + 128),
            *reinterpret_cast<const uint32_t*>(qb + 256), op);
    const float sc = (float)(int8_t)sp[kq];
    const float d = __half2float(*reinterpret_cast<const __half*>(a.aux + (q * (a.kg / 4) + g / 4) * 256 + row * 2));
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float2 e = __half22float2(*reinterpret_cast<const __half2*>(&op[j]));
      const float mul = j < 6 ? 256.0f : 1024.0f;
      const int base = (j >> 1) * 4 + (j & 1);
      w[base] = (d * sc) * ((e.x - 1.0f) * mul - 32.0f);
      w[base + 2] = (d * sc) * ((e.y - 1.0f) * mul - 32.0f);
    }
  } else {
  const uint2 v = *reinterpret_cast<const uint2*>(tc + ((rt * F::CH + (kq >> 1)) * 32 + lane) * 16 + (kq & 1) * 8);
#pragma unroll
  for (int wi = 0; wi < 2; ++wi) {
    const uint32_t wd = wi ? v.y : v.x;
    float* o = w + wi * 8;
    if constexpr (FMT == FMT_NVFP4 || FMT == FMT_MXFP4) {
      float S;
      if (FMT == FMT_NVFP4) {
        const uint32_t sw = *reinterpret_cast<const uint32_t*>(sp);
        const float2 s01 = (kq >> 1) ? e4m3x2_f32<1>(sw) : e4m3x2_f32<0>(sw);
        S = (kq & 1) ? s01.y : s01.x;
      } else {
        S = e8m0_f32(sp[kq >> 1]);
      }
      const uint32_t h[4] = {e2m1x2_h2<0>(wd), e2m1x2_h2<1>(wd), e2m1x2_h2<2>(wd), e2m1x2_h2<3>(wd)};
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const float2 e = __half22float2(*reinterpret_cast<const __half2*>(&h[b]));
        float lo = S * e.x, hi = S * e.y;  // exact: <= 6 significant bits
        if (!a.bf16 && FMT == FMT_NVFP4) {
          lo = a.ts * lo;
          hi = a.ts * hi;
        }
        o[2 * b] = lo;
        o[2 * b + 1] = hi;
      }
    } else {
      // the GEMV's f16 operands: op0 = (n0, n4) and op2 = (n2, n6) are 1 + code/1024,
      // op1 = (n1, n5) and op3 = (n3, n7) are 1 + code/64
      uint32_t op[4];
      uint32_t hh = 0;
      if (fmt_q5(FMT))
        hh = q5_hi_for(*reinterpret_cast<const uint32_t*>(tc + kQ5Plane + (kq >> 1) * 512 + row * 4),
                       2 * (kq & 1) + wi);
      int_ops<FMT>(wd, hh, op);
      float code[8];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 e = __half22float2(*reinterpret_cast<const __half2*>(&op[j]));
        const float mul = (j & 1) ? 64.0f : 1024.0f;
        code[j] = (e.x - 1.0f) * mul;  // exact
        code[j + 4] = (e.y - 1.0f) * mul;
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (FMT == FMT_MLX) {
          const uint32_t sw = *reinterpret_cast<const uint32_t*>(sp);
          const float s = __half2float(__ushort_as_half((unsigned short)(sw & 0xFFFFu)));
          const float bias = __half2float(__ushort_as_half((unsigned short)(sw >> 16)));
          o[j] = fmaf(s, code[j], bias);
        } else if (fmt_q5(FMT)) {
          const float2 sb = q5_affine<FMT>(sp, a.aux + (q * (a.kg / 4) + g / 4) * fmt_aux(FMT) + row * fmt_aux_row(FMT),
                                           kq >> 1);
          o[j] = fmaf(sb.x, code[j], sb.y);  // one rounding of the exact value
        } else {
          const float sc = (float)(int8_t)sp[kq];
          const float d = __half2float(*reinterpret_cast<const __half*>(a.aux + (q * (a.kg / 4) + g / 4) * 256 + row * 2));
          o[j] = (d * sc) * (code[j] - 32.0f);
        }
      }
    }
  }
  }
  if (n >= a.n) return;
  const int64_t k0 = g * 64 + kq * 16;
  if (k0 >= a.k) return;
  if (a.bf16) {
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out) + n * a.ldo + k0;
#pragma unroll
    for (int i = 0; i < 16; ++i) out[i] = __float2bfloat16_rn(w[i]);
  } else {
    float* out = static_cast<float*>(a.out) + n * a.ldo + k0;
#pragma unroll
    for (int i = 0; i < 16; ++i) out[i] = w[i];
  }
}

int launch_dequant(const Geometry& g, const qg_weight* w, int out_dtype, void* out, int64_t ldo, void* stream) {
  DequantArgs a;
  a.codes = static_cast<const uint8_t*>(w->codes);
  a.scales = static_cast<const uint8_t*>(w->scales);
  a.aux = static_cast<const uint8_t*>(w->aux);
  a.n = g.n;
  a.k = g.k;
  a.kg = g.kg;
  a.items = g.np * g.kg * 4;
  a.ts = (g.fmt == FMT_NVFP4) ? w->tensor_scale : 1.0f;
  a.out = out;
  a.ldo = ldo;
  a.bf16 = out_dtype == QG_OUT_BF16;
  const int threads = 256;
  const int64_t blocks = (a.items + threads - 1) / threads;
  if (blocks > 0x7FFFFFFF) return QG_ERR_UNSUPPORTED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  switch (g.fmt) {
    case FMT_MLX: dequant_kernel<FMT_MLX><<<(unsigned)blocks, threads, 0, s>>>(a); break;
    case FMT_MXFP4: dequant_kernel<FMT_MXFP4><<<(unsigned)blocks, threads, 0, s>>>(a); break;
    case FMT_NVFP4: dequant_kernel<FMT_NVFP4><<<(unsigned)blocks, threads, 0, s>>>(a); break;
    case FMT_Q50: dequant_kernel<FMT_Q50><<<(unsigned)blocks, threads, 0, s>>>(a); break;
    case FMT_Q51: dequant_kernel<FMT_Q51><<<(unsigned)blocks, threads, 0, s>>>(a); break;
    case FMT_Q5K: dequant_kernel<FMT_Q5K><<<(unsigned)blocks, threads, 0, s>>>(a); break;
    default: dequant_kernel<FMT_Q6K><<<(unsigned)blocks, threads, 0, s>>>(a); break;
  }
  return cudaGetLastError() == cudaSuccess ? QG_OK : QG_ERR_CUDA;
}

}  // namespace qg
