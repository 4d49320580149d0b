// GEMV building blocks shared by the dense and the grouped (mixture-of-experts)
// quantized GEMV kernels: pipeline-stage geometry, activation staging as exact f16,
// and the per-quarter decode + mixed-precision FMA + block-scale fold.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "qg_common.cuh"

namespace qg {

// Consumer warps: 16 for 1-3 rows (96 registers a thread); 12 for 4 rows, whose
// accumulators and activations need the 128 registers a 13-warp CTA allows (warps are
// allocated in groups of four).
__host__ __device__ constexpr int consumer_warps(int m) { return m >= 4 ? 12 : 16; }
// The dense GEMV multiplies the E2M1 formats on the tensor cores (consume_mma) from
// kMmaMinRows activation rows on; its few accumulators leave room for 16 consumer warps.
constexpr int kMmaMinRows = 2;
__host__ __device__ constexpr bool gemv_mma(int fmt, int m) {
  return (fmt == FMT_NVFP4 || fmt == FMT_MXFP4) && m >= kMmaMinRows;
}
__host__ __device__ constexpr int gemv_warps(int fmt, int m) { return gemv_mma(fmt, m) ? 16 : consumer_warps(m); }
constexpr int kMaxStages = 48;

// One pipeline stage holds a chunk of C consecutive units (tile index = unit index,
// so a chunk is one contiguous range of codes and one of scales): a single bulk
// copy per array per chunk keeps the copy engine at HBM speed, which 4-6 KB
// copies do not reach.
template <int FMT> struct Stage {
  static constexpr int CODE = Fmt<FMT>::TB;            // per unit
  static constexpr int SCALE = 128 * Fmt<FMT>::SB;     // per unit
  static constexpr int AUX = fmt_aux(FMT);             // per 4 units (Q6_K d, Q5_K d and dmin)
  // C consecutive units touch at most (C + 3) / 4 + 1 groups of four units' aux records
  __host__ __device__ static constexpr int bytes(int C) { return C * (CODE + SCALE) + ((C + 3) / 4 + 1) * AUX; }
};

__host__ __device__ inline int64_t owner_cta(int64_t u, int64_t U, int64_t G) {
  // CTA b owns units [b*U/G, (b+1)*U/G); the owner of u is the largest b with b*U/G <= u.
  return ((u + 1) * G - 1) / U;
}

__device__ __forceinline__ void bf16x2_to_f32(uint32_t v, float& lo, float& hi) {
  lo = __uint_as_float(v << 16);
  hi = __uint_as_float(v & 0xFFFF0000u);
}

// Stage 16 activations (eight bf16 pairs `u`) of one row as f16, exactly: the quarter is
// scaled by its own power of two 2^p chosen from its largest |x|, so each bf16 value
// (8 significant bits) lands inside f16's range; a value more than 2^27 below the
// quarter's maximum would round, far below the stated tolerance.  Writes the two 16-byte
// staging words to `dst` and returns the quarter's record {2^-p (E2M1) or 64 * 2^-p
// (integer formats), Z, X, 0}: Z, in scaled units, is the integer operands' constant part
// (for Q6_K also half the quarter's scaled sum, the zero point 32 / 64), so the fold
// subtracts it before anything leaves the scaled range; X is the quarter's sum in
// unscaled units (the affine formats' bias term).  Every product the fold forms is then
// within fp32's range whenever the true partial sum is, even for activations near bf16's
// largest values.
// Layout per 8 inputs (one code word): four f16x2 words in the order the decoder
// produces operand pairs -- E2M1: (x0,x1) (x2,x3) (x4,x5) (x6,x7); integer formats:
// (16x0,16x4) (x1,x5) (16x2,16x6) (x3,x7).
template <int FMT>
__device__ __forceinline__ float4 stage_quarter(const uint32_t (&u)[8], uint32_t* dst) {
  constexpr bool kInt = fmt_int(FMT);
  uint32_t mb = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) mb = max(mb, max(u[i] & 0x7FFFu, (u[i] >> 16) & 0x7FFFu));
  const int e = mb >= 0x80 ? (int)(mb >> 7) - 127 : -127;
  int p = (kInt ? 10 : 14) - e;
  if (mb >= 0x7F80u || mb == 0) p = 0;  // inf / nan / all zero: leave as is
  p = max(-126, min(126, p));
  const float scale = __uint_as_float((uint32_t)(p + 127) << 23);
  const float inv = __uint_as_float((uint32_t)(127 - p) << 23);
  float v[16];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    float lo, hi;
    bf16x2_to_f32(u[i], lo, hi);
    v[2 * i] = __half2float(__float2half_rn(lo * scale));
    v[2 * i + 1] = __half2float(__float2half_rn(hi * scale));
  }
  auto h2 = [](float lo, float hi) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  };
  float4 z = make_float4(inv, 0.0f, 0.0f, 0.0f);
  if (FMT == FMT_Q6K) {
    // operand order of q6k_ops: (x0,x2) (x1,x3) (x4,x6) (x5,x7) (x8,x10) (x9,x11) of class 256
    // (activations x4), (x12,x14) (x13,x15) of class 1024 (activations x16)
    const float* q = v;
    reinterpret_cast<uint4*>(dst)[0] = make_uint4(h2(4.0f * q[0], 4.0f * q[2]), h2(4.0f * q[1], 4.0f * q[3]),
                                                  h2(4.0f * q[4], 4.0f * q[6]), h2(4.0f * q[5], 4.0f * q[7]));
    reinterpret_cast<uint4*>(dst)[1] = make_uint4(h2(4.0f * q[8], 4.0f * q[10]), h2(4.0f * q[9], 4.0f * q[11]),
                                                  h2(16.0f * q[12], 16.0f * q[14]), h2(16.0f * q[13], 16.0f * q[15]));
    float x4 = 0.0f, x16 = 0.0f;
#pragma unroll
    for (int i = 0; i < 12; ++i) x4 += q[i];
#pragma unroll
    for (int i = 12; i < 16; ++i) x16 += q[i];
    const float xs = x4 + x16;                         // the quarter's scaled sum
    const float xop = fmaf(4.0f, x4, 16.0f * x16);     // the operands' constant part, scaled
    z.x = 64.0f * inv;
    z.y = fmaf(0.5f, xs, xop);  // and the zero point: 32 * sum / 64
    z.z = xs * inv;
  } else if (kInt) {
    float x16 = 0.0f, x1 = 0.0f;
#pragma unroll
    for (int w = 0; w < 2; ++w) {
      const float* q = v + 8 * w;
      reinterpret_cast<uint4*>(dst)[w] = make_uint4(h2(16.0f * q[0], 16.0f * q[4]), h2(q[1], q[5]),
                                                    h2(16.0f * q[2], 16.0f * q[6]), h2(q[3], q[7]));
      x16 += (q[0] + q[4]) + (q[2] + q[6]);
      x1 += (q[1] + q[5]) + (q[3] + q[7]);
    }
    z.x = 64.0f * inv;
    z.y = fmaf(16.0f, x16, x1);  // the operands' constant part, scaled
    z.z = (x16 + x1) * inv;      // X, unscaled
  } else {
#pragma unroll
    for (int i = 0; i < 2; ++i)
      reinterpret_cast<uint4*>(dst)[i] = make_uint4(h2(v[8 * i], v[8 * i + 1]), h2(v[8 * i + 2], v[8 * i + 3]),
                                                    h2(v[8 * i + 4], v[8 * i + 5]), h2(v[8 * i + 6], v[8 * i + 7]));
  }
  return z;
}

// One consumer warp, one unit, one 16-input quarter: accumulate 4 rows x M (of arrays
// sized MA >= M).  xr[m] points at row m's 8 staging words of this quarter, zr[m] at its
// record.
template <int FMT, int M, int MA = M>
__device__ __forceinline__ void consume(const uint8_t* st, const uint8_t* scl, const uint8_t* aux,
                                        const uint32_t* const (&xr)[MA], const float* const (&zr)[MA],
                                        const float* e4m3_lut, int kq, int lane, float (&acc)[4][MA]) {
  using F = Fmt<FMT>;
  uint32_t wd[4][2];
  uint32_t hw[4];
#pragma unroll
  for (int rt = 0; rt < 4; ++rt) {
    if (FMT != FMT_Q6K) {
      const uint2 v = *reinterpret_cast<const uint2*>(st + ((rt * F::CH + (kq >> 1)) * 32 + lane) * 16 + (kq & 1) * 8);
      wd[rt][0] = v.x;
      wd[rt][1] = v.y;
    }
    if (FMT == FMT_Q6K) {  // the row's three words of this quarter
      const uint8_t* qb = st + q6k_word_offset(rt, kq, 0, lane);
      wd[rt][0] = *reinterpret_cast<const uint32_t*>(qb);
      wd[rt][1] = *reinterpret_cast<const uint32_t*>(qb + 128);
      hw[rt] = *reinterpret_cast<const uint32_t*>(qb + 256);
    }
    if (fmt_q5(FMT))  // the row's fifth-bit word of this quarter's 32-input half
      hw[rt] = *reinterpret_cast<const uint32_t*>(st + kQ5Plane + (kq >> 1) * 512 + (rt * 32 + lane) * 4);
  }
  // Activations of the quarter for every row m (both code words), then one 32-row group
  // at a time: decode, accumulate, fold -- so only one group's partials are live.
  uint4 X[M][2];
#pragma unroll
  for (int m = 0; m < M; ++m) {
    X[m][0] = *reinterpret_cast<const uint4*>(xr[m]);
    X[m][1] = *reinterpret_cast<const uint4*>(xr[m] + 4);
  }
  float4 zq[M];
#pragma unroll
  for (int m = 0; m < M; ++m) zq[m] = *reinterpret_cast<const float4*>(zr[m]);
#pragma unroll
  for (int rt = 0; rt < 4; ++rt) {
    float P[M][2];
#pragma unroll
    for (int m = 0; m < M; ++m) P[m][0] = P[m][1] = 0.0f;
    uint32_t q6[8];
    if (FMT == FMT_Q6K) q6k_ops(wd[rt][0], wd[rt][1], hw[rt], q6);
#pragma unroll
    for (int wi = 0; wi < 2; ++wi) {
      const uint32_t w = wd[rt][wi];
      uint32_t o0, o1, o2, o3;
      if constexpr (FMT == FMT_Q6K) {
        o0 = q6[4 * wi];
        o1 = q6[4 * wi + 1];
        o2 = q6[4 * wi + 2];
        o3 = q6[4 * wi + 3];
      } else if constexpr (FMT == FMT_MXFP4 || FMT == FMT_NVFP4) {
        o0 = e2m1x2_h2<0>(w);
        o1 = e2m1x2_h2<1>(w);
        o2 = e2m1x2_h2<2>(w);
        o3 = e2m1x2_h2<3>(w);
      } else {
        uint32_t op[4];
        const uint32_t h = fmt_q5(FMT) ? q5_hi_for(hw[rt], 2 * (kq & 1) + wi) : 0u;
        int_ops<FMT>(w, h, op);
        o0 = op[0];
        o1 = op[1];
        o2 = op[2];
        o3 = op[3];
      }
#pragma unroll
      for (int m = 0; m < M; ++m) {
        const uint4 x = X[m][wi];
        float p0 = P[m][0], p1 = P[m][1];
        p0 = hfma_lo(o0, x.x, p0);
        p1 = hfma_hi(o0, x.x, p1);
        p0 = hfma_lo(o1, x.y, p0);
        p1 = hfma_hi(o1, x.y, p1);
        p0 = hfma_lo(o2, x.z, p0);
        p1 = hfma_hi(o2, x.z, p1);
        p0 = hfma_lo(o3, x.w, p0);
        p1 = hfma_hi(o3, x.w, p1);
        P[m][0] = p0;
        P[m][1] = p1;
      }
    }
    // Fold the quarter's partial with the block scale (once per block and row): the block
    // scale meets the scaled partial first and the power of two 2^-p last, so no product
    // leaves fp32's range unless the true partial sum does.
    const int row = rt * 32 + lane;
    const uint8_t* sp = scl + row * F::SB;
    if (FMT == FMT_NVFP4) {  // the table holds E4M3 x the tensor scale
      const float S = e4m3_lut[sp[kq]];
#pragma unroll
      for (int m = 0; m < M; ++m) acc[rt][m] = fmaf(S * (P[m][0] + P[m][1]), zq[m].x, acc[rt][m]);
    } else if (FMT == FMT_MXFP4) {
      const float S = e8m0_f32(sp[kq >> 1]);
#pragma unroll
      for (int m = 0; m < M; ++m) acc[rt][m] = fmaf(S * (P[m][0] + P[m][1]), zq[m].x, acc[rt][m]);
    } else if (FMT == FMT_MLX) {
      const uint32_t sw = *reinterpret_cast<const uint32_t*>(sp);
      const float s = __half2float(__ushort_as_half((unsigned short)(sw & 0xFFFFu)));
      const float bias = __half2float(__ushort_as_half((unsigned short)(sw >> 16)));
#pragma unroll
      for (int m = 0; m < M; ++m) {
        const float dot = (P[m][0] + P[m][1]) - zq[m].y;  // sum code * x / 64, scaled
        acc[rt][m] = fmaf(s * dot, zq[m].x, fmaf(bias, zq[m].z, acc[rt][m]));
      }
    } else if (FMT == FMT_Q6K) {
      const float sc = (float)(int8_t)sp[kq];
      const float d = __half2float(*reinterpret_cast<const __half*>(aux + row * 2));
      const float ds = d * sc;
#pragma unroll
      for (int m = 0; m < M; ++m) {
        const float dot = (P[m][0] + P[m][1]) - zq[m].y;  // sum (code - 32) * x / 64, scaled
        acc[rt][m] = fmaf(ds * dot, zq[m].x, acc[rt][m]);
      }
    } else {  // 5-bit: w = s * code + bias over the quarter's 32-input block
      const float2 sb = q5_affine<FMT>(sp, aux + row * fmt_aux_row(FMT), kq >> 1);
#pragma unroll
      for (int m = 0; m < M; ++m) {
        const float dot = (P[m][0] + P[m][1]) - zq[m].y;
        acc[rt][m] = fmaf(sb.x * dot, zq[m].x, fmaf(sb.y, zq[m].z, acc[rt][m]));
      }
    }
  }
}

// ---------------------------------------------------------------- tensor-core consumer
// Exponent p of the power of two 2^p that puts a token's largest |x| (bf16 magnitude bits
// `mb`, subnormals included) in [2^14, 2^15): the f16 staging scale of the tensor-core
// GEMV.  0 for an all-zero token or one holding inf or NaN (those propagate unscaled).
__device__ __forceinline__ int tok_exp(uint32_t mb) {
  if (mb == 0 || mb >= 0x7F80u) return 0;
  const int e = mb >= 0x80u ? (int)(mb >> 7) - 127 : (31 - __clz((int)mb)) - 133;
  return 14 - e;
}
// v * 2^p for |p| <= 150, as two multiplies by normal powers of two (each exact unless the
// result leaves fp32's range or turns subnormal, where it rounds once).
__device__ __forceinline__ float mul_pow2(float v, int p) {
  const int p1 = p / 2, p2 = p - p1;
  return v * __uint_as_float((uint32_t)(p1 + 127) << 23) * __uint_as_float((uint32_t)(p2 + 127) << 23);
}

// mma.sync m16n8k16 (row.col), f16 x f16 products accumulated in fp32: d += a * b.
// Fragments (g = lane / 4, t = lane % 4): a0 = A(g, 2t..2t+1), a1 = A(g+8, 2t..2t+1),
// a2 = A(g, 2t+8..2t+9), a3 = A(g+8, 2t+8..2t+9); b0 = B(2t..2t+1, g), b1 = B(2t+8..2t+9, g);
// d0, d1 = D(g, 2t..2t+1), d2, d3 = D(g+8, 2t..2t+1).
__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// One consumer warp, one unit (128 x 64 tile), the 32 rows 32 rq .. 32 rq + 31 (two groups of
// 16), all 64 inputs, on the tensor cores: the 1-4 activation rows are a dense contraction
// once each weight is an exact f16 operand, and the mixed-precision FMA's issue rate -- one
// product per lane and clock -- is what bounds a 2-4 row GEMV on CUDA cores.
//
// A = the decoded E2M1 values of 16 rows (lane (g, t) holds code word t of rows g and g + 8
// of each 32-input chunk: no re-arrangement of the packed layout), B = the staged f16
// activations (one power-of-two scale per token, stage_x_tok).  The MMA's eight columns
// are (token, quarter parity): column n takes token n % 4 from the inputs of quarter
// 2c + n / 4 only (the lanes whose code word lies in the other quarter supply zeros), so
// every output of the MMA is the sum over ONE 16-input quarter of one row for one token,
// which then takes its block scale with one FMA into the accumulator.  acc[j][i]: row
// 32 rq + 16 j + g (+ 8 for i >= 2), token 2 (t % 2) + i % 2, parity t / 2 (the two
// parities are summed once per segment).
// xslot: token 0's 64 staged activations (bytes) of this unit's input group, xtok the bytes
// between tokens.  The E4M3 table holds the block scale times the tensor scale.
template <int FMT, int M>
__device__ __forceinline__ void consume_mma(const uint8_t* st, const uint8_t* scl, const uint8_t* xslot,
                                            uint32_t xtok, const float* e4m3_lut, int rq, int lane,
                                            float (&acc)[2][4]) {
  static_assert(FMT == FMT_NVFP4 || FMT == FMT_MXFP4, "E2M1 formats only");
  const int g = lane >> 2, t = lane & 3, par = t >> 1;
  const int btok = g & 3;
  const bool bon = btok < M && par == (g >> 2);
  uint32_t sw[4];  // scale bytes of rows 32 rq + g + 8 i
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int row = 32 * rq + g + 8 * i;
    if (FMT == FMT_NVFP4)
      sw[i] = *reinterpret_cast<const uint32_t*>(scl + row * 4);
    else
      sw[i] = *reinterpret_cast<const uint16_t*>(scl + row * 2);
  }
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    uint4 bx = make_uint4(0u, 0u, 0u, 0u);
    if (bon) bx = *reinterpret_cast<const uint4*>(xslot + btok * xtok + 64 * c + 16 * t);
    const int q = 2 * c + par;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const uint8_t* base = st + (rq * 2 + c) * 512 + 256 * j + 4 * lane;
      const uint32_t wl = *reinterpret_cast<const uint32_t*>(base);
      const uint32_t wh = *reinterpret_cast<const uint32_t*>(base + 128);
      float d[4] = {0.0f, 0.0f, 0.0f, 0.0f};
      mma_f16(d, e2m1x2_h2<0>(wl), e2m1x2_h2<0>(wh), e2m1x2_h2<1>(wl), e2m1x2_h2<1>(wh), bx.x, bx.y);
      mma_f16(d, e2m1x2_h2<2>(wl), e2m1x2_h2<2>(wh), e2m1x2_h2<3>(wl), e2m1x2_h2<3>(wh), bx.z, bx.w);
      float sl, sh;
      if (FMT == FMT_NVFP4) {
        sl = e4m3_lut[(sw[2 * j] >> (8 * q)) & 0xFFu];
        sh = e4m3_lut[(sw[2 * j + 1] >> (8 * q)) & 0xFFu];
      } else {
        sl = e8m0_f32(sw[2 * j] >> (8 * c));
        sh = e8m0_f32(sw[2 * j + 1] >> (8 * c));
      }
      acc[j][0] = fmaf(sl, d[0], acc[j][0]);
      acc[j][2] = fmaf(sh, d[2], acc[j][2]);
      if (M > 1) {
        acc[j][1] = fmaf(sl, d[1], acc[j][1]);
        acc[j][3] = fmaf(sh, d[3], acc[j][3]);
      }
    }
  }
}

}  // namespace qg
