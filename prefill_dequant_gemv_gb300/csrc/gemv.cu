// Quantized GEMV for 1..4 activation rows on GB300 (sm_103a).
//
// What it computes (TurboEXL3 article §2.2, W4A16; §4.2 and §4.3 for the 1-4 row
// GEMV): y[m, n] = bf16( sum_k w[n, k] x[m, k] (+ res[m, n]) ), fp32 accumulation,
// every weight read from HBM once for all m rows.
//
// How (GB300 design, not the pages' Metal tile):
//  * Work unit = one 128-row x 64-input tile of the packed layout (4.25-6.9 KB,
//    contiguous).  The U = NT * KG units are cut into `gridDim.x` equal contiguous
//    ranges (stream-K), one CTA per SM, so every SM streams the same byte count.
//  * One producer lane issues 1-D bulk async copies of whole tiles into a deep
//    ring of shared-memory stages (mbarrier completion, bounded waits); twelve
//    consumer warps decode from shared memory.  Warp w takes the 16-input quarter
//    (w % 4) of every 3rd unit; each lane owns 4 rows (one per 32-row tile), so
//    every activation value read from shared memory feeds 4 rows.
//  * Decode in registers to fp32 operands (qg_common.cuh), packed f32x2 FMAs into
//    per-block partials, block scale applied once per block (Q6_K operand PR #19:
//    the epilogue is one fma(dot, scale) per chain).
//  * Row tiles split across CTAs are finished by the CTA that arrives last on the
//    tile's ticket (TurboEXL3 article §4.3: "the threadgroup that arrives last runs
//    the finish"); it sums the partials in CTA order, so results are deterministic.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>

#include "qg_common.cuh"
#include "qg_internal.h"
#include "qg_sync.cuh"

namespace qg {

constexpr int kCW = 12;                 // consumer warps (13 warps in all -> 128 registers)
constexpr int kCT = kCW * 32;           // consumer threads
constexpr int kGemvThreads = kCT + 32;  // + one producer warp
constexpr int kGroups = kCW / 4;        // unit groups (4 warps: one per 16-input quarter)
constexpr int kMaxStages = 48;

struct GemvArgs {
  const uint8_t* codes;
  const uint8_t* scales;
  const uint8_t* aux;
  const __nv_bfloat16* x;
  const __nv_bfloat16* res;
  __nv_bfloat16* y;
  int64_t ldx, ldr, ldy;
  int64_t n, k;
  int64_t U;
  int KG;
  int nslots;
  int stages;
  float ts;
  float* ws_part;  // [grid][2][M][128]
  int* ws_cnt;     // [NT]
  int* status;
};

template <int FMT> struct Stage {
  static constexpr int CODE = Fmt<FMT>::TB;
  static constexpr int SCALE = 128 * Fmt<FMT>::SB;
  static constexpr int AUX = (FMT == FMT_Q6K) ? 256 : 0;
  static constexpr int BYTES = CODE + SCALE + AUX;
};

struct SmemLayout {
  size_t bars, stages, xs, sums, red, flag, total;
};

__host__ __device__ inline SmemLayout gemv_smem_layout(int stage_bytes, int S, int M, int nslots) {
  SmemLayout L;
  size_t o = 0;
  L.bars = o;
  o += (size_t)2 * S * 8;
  o = (o + 127) & ~(size_t)127;
  L.stages = o;
  o += (size_t)S * stage_bytes;
  o = (o + 127) & ~(size_t)127;
  L.xs = o;
  o += (size_t)M * nslots * 64 * 4;
  L.sums = o;
  o += (size_t)M * nslots * 8 * 4;  // (Z, X) per 16-input quarter
  L.red = o;
  o += (size_t)kCW * M * 128 * 4;
  L.flag = o;
  o += 16;
  L.total = o;
  return L;
}

__host__ __device__ inline int64_t owner_cta(int64_t u, int64_t U, int64_t G) {
  // CTA b owns units [b*U/G, (b+1)*U/G); the owner of u is the largest b with b*U/G <= u.
  return ((u + 1) * G - 1) / U;
}

__device__ __forceinline__ void bf16x2_to_f32(uint32_t v, float& lo, float& hi) {
  lo = __uint_as_float(v << 16);
  hi = __uint_as_float(v & 0xFFFF0000u);
}

// Stage x rows (bf16) into shared memory as fp32, 16 inputs per item.  Integer
// formats store each group of eight in the operand-pair order [3,4,5,6,7,0,1,2]
// and record, per 16-input quarter, Z = c12 * X_odd + c16 * X_even and X = X_odd +
// X_even (sums over odd / even input positions), which remove the operands'
// constant 1 and the zero point in the fold.
template <int FMT, int M>
__device__ void stage_x(const GemvArgs& a, float* xs, float* sums, int sbase, int nslots, int tid) {
  constexpr bool kInt = (FMT == FMT_MLX || FMT == FMT_Q6K);
  constexpr float c12 = (FMT == FMT_Q6K) ? 2080.0f : 2048.0f;  // 2^11 (+32 for the Q6_K zero point)
  constexpr float c16 = (FMT == FMT_Q6K) ? 160.0f : 128.0f;    // 2^7  (+32)
  const int items = M * nslots * 4;
  for (int it = tid; it < items; it += kCT) {
    const int kq = it & 3;
    const int s = (it >> 2) % nslots;
    const int m = (it >> 2) / nslots;
    const int g = (sbase + s) % a.KG;
    const int64_t k0 = (int64_t)g * 64 + kq * 16;
    float v[16];
    if (k0 < a.k) {
      const uint4* src = reinterpret_cast<const uint4*>(a.x + m * a.ldx + k0);
      const uint4 r0 = src[0], r1 = src[1];
      const uint32_t u[8] = {r0.x, r0.y, r0.z, r0.w, r1.x, r1.y, r1.z, r1.w};
#pragma unroll
      for (int i = 0; i < 8; ++i) bf16x2_to_f32(u[i], v[2 * i], v[2 * i + 1]);
    } else {
#pragma unroll
      for (int i = 0; i < 16; ++i) v[i] = 0.0f;
    }
    float* dst = xs + (size_t)(m * nslots + s) * 64 + kq * 16;
    if (kInt) {
      float xo = 0.0f, xe = 0.0f;
#pragma unroll
      for (int w = 0; w < 2; ++w) {
        const float* s8 = v + 8 * w;
        reinterpret_cast<float4*>(dst)[2 * w] = make_float4(s8[3], s8[4], s8[5], s8[6]);
        reinterpret_cast<float4*>(dst)[2 * w + 1] = make_float4(s8[7], s8[0], s8[1], s8[2]);
        xo += (s8[1] + s8[3]) + (s8[5] + s8[7]);
        xe += (s8[0] + s8[2]) + (s8[4] + s8[6]);
      }
      float* z = sums + ((size_t)(m * nslots + s) * 4 + kq) * 2;
      z[0] = c12 * xo + c16 * xe;
      z[1] = xo + xe;
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i)
        reinterpret_cast<float4*>(dst)[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
    }
  }
}

// One consumer warp, one unit, one 16-input quarter: accumulate 4 rows x M.
template <int FMT, int M>
__device__ __forceinline__ void consume(const uint8_t* st, const float* xq, int mstride, const float* sq,
                                        int sstride, int kq, int lane, float (&acc)[4][M]) {
  using F = Fmt<FMT>;
  using SG = Stage<FMT>;
  uint32_t wd[4][2];
  uint32_t hw[4];
#pragma unroll
  for (int rt = 0; rt < 4; ++rt) {
    const uint2 v = *reinterpret_cast<const uint2*>(st + ((rt * F::CH + (kq >> 1)) * 32 + lane) * 16 + (kq & 1) * 8);
    wd[rt][0] = v.x;
    wd[rt][1] = v.y;
    if (FMT == FMT_Q6K) hw[rt] = *reinterpret_cast<const uint32_t*>(st + ((rt * 3 + 2) * 32 + lane) * 16 + kq * 4);
  }
  float2 P[4][M];
#pragma unroll
  for (int rt = 0; rt < 4; ++rt)
#pragma unroll
    for (int m = 0; m < M; ++m) P[rt][m] = make_float2(0.0f, 0.0f);

#pragma unroll
  for (int wi = 0; wi < 2; ++wi) {
    float4 xa[M], xb[M];
#pragma unroll
    for (int m = 0; m < M; ++m) {
      xa[m] = *reinterpret_cast<const float4*>(xq + m * mstride + wi * 8);
      xb[m] = *reinterpret_cast<const float4*>(xq + m * mstride + wi * 8 + 4);
    }
#pragma unroll
    for (int rt = 0; rt < 4; ++rt) {
      const uint32_t w = wd[rt][wi];
      float2 p0, p1, p2, p3;
      if (FMT == FMT_MXFP4 || FMT == FMT_NVFP4) {
        p0 = e2m1x2_f32<0>(w);
        p1 = e2m1x2_f32<1>(w);
        p2 = e2m1x2_f32<2>(w);
        p3 = e2m1x2_f32<3>(w);
      } else if (FMT == FMT_MLX) {
        p0 = int4_pair(w);
        p1 = int4_pair(rot8(w));
        p2 = int4_pair(rot16(w));
        p3 = int4_pair(rot24(w));
      } else {
        const uint32_t h = q6k_hi_for(hw[rt], wi);
        p0 = int6_pair(w, h);
        p1 = int6_pair(rot8(w), rot8(h));
        p2 = int6_pair(rot16(w), rot16(h));
        p3 = int6_pair(rot24(w), rot24(h));
      }
#pragma unroll
      for (int m = 0; m < M; ++m) {
        P[rt][m] = ffma2(p0, make_float2(xa[m].x, xa[m].y), P[rt][m]);
        P[rt][m] = ffma2(p1, make_float2(xa[m].z, xa[m].w), P[rt][m]);
        P[rt][m] = ffma2(p2, make_float2(xb[m].x, xb[m].y), P[rt][m]);
        P[rt][m] = ffma2(p3, make_float2(xb[m].z, xb[m].w), P[rt][m]);
      }
    }
  }
  // Fold the quarter's partial with the block scale (once per block and row).
#pragma unroll
  for (int rt = 0; rt < 4; ++rt) {
    const int row = rt * 32 + lane;
    const uint8_t* sp = st + SG::CODE + row * F::SB;
    if (FMT == FMT_NVFP4) {
      const uint32_t sw = *reinterpret_cast<const uint32_t*>(sp);
      const float2 s01 = (kq >> 1) ? e4m3x2_f32<1>(sw) : e4m3x2_f32<0>(sw);
      const float S = (kq & 1) ? s01.y : s01.x;
#pragma unroll
      for (int m = 0; m < M; ++m) acc[rt][m] = fmaf(S, P[rt][m].x + P[rt][m].y, acc[rt][m]);
    } else if (FMT == FMT_MXFP4) {
      const float S = e8m0_f32(sp[kq >> 1]);
#pragma unroll
      for (int m = 0; m < M; ++m) acc[rt][m] = fmaf(S, P[rt][m].x + P[rt][m].y, acc[rt][m]);
    } else if (FMT == FMT_MLX) {
      const uint32_t sw = *reinterpret_cast<const uint32_t*>(sp);
      const float s = __half2float(__ushort_as_half((unsigned short)(sw & 0xFFFFu)));
      const float bias = __half2float(__ushort_as_half((unsigned short)(sw >> 16)));
#pragma unroll
      for (int m = 0; m < M; ++m) {
        const float dot = fmaf(kClass12, P[rt][m].x, fmaf(kClass16, P[rt][m].y, -sq[m * sstride]));
        acc[rt][m] = fmaf(s, dot, fmaf(bias, sq[m * sstride + 1], acc[rt][m]));
      }
    } else {
      const float sc = (float)(int8_t)sp[kq];
      const float d = __half2float(*reinterpret_cast<const __half*>(st + SG::CODE + SG::SCALE + row * 2));
      const float ds = d * sc;
#pragma unroll
      for (int m = 0; m < M; ++m) {
        const float dot = fmaf(kClass12, P[rt][m].x, fmaf(kClass16, P[rt][m].y, -sq[m * sstride]));
        acc[rt][m] = fmaf(ds, dot, acc[rt][m]);
      }
    }
  }
}

template <int M>
__device__ __forceinline__ void finish_out(const GemvArgs& a, int64_t q, int e, float v) {
  const int m = e / 128, row = e % 128;
  const int64_t n = q * 128 + row;
  if (n >= a.n) return;
  float r = a.ts * v;
  if (a.res) r += __bfloat162float(a.res[m * a.ldr + n]);
  a.y[m * a.ldy + n] = __float2bfloat16_rn(r);
}

template <int FMT, int M>
__global__ void __launch_bounds__(kGemvThreads, 1) gemv_kernel(const GemvArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  using SG = Stage<FMT>;
  const int S = a.stages, nslots = a.nslots;
  const SmemLayout L = gemv_smem_layout(SG::BYTES, S, M, nslots);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bars);
  uint64_t* empty = full + S;
  uint8_t* stages = smem + L.stages;
  float* xs = reinterpret_cast<float*>(smem + L.xs);
  float* sums = reinterpret_cast<float*>(smem + L.sums);
  float* red = reinterpret_cast<float*>(smem + L.red);
  int* flag = reinterpret_cast<int*>(smem + L.flag);

  const int64_t U = a.U;
  const int64_t G = gridDim.x;
  const int64_t b = blockIdx.x;
  const int64_t u0 = b * U / G, u1 = (b + 1) * U / G;
  if (u0 >= u1) return;
  const int64_t len = u1 - u0;
  const int KG = a.KG;
  const int sbase = len >= KG ? 0 : (int)(u0 % KG);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 4);
    }
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kCW) {  // producer: stream whole tiles into the ring
    if (lane == 0) {
      for (int64_t i = 0; i < len; ++i) {
        const int s = (int)(i % S);
        const uint32_t use = (uint32_t)(i / S);
        if (use > 0 && !mbar_wait_bounded(&empty[s], (use - 1) & 1, a.status)) break;
        const int64_t uu = u0 + i, q = uu / KG;
        const int g = (int)(uu % KG);
        const int64_t t = q * KG + g;
        uint8_t* dst = stages + (size_t)s * SG::BYTES;
        mbar_arrive_expect_tx(&full[s], SG::BYTES);
        bulk_g2s(dst, a.codes + t * SG::CODE, SG::CODE, &full[s]);
        bulk_g2s(dst + SG::CODE, a.scales + t * SG::SCALE, SG::SCALE, &full[s]);
        if (SG::AUX) bulk_g2s(dst + SG::CODE + SG::SCALE, a.aux + (q * (KG / 4) + g / 4) * 256, 256, &full[s]);
      }
    }
    return;
  }

  stage_x<FMT, M>(a, xs, sums, sbase, nslots, tid);
  named_sync(1, kCT);

  const int ug = warp >> 2, kq = warp & 3;
  bool ok = true;
  int64_t u = u0;
  while (u < u1) {
    const int64_t q = u / KG;
    const int64_t seg_end = min(u1, (q + 1) * KG);
    float acc[4][M];
#pragma unroll
    for (int rt = 0; rt < 4; ++rt)
#pragma unroll
      for (int m = 0; m < M; ++m) acc[rt][m] = 0.0f;
    int64_t i = u - u0;
    i += (ug - (int)(i % kGroups) + kGroups) % kGroups;
    for (; ok && i < seg_end - u0; i += kGroups) {
      const int s = (int)(i % S);
      const uint32_t use = (uint32_t)(i / S);
      if (!mbar_wait_bounded(&full[s], use & 1, a.status)) {
        ok = false;
        break;
      }
      const int g = (int)((u0 + i) % KG);
      const int slot = (g - sbase + KG) % KG;
      consume<FMT, M>(stages + (size_t)s * SG::BYTES, xs + (size_t)slot * 64 + kq * 16, nslots * 64,
                      sums + ((size_t)slot * 4 + kq) * 2, nslots * 8, kq, lane, acc);
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }
#pragma unroll
    for (int rt = 0; rt < 4; ++rt)
#pragma unroll
      for (int m = 0; m < M; ++m) red[(warp * M + m) * 128 + rt * 32 + lane] = acc[rt][m];
    named_sync(1, kCT);

    const bool whole = (u == q * KG) && (seg_end == (q + 1) * KG);
    const int slot_ws = (u == u0) ? 0 : 1;
    for (int e = tid; e < M * 128; e += kCT) {
      float v = 0.0f;
#pragma unroll 4
      for (int w2 = 0; w2 < kCW; ++w2) v += red[w2 * M * 128 + e];
      if (whole)
        finish_out<M>(a, q, e, v);
      else
        a.ws_part[(size_t)((b * 2 + slot_ws) * M) * 128 + e] = v;
    }
    if (!whole) {
      __threadfence();
      named_sync(1, kCT);
      const int64_t bf = owner_cta(q * KG, U, G), bl = owner_cta((q + 1) * KG - 1, U, G);
      if (tid == 0) {
        const int old = atomicAdd(&a.ws_cnt[q], 1);
        *flag = (old == (int)(bl - bf)) ? 1 : 0;
      }
      named_sync(1, kCT);
      if (*flag) {
        __threadfence();
        for (int e = tid; e < M * 128; e += kCT) {
          float v = 0.0f;
          for (int64_t bb = bf; bb <= bl; ++bb) {
            const int sl = ((bb * U / G) / KG == q) ? 0 : 1;
            v += __ldcg(&a.ws_part[(size_t)((bb * 2 + sl) * M) * 128 + e]);
          }
          finish_out<M>(a, q, e, v);
        }
        if (tid == 0) a.ws_cnt[q] = 0;
      }
    }
    named_sync(1, kCT);
    u = seg_end;
  }
}

// ---------------------------------------------------------------- host side
static int stage_bytes_of(int fmt) {
  switch (fmt) {
    case FMT_MLX: return Stage<FMT_MLX>::BYTES;
    case FMT_MXFP4: return Stage<FMT_MXFP4>::BYTES;
    case FMT_NVFP4: return Stage<FMT_NVFP4>::BYTES;
    default: return Stage<FMT_Q6K>::BYTES;
  }
}

bool plan_gemv(const Geometry& g, int m, const DeviceInfo& dev, GemvPlan* p) {
  const int sbytes = stage_bytes_of(g.fmt);
  const int64_t U = g.nt * g.kg;
  const size_t budget = (size_t)dev.max_smem_optin;
  int64_t G = std::min<int64_t>(dev.sms, U);
  for (;;) {
    const int64_t len = (U + G - 1) / G;
    const int nslots = (int)std::min<int64_t>(len, g.kg);
    const SmemLayout L0 = gemv_smem_layout(sbytes, 2, m, nslots);
    if (L0.total <= budget || G >= U) {
      if (L0.total > budget) return false;
      int S = (int)std::min<int64_t>(len, (int64_t)kMaxStages);
      S = std::max(S, 2);
      while (S > 2 && gemv_smem_layout(sbytes, S, m, nslots).total > budget) --S;
      p->grid = (int)G;
      p->nslots = nslots;
      p->stages = S;
      p->smem = gemv_smem_layout(sbytes, S, m, nslots).total;
      p->units = U;
      p->off_cnt = kWsHeader;
      p->off_part = kWsHeader + (((size_t)g.nt * 4 + 255) & ~(size_t)255);
      p->ws_bytes = p->off_part + (size_t)G * 2 * m * 128 * 4;
      return true;
    }
    G = std::min<int64_t>(U, G * 2);
  }
}

template <int FMT, int M>
static int launch_t(const GemvArgs& a, const GemvPlan& p, cudaStream_t s) {
  static std::atomic<unsigned long long> configured{0};
  int dev = 0;
  DeviceInfo info;
  if (cudaGetDevice(&dev) != cudaSuccess || !device_info(dev, &info)) return QG_ERR_CUDA;
  const unsigned long long bit = 1ull << (dev & 63);
  if (!(configured.load() & bit)) {
    if (cudaFuncSetAttribute(gemv_kernel<FMT, M>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             info.max_smem_optin) != cudaSuccess)
      return QG_ERR_CUDA;
    configured.fetch_or(bit);
  }
  gemv_kernel<FMT, M><<<p.grid, kGemvThreads, p.smem, s>>>(a);
  return cudaGetLastError() == cudaSuccess ? QG_OK : QG_ERR_CUDA;
}

template <int FMT>
static int launch_m(const GemvArgs& a, int m, const GemvPlan& p, cudaStream_t s) {
  switch (m) {
    case 1: return launch_t<FMT, 1>(a, p, s);
    case 2: return launch_t<FMT, 2>(a, p, s);
    case 3: return launch_t<FMT, 3>(a, p, s);
    default: return launch_t<FMT, 4>(a, p, s);
  }
}

int launch_gemv(const Geometry& g, const qg_weight* w, const void* x, int m, int64_t ldx, const void* res,
                int64_t ldr, void* y, int64_t ldy, void* ws, const GemvPlan& p, void* stream) {
  GemvArgs a;
  a.codes = static_cast<const uint8_t*>(w->codes);
  a.scales = static_cast<const uint8_t*>(w->scales);
  a.aux = static_cast<const uint8_t*>(w->aux);
  a.x = static_cast<const __nv_bfloat16*>(x);
  a.res = static_cast<const __nv_bfloat16*>(res);
  a.y = static_cast<__nv_bfloat16*>(y);
  a.ldx = ldx;
  a.ldr = ldr;
  a.ldy = ldy;
  a.n = g.n;
  a.k = g.k;
  a.U = p.units;
  a.KG = (int)g.kg;
  a.nslots = p.nslots;
  a.stages = p.stages;
  a.ts = (g.fmt == FMT_NVFP4) ? w->tensor_scale : 1.0f;
  uint8_t* wsb = static_cast<uint8_t*>(ws);
  a.status = reinterpret_cast<int*>(wsb);
  a.ws_cnt = reinterpret_cast<int*>(wsb + p.off_cnt);
  a.ws_part = reinterpret_cast<float*>(wsb + p.off_part);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  switch (g.fmt) {
    case FMT_MLX: return launch_m<FMT_MLX>(a, m, p, s);
    case FMT_MXFP4: return launch_m<FMT_MXFP4>(a, m, p, s);
    case FMT_NVFP4: return launch_m<FMT_NVFP4>(a, m, p, s);
    default: return launch_m<FMT_Q6K>(a, m, p, s);
  }
}

}  // namespace qg
