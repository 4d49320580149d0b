// Quantized GEMV for 1..4 activation rows on GB300 (sm_103a).
//
// What it computes (TurboEXL3 article §2.2, W4A16; §4.2 and §4.3 for the 1-4 row
// GEMV): y[m, n] = bf16( sum_k w[n, k] x[m, k] (+ res[m, n]) ), fp32 accumulation,
// every weight read from HBM once for all m rows.
//
// How (GB300 design, not the pages' Metal tile):
//  * Work unit = one 128-row x 64-input tile of the packed layout (4.25-6.9 KB,
//    contiguous).  Three ways to cut the U = NT * KG units over the SMs, all
//    deterministic: one whole row tile per CTA when the row tiles nearly fill the GPU;
//    each row tile split over a thread-block cluster (equal input ranges, partials
//    summed in the first CTA's shared memory) when they fill less than half of it;
//    otherwise equal contiguous unit ranges per SM (stream-K), where a row tile split
//    across CTAs is finished by the last CTA to take its ticket -- the last arrival
//    runs the finish, as in the TurboEXL3 article §4.3 -- summing the partials in CTA
//    order.
//  * One producer lane issues 1-D bulk async copies of whole tiles into a deep ring of
//    shared-memory stages (mbarrier completion, bounded waits); it requests one chunk, then
//    waits until the consumers' activation loads are out.  16 consumer warps (12 at four
//    rows on CUDA cores) decode from shared memory; warp w takes half of unit w / 2 of
//    every chunk.
//  * CUDA-core consumer (every format at one row; the integer formats at 2-4): the warp's
//    half is two 16-input quarters; each lane owns 4 rows (one per 32-row tile), so every
//    activation value read from shared memory feeds 4 rows.  Weights become exact f16
//    operands in registers (qg_common.cuh) multiplied into fp32 with the mixed-precision
//    FMA; the block scale (and the integer formats' operand constant) is applied once per 16
//    inputs and row (Q6_K operand PR #19: one fma(dot, scale) per chain).
//  * Tensor-core consumer (E2M1 formats at 2-4 rows, consume_mma): the warp's half is 64
//    rows; the decoded weights are A of mma.sync m16n8k16, the 1-4 activation rows B (the
//    FMA's one product per lane and clock, not the bytes, bounds 2-4 rows on CUDA cores).
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>

#include "qg_common.cuh"
#include "qg_gemv_core.cuh"
#include "qg_internal.h"
#include "qg_sync.cuh"

namespace qg {

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
  int csplit;      // > 1: cluster mode (row tile q = cluster q, partials reduced over DSMEM)
  float* ws_part;  // [grid][2][M][128]
  int* ws_cnt;     // [NT]
  int* status;
};

constexpr int kMaxCsplit = 8;  // portable cluster size
// Weight chunks a CTA requests before its activation loads are out: the rest wait, so the
// activations -- on the critical path, since nothing is consumed before they are staged --
// do not queue behind this CTA's whole weight burst.
constexpr int kEarlyChunks = 1;

struct SmemLayout {
  size_t bars, stages, xs, sums, red, cbuf, lut, misc, total;
};

__host__ __device__ inline SmemLayout gemv_smem_layout(int stage_bytes, int S, int M, int nslots, int csplit,
                                                       int kCW) {
  // stage_bytes: bytes of one chunk stage; kCW: consumer warps
  SmemLayout L;
  size_t o = 0;
  L.bars = o;
  o += (size_t)2 * S * 8;
  o = (o + 127) & ~(size_t)127;
  L.stages = o;
  o += (size_t)S * stage_bytes;
  o = (o + 127) & ~(size_t)127;
  L.xs = o;
  o += (size_t)M * nslots * 64 * 2;  // f16 activations
  L.sums = o;
  o += (size_t)M * nslots * 16 * 4;  // {scale, Z, X, 0} per 16-input quarter
  L.red = o;
  o += (size_t)kCW * M * 128 * 4;
  L.cbuf = o;  // cluster mode: every rank's partial of the row tile, in rank 0's CTA
  o += csplit > 1 ? (size_t)csplit * M * 128 * 4 : 0;
  L.lut = o;
  o += 256 * 4;  // E4M3 -> fp32
  L.misc = o;
  o += 64;  // ticket flag
  L.total = o;
  return L;
}

// A thread's activation staging items -- (row m, slot s, quarter kq) of the CTA's
// M x nslots x 4 -- are every kCT-th item from item tid: kq is the thread's own (kCT is a
// multiple of 4) and (m, s) advances by kCT / 4 slots at a time, without a division.
struct XItem {
  int m, s, kq;
};
struct XStep {
  int dm, ds;  // kCT / 4 slots as whole rows and remaining slots
};
__device__ __forceinline__ XItem item_first(int tid, int nslots) {
  const int j = tid >> 2, m = j / nslots;
  return XItem{m, j - m * nslots, tid & 3};
}
__device__ __forceinline__ XStep item_step(int kCT, int nslots) {
  const int q = (kCT >> 2) / nslots;
  return XStep{q, (kCT >> 2) - q * nslots};
}
__device__ __forceinline__ void item_next(XItem& x, const XStep& st, int nslots) {
  x.m += st.dm;
  x.s += st.ds;
  if (x.s >= nslots) {
    x.s -= nslots;
    ++x.m;
  }
}

// The 16 activations of item x as eight bf16 pairs; inputs past K, and items past the last
// row (x.m >= M), read as zero.  The loads are unconditional (from x's first element when
// the item is outside) so that a thread's loads of several items all go out before any
// result is used, and volatile so that each is made exactly once where it stands.
template <int M>
__device__ __forceinline__ void load_quarter(const GemvArgs& a, const XItem& x, int sbase, uint32_t (&u)[8]) {
  int g = sbase + x.s;  // input group: sbase + s < 2 KG
  if (g >= a.KG) g -= a.KG;
  const int64_t k0 = (int64_t)g * 64 + x.kq * 16;
  const bool in = x.m < M && k0 < a.k;
  const __nv_bfloat16* src = in ? a.x + x.m * a.ldx + k0 : a.x;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(u[0]), "=r"(u[1]), "=r"(u[2]), "=r"(u[3]) : "l"(src));
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(u[4]), "=r"(u[5]), "=r"(u[6]), "=r"(u[7]) : "l"(src + 8));
  if (!in) {
#pragma unroll
    for (int i = 0; i < 8; ++i) u[i] = 0;
  }
}

// Stage the activation rows of a CTA's input groups into shared memory for the CUDA-core
// consumer (see stage_quarter): row m, slot s, quarter kq -> 8 staging words and one
// record.  xissued: every consumer warp arrives once its first loads are out (the producer
// holds the weight stream back until then).
template <int FMT, int M, int kCT>
__device__ void stage_x(const GemvArgs& a, uint32_t* xs, float* sums, int sbase, int nslots, int tid,
                        uint64_t* xissued) {
  constexpr int R = 2;  // items whose loads go out together
  const XStep st = item_step(kCT, nslots);
  XItem it = item_first(tid, nslots);
  XItem its[R];
  uint32_t u[R][8];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    its[r] = it;
    load_quarter<M>(a, it, sbase, u[r]);
    item_next(it, st, nslots);
  }
  __syncwarp();
  if ((tid & 31) == 0) mbar_arrive(xissued);
  auto stage = [&](const XItem& x, const uint32_t (&v)[8]) {
    const int j = x.m * nslots + x.s;
    const float4 z = stage_quarter<FMT>(v, xs + (size_t)j * 32 + x.kq * 8);
    reinterpret_cast<float4*>(sums)[(size_t)j * 4 + x.kq] = z;
  };
#pragma unroll
  for (int r = 0; r < R; ++r)
    if (its[r].m < M) stage(its[r], u[r]);
  for (; it.m < M; item_next(it, st, nslots)) {
    uint32_t v[8];
    load_quarter<M>(a, it, sbase, v);
    stage(it, v);
  }
}

// Largest bf16 magnitude bits of a quarter, folded into the token's running maximum.
template <int M>
__device__ __forceinline__ void fold_max(const uint32_t (&u)[8], int m, uint32_t (&mx)[M]) {
  uint32_t mb = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) mb = max(mb, max(u[i] & 0x7FFFu, (u[i] >> 16) & 0x7FFFu));
#pragma unroll
  for (int mm = 0; mm < M; ++mm)
    if (mm == m) mx[mm] = max(mx[mm], mb);
}

// Item x as f16 times its token's 2^p (p = tok_exp of the token's maximum in pmax), applied
// as two normal powers of two.
__device__ __forceinline__ void store_quarter_tok(uint32_t* xs, const XItem& x, int nslots, const uint32_t* pmax,
                                                  const uint32_t (&u)[8]) {
  const int p = tok_exp(pmax[x.m]), p1 = p / 2;
  const float a1 = __uint_as_float((uint32_t)(p1 + 127) << 23);
  const float a2 = __uint_as_float((uint32_t)(p - p1 + 127) << 23);
  uint32_t w[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    float lo, hi;
    bf16x2_to_f32(u[i], lo, hi);
    __half2 h = __floats2half2_rn(lo * a1 * a2, hi * a1 * a2);
    w[i] = *reinterpret_cast<uint32_t*>(&h);
  }
  uint4* dst = reinterpret_cast<uint4*>(xs + (size_t)(x.m * nslots + x.s) * 32 + x.kq * 8);
  dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
  dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
}

// Stage the activation rows for the tensor-core consumer: f16 with ONE power-of-two scale
// per token over this CTA's input groups, 2^p with p = tok_exp(the token's largest |x|),
// so B of every MMA shares it and the partial sums need no per-quarter rescaling.  The
// largest value lands in [2^14, 2^15); bf16 values more than 2^32 below it round onto f16's
// subnormal grid (absolute error under 2^-40 of the token's max: far inside the stated
// bound).  Two passes: the token maxima (each thread keeps its first R items in
// registers), a block-wide max in pmax[m] (zeroed before the kernel's first barrier), then
// the conversion.  Row m, slot s, quarter kq -> 8 staging words, natural pair order.
template <int M, int kCT>
__device__ void stage_x_tok(const GemvArgs& a, uint32_t* xs, uint32_t* pmax, int sbase, int nslots, int tid,
                            uint64_t* xissued) {
  constexpr int R = 4;
  const XStep st = item_step(kCT, nslots);
  uint32_t mx[M];
#pragma unroll
  for (int m = 0; m < M; ++m) mx[m] = 0;
  XItem it = item_first(tid, nslots);
  XItem its[R];
  uint32_t held[R][8];
  // every held item's loads first (one round trip to memory), then their maxima
#pragma unroll
  for (int r = 0; r < R; ++r) {
    its[r] = it;
    load_quarter<M>(a, it, sbase, held[r]);
    item_next(it, st, nslots);
  }
  __syncwarp();
  if ((tid & 31) == 0) mbar_arrive(xissued);
#pragma unroll
  for (int r = 0; r < R; ++r)
    if (its[r].m < M) fold_max<M>(held[r], its[r].m, mx);
  for (XItem x = it; x.m < M; item_next(x, st, nslots)) {
    uint32_t v[8];
    load_quarter<M>(a, x, sbase, v);
    fold_max<M>(v, x.m, mx);
  }
#pragma unroll
  for (int m = 0; m < M; ++m) {
    const uint32_t v = __reduce_max_sync(0xFFFFFFFFu, mx[m]);
    if ((tid & 31) == 0 && v) atomicMax(&pmax[m], v);
  }
  named_sync(1, kCT);
#pragma unroll
  for (int r = 0; r < R; ++r)
    if (its[r].m < M) store_quarter_tok(xs, its[r], nslots, pmax, held[r]);
  for (; it.m < M; item_next(it, st, nslots)) {
    uint32_t v[8];
    load_quarter<M>(a, it, sbase, v);
    store_quarter_tok(xs, it, nslots, pmax, v);
  }
}

// Output e = m * 128 + row of row tile q: ts * v (+ residual), rounded to bf16 once.
template <int M>
__device__ __forceinline__ void finish_out(const GemvArgs& a, uint32_t q, int e, float v, float ts) {
  const int m = e / 128, row = e % 128;
  const int64_t n = (int64_t)q * 128 + row;
  if (n >= a.n) return;
  float r = ts * v;
  if (a.res) r += __bfloat162float(a.res[m * a.ldr + n]);
  a.y[m * a.ldy + n] = __float2bfloat16_rn(r);
}

template <int FMT, int M>
__global__ void __launch_bounds__(gemv_warps(FMT, M) * 32 + 32, 1) gemv_kernel(const GemvArgs a) {
  constexpr bool kMma = gemv_mma(FMT, M);  // tensor-core consumer (E2M1 formats)
  constexpr int kCW = gemv_warps(FMT, M);  // consumer warps
  constexpr int kCT = kCW * 32;           // consumer threads (one producer warp follows)
  constexpr int kWPU = 2;                 // warps per unit: two 16-input quarters (CUDA cores) or
                                          // 64 rows (tensor cores) each, per chunk
  constexpr int kGroups = kCW / kWPU;     // unit groups
  extern __shared__ __align__(128) uint8_t smem[];
  using SG = Stage<FMT>;
  const int S = a.stages, nslots = a.nslots;
  const SmemLayout L = gemv_smem_layout(Stage<FMT>::bytes(kCW / 2), S, M, nslots, a.csplit, kCW);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bars);
  uint64_t* empty = full + S;
  uint8_t* stages = smem + L.stages;
  uint32_t* xs = reinterpret_cast<uint32_t*>(smem + L.xs);
  float* sums = reinterpret_cast<float*>(smem + L.sums);
  float* red = reinterpret_cast<float*>(smem + L.red);
  float* cbuf = reinterpret_cast<float*>(smem + L.cbuf);
  float* lut = reinterpret_cast<float*>(smem + L.lut);
  int* flag = reinterpret_cast<int*>(smem + L.misc);
  uint64_t* xissued = reinterpret_cast<uint64_t*>(smem + L.misc + 16);  // the activation loads are out
  const bool clustered = a.csplit > 1;

  const int64_t U = a.U;
  const int64_t G = gridDim.x;
  const int64_t b = blockIdx.x;
  const int64_t u0 = b * U / G, u1 = (b + 1) * U / G;
  if (u0 >= u1 && !clustered) return;
  const int64_t len = u1 - u0;
  const int KG = a.KG;
  const int sbase = len >= KG ? 0 : (int)(u0 % KG);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  constexpr int C = kGroups;  // units per chunk: one per unit group
  const int SB = Stage<FMT>::bytes(C);
  for (int s = tid; s < S; s += blockDim.x) {
    mbar_init(&full[s], 1);
    mbar_init(&empty[s], kCW);  // every consumer warp releases each chunk once
  }
  if (tid == 0) mbar_init(xissued, kCW);
  if (tid < S + 1) fence_mbar_init();
  uint32_t* pmax = reinterpret_cast<uint32_t*>(sums);  // tensor-core staging: token maxima
  if (kMma && tid < M) pmax[tid] = 0;
  __syncthreads();
  // The next kernel may start streaming its weights while this one runs; it reads
  // activations and the workspace only after this grid has completed (pdl_wait).
  if (tid == 0) pdl_launch_dependents();

  // All loop indices below are 32-bit and advanced incrementally (the host
  // guarantees fewer than 2^31 units): 64-bit division in the per-unit path costs
  // more than the decode itself.
  const uint32_t uu0 = (uint32_t)u0, uu1 = (uint32_t)u1;
  const int nch = (int)((len + C - 1) / C);
  if (warp == kCW) {  // producer: stream chunks of whole tiles into the ring
    if (lane == 0) {
      const uint64_t pol = l2_evict_first();  // each weight is read once per call
      int s = 0;
      uint32_t ph = 0;
      uint32_t ua = uu0;
      for (int j = 0; j < nch; ++j) {
        if (j >= S && !mbar_wait_bounded(&empty[s], ph ^ 1u, a.status)) break;
        // With several activation rows, two chunks go out at once and the rest wait until the
        // activations are staged, so their loads do not queue behind this CTA's whole weight
        // burst (17408 x 5120 at four rows: 27.7 -> 26.4 us; one row stages too little to gain).
        if (j == kEarlyChunks && !mbar_wait_bounded(xissued, 0, a.status)) break;
        const uint32_t ub = min(uu1, ua + C);
        const uint32_t nu = ub - ua;
        uint8_t* dst = stages + (size_t)s * SB;
        uint32_t bytes = nu * (SG::CODE + SG::SCALE);
        uint32_t aux_a = 0, aux_n = 0;
        if (SG::AUX) {
          aux_a = ua >> 2;
          aux_n = ((ub - 1) >> 2) - aux_a + 1;
          bytes += aux_n * SG::AUX;
        }
        mbar_arrive_expect_tx(&full[s], bytes);
        bulk_g2s_hint(dst, a.codes + (size_t)ua * SG::CODE, nu * SG::CODE, &full[s], pol);
        bulk_g2s_hint(dst + C * SG::CODE, a.scales + (size_t)ua * SG::SCALE, nu * SG::SCALE, &full[s], pol);
        if (SG::AUX)
          bulk_g2s_hint(dst + C * (SG::CODE + SG::SCALE), a.aux + (size_t)aux_a * SG::AUX, aux_n * SG::AUX, &full[s],
                        pol);
        ua = ub;
        if (++s == S) {
          s = 0;
          ph ^= 1u;
        }
      }
    }
    __syncwarp();  // lane 0 rejoins the warp before the cluster barrier
    if (clustered) cluster_sync_all();  // every thread of the cluster takes the one barrier
    return;
  }

  // E4M3 -> fp32 table, two entries per thread: the block scale times the tensor scale
  // (one rounding), so that no partial sum carries the factor 1 / ts.
  if (FMT == FMT_NVFP4 && tid < 128) {
    const float2 v = e4m3x2_f32<0>((uint32_t)(2 * tid) | ((uint32_t)(2 * tid + 1) << 8));
    lut[2 * tid] = v.x * a.ts;
    lut[2 * tid + 1] = v.y * a.ts;
  }
  pdl_wait();  // activations, residual and workspace may come from the preceding kernel
  if constexpr (kMma)
    stage_x_tok<M, kCT>(a, xs, pmax, sbase, nslots, tid, xissued);
  else
    stage_x<FMT, M, kCT>(a, xs, sums, sbase, nslots, tid, xissued);
  named_sync(1, kCT);

  // This warp's units: relative index i = C * chunk + ug, one per chunk, processed
  // in order; (stage, parity, activation slot) advance incrementally.  Within a unit the
  // warp takes half kh: quarters 2 kh, 2 kh + 1 (CUDA cores) or rows 64 kh .. 64 kh + 63
  // (tensor cores).
  const int ug = warp / kWPU, kh = warp % kWPU;
  bool ok = true;
  uint32_t i = (uint32_t)ug;
  int s = 0;
  uint32_t ph = 0;
  int slot = (int)((uu0 + i) % (uint32_t)KG) - sbase;
  if (slot < 0) slot += KG;
  uint32_t u = uu0;
  const uint32_t crank = clustered ? cluster_rank() : 0;
  uint32_t part_q0 = 0, part_q1 = 0;  // row tiles this CTA holds only part of
  int nparts = 0;
  const float ts_out = FMT == FMT_NVFP4 ? 1.0f : a.ts;  // the E4M3 table carries ts
  while (u < uu1) {
    const uint32_t q = u / (uint32_t)KG;
    const uint32_t seg_end = min(uu1, (q + 1) * (uint32_t)KG);
    float acc[4][M];
#pragma unroll
    for (int rt = 0; rt < 4; ++rt)
#pragma unroll
      for (int m = 0; m < M; ++m) acc[rt][m] = 0.0f;
    float acc2[2][2][4];  // tensor-core consumer (consume_mma), one set per 32-row quarter
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
      for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc2[h][j][i] = 0.0f;
    for (; ok && uu0 + i < seg_end; i += C) {
      if (!mbar_try_wait(&full[s], ph) && !mbar_wait_bounded(&full[s], ph, a.status)) {
        ok = false;
        break;
      }
      const uint8_t* st = stages + (size_t)s * SB;
      const uint32_t uu = uu0 + i;
      if constexpr (kMma) {
#pragma unroll
        for (int h = 0; h < 2; ++h)
          consume_mma<FMT, M>(st + ug * SG::CODE, st + C * SG::CODE + ug * SG::SCALE,
                              reinterpret_cast<const uint8_t*>(xs) + (size_t)slot * 128, (uint32_t)nslots * 128, lut,
                              2 * kh + h, lane, acc2[h]);
      } else {
        const uint8_t* aux = st + C * (SG::CODE + SG::SCALE) + ((uu >> 2) - ((uu - ug) >> 2)) * SG::AUX;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int kq = 2 * kh + h;
          const uint32_t* xr[M];
          const float* zr[M];
#pragma unroll
          for (int m = 0; m < M; ++m) {
            xr[m] = xs + (size_t)(m * nslots + slot) * 32 + kq * 8;
            zr[m] = sums + (size_t)(m * nslots + slot) * 16 + kq * 4;
          }
          consume<FMT, M>(st + ug * SG::CODE, st + C * SG::CODE + ug * SG::SCALE, aux, xr, zr, lut, kq, lane, acc);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
      if (++s == S) {
        s = 0;
        ph ^= 1u;
      }
      slot += C;
      while (slot >= KG) slot -= KG;
    }
    // Partials in shared memory: per warp (CUDA-core consumer) or per unit group (tensor-core
    // consumer: the four warps of a group own disjoint rows), summed below in fixed order.
    if constexpr (kMma) {
      const int g = lane >> 2, t = lane & 3;
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
          for (int i = 0; i < 4; ++i) acc2[h][j][i] += __shfl_xor_sync(0xFFFFFFFFu, acc2[h][j][i], 2);  // parities
      if (t < 2) {
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int j = 0; j < 2; ++j)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int m = 2 * t + (i & 1), row = 32 * (2 * kh + h) + 16 * j + g + 8 * (i >> 1);
              if (m < M) red[(ug * M + m) * 128 + row] = acc2[h][j][i];
            }
      }
    } else {
#pragma unroll
      for (int rt = 0; rt < 4; ++rt)
#pragma unroll
        for (int m = 0; m < M; ++m) red[(warp * M + m) * 128 + rt * 32 + lane] = acc[rt][m];
    }
    named_sync(1, kCT);

    const bool whole = (u == q * (uint32_t)KG) && (seg_end == (q + 1) * (uint32_t)KG);
    const int slot_ws = (u == uu0) ? 0 : 1;
    constexpr int kParts = kMma ? kGroups : kCW;
    for (int e = tid; e < M * 128; e += kCT) {
      float v = 0.0f;
#pragma unroll 4
      for (int w2 = 0; w2 < kParts; ++w2) v += red[w2 * M * 128 + e];
      if (kMma) v = mul_pow2(v, -tok_exp(pmax[e / 128]));  // back from the token's staging scale
      if (whole)
        finish_out<M>(a, q, e, v, ts_out);
      else if (clustered)  // into rank 0's buffer, slot = this CTA's rank
        st_cluster_f32(cluster_map(cbuf + (size_t)crank * M * 128 + e, 0), v);
      else
        a.ws_part[(size_t)((b * 2 + slot_ws) * M) * 128 + e] = v;
    }
    if (!whole && !clustered) {  // the same on every thread
      if (nparts == 0)
        part_q0 = q;
      else
        part_q1 = q;
      ++nparts;
    }
    named_sync(1, kCT);  // `red` is rewritten by the next segment
    u = seg_end;
  }

  // Row tiles split across CTAs (at most two per CTA: its first and its last): one ticket
  // each, taken after all of this CTA's work, so no ticket latency stalls the stream.  The
  // CTA that takes a tile's last ticket sums the tile's partials in CTA order (its first
  // contributor may hold the tile as its last segment, slot 1; every later contributor
  // starts inside the tile, slot 0) and writes the output.
  if (nparts > 0) {  // uniform: every consumer thread reaches the barriers below
    if (tid == 0) {
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        if (i >= nparts) break;
        const uint32_t q = i ? part_q1 : part_q0;
        const int64_t qk = (int64_t)q * KG;
        const int64_t bf = owner_cta(qk, U, G), bl = owner_cta(qk + KG - 1, U, G);
        const int old = ticket_add(&a.ws_cnt[q], 1);
        flag[i] = (old == (int)(bl - bf)) ? 1 : 0;
      }
    }
    named_sync(1, kCT);
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      if (i >= nparts || !flag[i]) continue;
      const uint32_t q = i ? part_q1 : part_q0;
      const int64_t qk = (int64_t)q * KG;
      const int64_t bf = owner_cta(qk, U, G), bl = owner_cta(qk + KG - 1, U, G);
      const int first_sl = (bf * U / G < qk) ? 1 : 0;
      const int nc = (int)(bl - bf + 1);
      const float* part = a.ws_part + (size_t)(bf * 2) * M * 128;
      for (int e = tid; e < M * 128; e += kCT) {
        float v = __ldcg(part + (size_t)first_sl * M * 128 + e);
        int c = 1;
        for (; c + 4 <= nc; c += 4) {  // independent loads, summed in order
          const float v0 = __ldcg(part + (size_t)(2 * c) * M * 128 + e);
          const float v1 = __ldcg(part + (size_t)(2 * c + 2) * M * 128 + e);
          const float v2 = __ldcg(part + (size_t)(2 * c + 4) * M * 128 + e);
          const float v3 = __ldcg(part + (size_t)(2 * c + 6) * M * 128 + e);
          v += v0;
          v += v1;
          v += v2;
          v += v3;
        }
        for (; c < nc; ++c) v += __ldcg(part + (size_t)(2 * c) * M * 128 + e);
        finish_out<M>(a, q, e, v, ts_out);
      }
      if (tid == 0) a.ws_cnt[q] = 0;
    }
  }
  if (clustered) {
    // Row tile q = this cluster: rank 0 sums the ranks' partials in rank order.
    __syncwarp();
    cluster_sync_all();
    if (crank == 0) {
      const uint32_t q = (uint32_t)(b / a.csplit);
      for (int e = tid; e < M * 128; e += kCT) {
        float v = cbuf[e];
        for (int r = 1; r < a.csplit; ++r) v += cbuf[(size_t)r * M * 128 + e];
        finish_out<M>(a, q, e, v, ts_out);
      }
    }
  }
}

// ---------------------------------------------------------------- host side
static int stage_bytes_of(int fmt, int m) {
  const int C = gemv_warps(fmt, m) / 2;  // units per chunk: one per two consumer warps
  switch (fmt) {
    case FMT_MLX: return Stage<FMT_MLX>::bytes(C);
    case FMT_MXFP4: return Stage<FMT_MXFP4>::bytes(C);
    case FMT_NVFP4: return Stage<FMT_NVFP4>::bytes(C);
    case FMT_Q50: return Stage<FMT_Q50>::bytes(C);
    case FMT_Q51: return Stage<FMT_Q51>::bytes(C);
    case FMT_Q5K: return Stage<FMT_Q5K>::bytes(C);
    default: return Stage<FMT_Q6K>::bytes(C);
  }
}

bool plan_gemv(const Geometry& g, int m, const DeviceInfo& dev, GemvPlan* p) {
  const int sbytes = stage_bytes_of(g.fmt, m);
  const int kcw = gemv_warps(g.fmt, m);
  const int C = kcw / 2;
  const int64_t U = g.nt * g.kg;
  if (U >= (int64_t(1) << 31)) return false;
  const size_t budget = (size_t)dev.max_smem_optin;
  int64_t G = std::min<int64_t>(dev.sms, U);
  int csplit = 1;
  if (g.nt < dev.sms && g.nt * 8 >= (int64_t)dev.sms * 7) {
    // Nearly one row tile per SM: every CTA takes one whole row tile -- no partials,
    // tickets or finishing pass, for a few idle SMs.
    G = g.nt;
  } else if (g.nt * 2 <= dev.sms) {
    // Few row tiles: split each across a cluster of csplit CTAs (equal K ranges); the
    // partials meet in the first CTA's shared memory instead of going through tickets.
    csplit = (int)std::min<int64_t>(kMaxCsplit, std::min<int64_t>(dev.sms / g.nt, g.kg));
    if (csplit > 1) G = g.nt * csplit;
  }
  for (;;) {
    const int64_t len = (U + G - 1) / G;
    const int nslots = (int)std::min<int64_t>(len, g.kg);
    const SmemLayout L0 = gemv_smem_layout(sbytes, 2, m, nslots, csplit, kcw);
    if (L0.total <= budget || G >= U) {
      if (L0.total > budget) return false;
      int S = (int)std::min<int64_t>((len + C - 1) / C, (int64_t)kMaxStages);
      S = std::max(S, 2);
      while (S > 2 && gemv_smem_layout(sbytes, S, m, nslots, csplit, kcw).total > budget) --S;
      p->grid = (int)G;
      p->nslots = nslots;
      p->stages = S;
      p->smem = gemv_smem_layout(sbytes, S, m, nslots, csplit, kcw).total;
      p->csplit = csplit;
      p->units = U;
      p->off_cnt = kWsHeader;
      p->off_part = kWsHeader + (((size_t)g.nt * 4 + 255) & ~(size_t)255);
      p->ws_bytes = p->off_part + (size_t)G * 2 * m * 128 * 4;
      return true;
    }
    if (csplit > 1) return false;  // cluster mode keeps its grid
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
  // Programmatic serialization: this launch may begin while the preceding kernel in the
  // stream finishes (the kernel waits for it before reading anything that kernel writes).
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)p.grid);
  cfg.blockDim = dim3((unsigned)(gemv_warps(FMT, M) * 32 + 32));
  cfg.dynamicSmemBytes = p.smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (p.csplit > 1) {
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = (unsigned)p.csplit;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.numAttrs = 2;
  }
  if (cudaLaunchKernelEx(&cfg, gemv_kernel<FMT, M>, a) != cudaSuccess) return QG_ERR_CUDA;
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
  a.csplit = p.csplit;
  uint8_t* wsb = static_cast<uint8_t*>(ws);
  a.status = reinterpret_cast<int*>(wsb);
  a.ws_cnt = reinterpret_cast<int*>(wsb + p.off_cnt);
  a.ws_part = reinterpret_cast<float*>(wsb + p.off_part);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  switch (g.fmt) {
    case FMT_MLX: return launch_m<FMT_MLX>(a, m, p, s);
    case FMT_MXFP4: return launch_m<FMT_MXFP4>(a, m, p, s);
    case FMT_NVFP4: return launch_m<FMT_NVFP4>(a, m, p, s);
    case FMT_Q50: return launch_m<FMT_Q50>(a, m, p, s);
    case FMT_Q51: return launch_m<FMT_Q51>(a, m, p, s);
    case FMT_Q5K: return launch_m<FMT_Q5K>(a, m, p, s);
    default: return launch_m<FMT_Q6K>(a, m, p, s);
  }
}

}  // namespace qg
