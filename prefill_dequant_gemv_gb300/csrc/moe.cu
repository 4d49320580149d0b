// Mixture-of-experts layer for 1..4 tokens (decode and speculative verify), in the five
// dependent launches of the TurboEXL3 article §4.2: route (route.cu), gate/up, mid, down,
// finish.  The shared expert runs as extra groups of the routed gate/up and down launches
// (§4.2: "extra grid rows of the routed launches").
//
//   gate/up  grouped GEMV: every active expert's 2F x H weights are read from HBM once
//            for all the tokens that chose it (§4.2: "two tokens that chose the same
//            expert share one decode of its weights"), fp32 results per (token, expert)
//   down     grouped GEMV on h = bf16( silu(gate) * up ) (§4.1 "Mid": SwiGLU in 32-bit),
//            which each CTA computes from the fp32 gate/up rows while staging its inputs
//            (only the rows of the experts it works on), so the mid step needs no launch of
//            its own; fp32 results per (token, expert)
//   finish   out[t] = bf16( sum_j p[t, j] * down_{e_j}[t] + shared[t] ) (§4.1 "Finish")
//
// The grouped GEMV is the dense GEMV's stream-K pipeline (qg_gemv_core.cuh) over a unit
// space of (group, 128-row tile, 64-input group) with groups = active experts (ascending)
// then the shared expert once per token; each group is padded to whole chunks so a chunk never spans two
// experts' weights.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>

#include "qg_common.cuh"
#include "qg_gemv_core.cuh"
#include "qg_internal.h"
#include "qg_route.h"
#include "qg_sync.cuh"

namespace qg {

constexpr int kGCW = 12;              // consumer warps (3 units per chunk, 128 registers a thread: no spills)
constexpr int kGCT = kGCW * 32;
constexpr int kGC = kGCW / 4;         // units per chunk
constexpr int kGThreads = kGCT + 32;
constexpr int kGMaxRows = 4;

struct GroupedArgs {
  const uint8_t* codes;
  const uint8_t* scales;
  const uint8_t* aux;
  int64_t cstride, sstride, astride;  // bytes per routed expert
  const uint8_t* sh_codes;            // shared expert (null when absent)
  const uint8_t* sh_scales;
  const uint8_t* sh_aux;
  float ts, sh_ts;
  int64_t n, k;
  int NT, KG;
  int T, topk;
  int mode;  // 0: input rows are tokens (x); 1: input rows are grouped pairs, shared rows
             // after: bf16 rows of x, or (gu non-null) the SwiGLU of the fp32 gate/up rows gu
  const __nv_bfloat16* x;
  int64_t ldx;
  const float* gu;
  int64_t ldg;
  int nrows;  // input rows (staging slots)
  float* out;
  int64_t ldo;
  const int* meta;
  const int* groups;  // router's group table (kGroupInts ints per active expert)
  int has_shared;
  int stages;
  float* ws_part;
  int* ws_cnt;
  int* status;
};

// Per-group description: weight base, rows (input row index, output row index), count.
struct GroupInfo {
  const uint8_t* codes;
  const uint8_t* scales;
  const uint8_t* aux;
  float ts;
  int m;
  int in_row[kGMaxRows];
  int out_row[kGMaxRows];
};
constexpr int kGInfoCache = 8;

struct GroupedSmem {
  size_t bars, stages, xs, sums, red, lut, misc, ginfo, total;
};

__host__ __device__ inline GroupedSmem grouped_smem(int stage_bytes, int S, int nrows, int KG) {
  GroupedSmem L;
  size_t o = 0;
  L.bars = o;
  o += (size_t)2 * S * 8;
  o = (o + 127) & ~(size_t)127;
  L.stages = o;
  o += (size_t)S * stage_bytes;
  o = (o + 127) & ~(size_t)127;
  L.xs = o;
  o += (size_t)nrows * KG * 128;  // f16 activations, all K
  L.sums = o;
  o += (size_t)nrows * KG * 64;   // {scale, Z, X, 0} per 16-input quarter
  L.red = o;
  o += (size_t)kGCW * kGMaxRows * 128 * 4;
  L.lut = o;
  o += 256 * 4;
  L.misc = o;
  o += 64;
  L.ginfo = o;  // descriptors of the first kGInfoCache groups this CTA touches
  o += (size_t)kGInfoCache * sizeof(GroupInfo);
  L.total = o;
  return L;
}

__device__ __forceinline__ GroupInfo group_info(const GroupedArgs& a, int g, int n_active) {
  GroupInfo gi;
  if (g < n_active) {  // one 32-byte entry of the router's group table
    const int4* ge = reinterpret_cast<const int4*>(a.groups + (size_t)g * kGroupInts);
    const int4 h = ge[0], rows = ge[1];
    const int e = h.x, first = h.y;
    gi.codes = a.codes + (int64_t)e * a.cstride;
    gi.scales = a.scales + (int64_t)e * a.sstride;
    gi.aux = a.aux ? a.aux + (int64_t)e * a.astride : nullptr;
    gi.ts = a.ts;
    gi.m = min(kGMaxRows, h.z);
    const int tok[kGroupRows] = {rows.x, rows.y, rows.z, rows.w};
#pragma unroll
    for (int i = 0; i < kGMaxRows; ++i) {
      const int j = min(i, gi.m - 1);
      gi.out_row[i] = first + j;
      gi.in_row[i] = a.mode == 0 ? tok[j] : first + j;
    }
  } else {  // shared expert, token t = g - n_active
    const int t = g - n_active;
    gi.codes = a.sh_codes;
    gi.scales = a.sh_scales;
    gi.aux = a.sh_aux;
    gi.ts = a.sh_ts;
    gi.m = 1;
#pragma unroll
    for (int i = 0; i < kGMaxRows; ++i) {
      gi.out_row[i] = a.T * a.topk + t;
      gi.in_row[i] = a.mode == 0 ? t : a.T * a.topk + t;
    }
  }
  return gi;
}

// Two SwiGLU outputs bf16( silu(g) * u ), silu(g) = g / (1 + e^-g) in IEEE fp32 (§4.1
// "Mid"), packed as a bf16 pair (first in the low half).
__device__ __forceinline__ uint32_t swiglu_bf16x2(float g0, float u0, float g1, float u1) {
  const float h0 = g0 / (1.0f + expf(-g0)) * u0, h1 = g1 / (1.0f + expf(-g1)) * u1;
  const __nv_bfloat162 b = __floats2bfloat162_rn(h0, h1);
  return *reinterpret_cast<const uint32_t*>(&b);
}

template <int FMT>
__global__ void __launch_bounds__(kGThreads, 1) grouped_gemv_kernel(const GroupedArgs a) {
  using SG = Stage<FMT>;
  extern __shared__ __align__(128) uint8_t smem[];
  const int S = a.stages, KG = a.KG, NT = a.NT;
  const int SBY = SG::bytes(kGC);
  const GroupedSmem L = grouped_smem(SBY, S, a.nrows, KG);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bars);
  uint64_t* empty = full + S;
  uint8_t* stages = smem + L.stages;
  uint32_t* xs = reinterpret_cast<uint32_t*>(smem + L.xs);
  float* sums = reinterpret_cast<float*>(smem + L.sums);
  float* red = reinterpret_cast<float*>(smem + L.red);
  float* lut = reinterpret_cast<float*>(smem + L.lut);
  int* flag = reinterpret_cast<int*>(smem + L.misc);
  GroupInfo* ginfo = reinterpret_cast<GroupInfo*>(smem + L.ginfo);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  for (int s = tid; s < S; s += blockDim.x) {
    mbar_init(&full[s], 1);
    mbar_init(&empty[s], kGCW);
  }
  if (tid < S) fence_mbar_init();
  __syncthreads();
  // The next launch of the chain may start its prologue now; everything below reads the
  // router's (or the previous step's) outputs, so wait for the preceding kernel first.
  if (tid == 0) pdl_launch_dependents();
  pdl_wait();

  const int n_active = a.meta[0];
  // The shared expert runs as one single-row group per token: its weights are read once per
  // token (the repeats hit L2) but every chunk then costs the same, so the equal split of
  // chunks over CTAs stays balanced (a 4-row chunk costs ~2.4 one-row chunks).
  const int n_groups = n_active + (a.has_shared ? a.T : 0);
  const int upg_real = NT * KG;
  const int cpg = (upg_real + kGC - 1) / kGC;  // chunks per group
  const int upg = cpg * kGC;                   // padded units per group
  const int64_t NCH = (int64_t)n_groups * cpg;
  // Only as many CTAs as chunks take part, so every participating CTA owns at least one
  // chunk and the contributors to a split row tile are consecutive CTAs.
  const int64_t G = min((int64_t)gridDim.x, NCH), b = blockIdx.x;
  if (b >= G) return;
  const int64_t c0 = b * NCH / G, c1 = (b + 1) * NCH / G;
  const uint32_t uu0 = (uint32_t)(c0 * kGC), uu1 = (uint32_t)(c1 * kGC);
  const int nch = (int)(c1 - c0);

  if (warp == kGCW) {  // producer: chunks never span two groups
    if (lane == 0) {
      int s = 0;
      uint32_t ph = 0;
      int gcur = -1;  // the group whose weight bases are loaded (reloaded only on a change)
      const uint8_t *bc = nullptr, *bs = nullptr, *ba = nullptr;
      for (int j = 0; j < nch; ++j) {
        if (j >= S && !mbar_wait_bounded(&empty[s], ph ^ 1u, a.status)) break;
        const int64_t c = c0 + j;
        const int g = (int)(c / cpg);
        const int l0 = (int)(c % cpg) * kGC;
        const int nu = min(kGC, upg_real - l0);
        if (g != gcur) {
          gcur = g;
          if (g < n_active) {
            const int e = a.groups[(size_t)g * kGroupInts];
            bc = a.codes + (int64_t)e * a.cstride;
            bs = a.scales + (int64_t)e * a.sstride;
            ba = a.aux ? a.aux + (int64_t)e * a.astride : nullptr;
          } else {
            bc = a.sh_codes;
            bs = a.sh_scales;
            ba = a.sh_aux;
          }
        }
        uint8_t* dst = stages + (size_t)s * SBY;
        uint32_t bytes = (uint32_t)nu * (SG::CODE + SG::SCALE);
        int aux_a = 0, aux_n = 0;
        if (SG::AUX) {
          aux_a = l0 >> 2;
          aux_n = ((l0 + nu - 1) >> 2) - aux_a + 1;
          bytes += (uint32_t)aux_n * SG::AUX;
        }
        mbar_arrive_expect_tx(&full[s], bytes);
        bulk_g2s(dst, bc + (size_t)l0 * SG::CODE, (uint32_t)nu * SG::CODE, &full[s]);
        bulk_g2s(dst + kGC * SG::CODE, bs + (size_t)l0 * SG::SCALE, (uint32_t)nu * SG::SCALE, &full[s]);
        if (SG::AUX)
          bulk_g2s(dst + kGC * (SG::CODE + SG::SCALE), ba + (size_t)aux_a * SG::AUX, (uint32_t)aux_n * SG::AUX,
                   &full[s]);
        if (++s == S) {
          s = 0;
          ph ^= 1u;
        }
      }
    }
    return;
  }

  if (FMT == FMT_NVFP4 && tid < 128) {
    const float2 v = e4m3x2_f32<0>((uint32_t)(2 * tid) | ((uint32_t)(2 * tid + 1) << 8));
    lut[2 * tid] = v.x;
    lut[2 * tid + 1] = v.y;
  }
  // The groups this CTA touches: their descriptors are read once here instead of at every
  // segment.
  const int g_first = (int)(uu0 / (uint32_t)upg);
  const int g_span = (int)((uu1 - 1) / (uint32_t)upg) - g_first + 1;
  if (tid < kGInfoCache && g_first + tid < n_groups) ginfo[tid] = group_info(a, g_first + tid, n_active);
  // Stage the input rows over all of K.  Mode 0: every token row of x.  Mode 1: the rows of
  // the groups this CTA touches (all rows if it touches more than kGInfoCache groups), each
  // computed as h = bf16( silu(g) * u ) from the fp32 gate/up outputs.
  const bool by_group = a.mode == 1 && g_span <= kGInfoCache;
  if (a.mode == 1) named_sync(1, kGCT);  // the row lists come from the descriptors
  const int nslot = by_group ? g_span * kGMaxRows : a.nrows;
  for (int it = tid; it < nslot * KG * 4; it += kGCT) {
    const int kq = it & 3, sl = (it >> 2) % KG, slot = (it >> 2) / KG;
    int row = slot;
    if (by_group) {
      const GroupInfo& gs = ginfo[slot / kGMaxRows];
      if (slot % kGMaxRows >= gs.m) continue;
      row = gs.in_row[slot % kGMaxRows];
    }
    const int64_t k0 = (int64_t)sl * 64 + kq * 16;
    uint32_t u[8];
    if (k0 >= a.k) {
#pragma unroll
      for (int i = 0; i < 8; ++i) u[i] = 0;
    } else if (a.gu == nullptr) {  // bf16 rows of x (mode 0) or of h (mode 1, staged calls)
      const uint4* src = reinterpret_cast<const uint4*>(a.x + (int64_t)row * a.ldx + k0);
      const uint4 r0 = src[0], r1 = src[1];
      u[0] = r0.x; u[1] = r0.y; u[2] = r0.z; u[3] = r0.w;
      u[4] = r1.x; u[5] = r1.y; u[6] = r1.z; u[7] = r1.w;
    } else {
      const float4* gp = reinterpret_cast<const float4*>(a.gu + (int64_t)row * a.ldg + k0);
      const float4* up = reinterpret_cast<const float4*>(a.gu + (int64_t)row * a.ldg + a.k + k0);
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        const float4 g4 = __ldcg(gp + q4), u4 = __ldcg(up + q4);
        u[2 * q4] = swiglu_bf16x2(g4.x, u4.x, g4.y, u4.y);
        u[2 * q4 + 1] = swiglu_bf16x2(g4.z, u4.z, g4.w, u4.w);
      }
    }
    const float4 z = stage_quarter<FMT>(u, xs + (size_t)(row * KG + sl) * 32 + kq * 8);
    reinterpret_cast<float4*>(sums)[(size_t)(row * KG + sl) * 4 + kq] = z;
  }
  named_sync(1, kGCT);

  const int ug = warp >> 2, kq = warp & 3;
  bool ok = true;
  uint32_t i = (uint32_t)ug;  // relative unit index; one per chunk
  int s = 0;
  uint32_t ph = 0;
  uint32_t u = uu0;
  int nparts = 0;  // segments of row tiles this CTA holds only part of (at most 2)
  int pg0 = 0, pq0 = 0, pg1 = 0, pq1 = 0;
  uint32_t ps0 = 0, pe0 = 0, ps1 = 0, pe1 = 0;
  while (u < uu1) {
    const uint32_t g = u / (uint32_t)upg;
    const uint32_t l = u - g * (uint32_t)upg;
    const uint32_t q = min(l / (uint32_t)KG, (uint32_t)(NT - 1));
    const uint32_t seg_start = g * upg + q * KG;
    const uint32_t seg_end_full = (q == (uint32_t)(NT - 1)) ? (g + 1) * upg : seg_start + KG;
    const uint32_t seg_end = min(uu1, seg_end_full);
    const GroupInfo gi = ((int)g - g_first < kGInfoCache) ? ginfo[(int)g - g_first] : group_info(a, (int)g, n_active);
    float acc[4][kGMaxRows];
#pragma unroll
    for (int rt = 0; rt < 4; ++rt)
#pragma unroll
      for (int m = 0; m < kGMaxRows; ++m) acc[rt][m] = 0.0f;
    const uint32_t* xr[kGMaxRows];
    const float* zr[kGMaxRows];
    for (; ok && uu0 + i < seg_end; i += kGC) {
      if (!mbar_wait_bounded(&full[s], ph, a.status)) {
        ok = false;
        break;
      }
      const uint32_t uu = uu0 + i;
      const int ul = (int)(uu - g * upg);
      if (ul < upg_real) {  // padding units carry no data
        const int kg = ul % KG;
        const uint8_t* st = stages + (size_t)s * SBY;
        const int l0 = ul - ug;  // first unit of this chunk within the group
        const uint8_t* aux = st + kGC * (SG::CODE + SG::SCALE) + ((ul >> 2) - (l0 >> 2)) * SG::AUX;
#pragma unroll
        for (int m = 0; m < kGMaxRows; ++m) {
          xr[m] = xs + (size_t)(gi.in_row[m] * KG + kg) * 32 + kq * 8;
          zr[m] = sums + ((size_t)(gi.in_row[m] * KG + kg) * 4 + kq) * 4;
        }
        const uint8_t* cst = st + ug * SG::CODE;
        const uint8_t* sst = st + kGC * SG::CODE + ug * SG::SCALE;
        switch (gi.m) {
          case 1: consume<FMT, 1, kGMaxRows>(cst, sst, aux, xr, zr, lut, kq, lane, acc); break;
          case 2: consume<FMT, 2, kGMaxRows>(cst, sst, aux, xr, zr, lut, kq, lane, acc); break;
          case 3: consume<FMT, 3, kGMaxRows>(cst, sst, aux, xr, zr, lut, kq, lane, acc); break;
          default: consume<FMT, 4, kGMaxRows>(cst, sst, aux, xr, zr, lut, kq, lane, acc); break;
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
      if (++s == S) {
        s = 0;
        ph ^= 1u;
      }
    }
#pragma unroll
    for (int rt = 0; rt < 4; ++rt)
#pragma unroll
      for (int m = 0; m < kGMaxRows; ++m) red[(warp * kGMaxRows + m) * 128 + rt * 32 + lane] = acc[rt][m];
    named_sync(1, kGCT);

    const int M = gi.m;
    const bool whole = (u == seg_start) && (seg_end == seg_end_full);
    const int slot_ws = (u == uu0) ? 0 : 1;
    for (int e = tid; e < M * 128; e += kGCT) {
      float v = 0.0f;
#pragma unroll 4
      for (int w2 = 0; w2 < kGCW; ++w2) v += red[w2 * kGMaxRows * 128 + e];
      v *= gi.ts;
      if (whole) {
        const int64_t n = (int64_t)q * 128 + (e & 127);
        if (n < a.n) a.out[(int64_t)gi.out_row[e >> 7] * a.ldo + n] = v;
      } else {
        a.ws_part[(size_t)((b * 2 + slot_ws) * kGMaxRows) * 128 + e] = v;
      }
    }
    if (!whole) {  // the same on every thread: settled after all of this CTA's work
      if (nparts == 0) {
        pg0 = (int)g; pq0 = (int)q; ps0 = seg_start; pe0 = seg_end_full;
      } else {
        pg1 = (int)g; pq1 = (int)q; ps1 = seg_start; pe1 = seg_end_full;
      }
      ++nparts;
    }
    named_sync(1, kGCT);
    u = seg_end;
  }

  // Row tiles split across CTAs (at most two per CTA): one ticket each, taken after all of
  // this CTA's work; the CTA that takes a segment's last ticket sums its partials in CTA
  // order (the first contributor may hold it as its last segment, slot 1).
  if (nparts > 0) {  // uniform: every consumer thread reaches the barriers below
    if (tid == 0) {
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        if (i >= nparts) break;
        const int pg = i ? pg1 : pg0, pq = i ? pq1 : pq0;
        const uint32_t ps = i ? ps1 : ps0, pe = i ? pe1 : pe0;
        const int64_t cs = ps / kGC, ce = (pe - 1) / kGC;
        const int64_t bf = ((cs + 1) * G - 1) / NCH, bl = ((ce + 1) * G - 1) / NCH;
        const int old = ticket_add(&a.ws_cnt[(int64_t)pg * NT + pq], 1);
        flag[i] = (old == (int)(bl - bf)) ? 1 : 0;
      }
    }
    named_sync(1, kGCT);
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      if (i >= nparts || !flag[i]) continue;
      const int pg = i ? pg1 : pg0, pq = i ? pq1 : pq0;
      const uint32_t ps = i ? ps1 : ps0, pe = i ? pe1 : pe0;
      const GroupInfo gi = (pg - g_first < kGInfoCache) ? ginfo[pg - g_first] : group_info(a, pg, n_active);
      const int64_t cs = ps / kGC, ce = (pe - 1) / kGC;
      const int64_t bf = ((cs + 1) * G - 1) / NCH, bl = ((ce + 1) * G - 1) / NCH;
      const int first_sl = ((bf * NCH / G) * kGC < (int64_t)ps) ? 1 : 0;
      const int nc = (int)(bl - bf + 1);
      const float* part = a.ws_part + (size_t)(bf * 2) * kGMaxRows * 128;
      for (int e = tid; e < gi.m * 128; e += kGCT) {
        float v = __ldcg(part + (size_t)first_sl * kGMaxRows * 128 + e);
        for (int c = 1; c < nc; ++c) v += __ldcg(part + (size_t)(2 * c) * kGMaxRows * 128 + e);
        const int64_t n = (int64_t)pq * 128 + (e & 127);
        if (n < a.n) a.out[(int64_t)gi.out_row[e >> 7] * a.ldo + n] = v;
      }
      if (tid == 0) a.ws_cnt[(int64_t)pg * NT + pq] = 0;
    }
  }
}

// h[r][f] = bf16( silu(gu[r][f]) * gu[r][F + f] ) for every row (the staged gate/up call
// writes h for the caller; the fused chain computes it inside the down GEMV instead).
__global__ void __launch_bounds__(256) mid_kernel(const float* gu, int64_t ldg, __nv_bfloat16* h, int64_t ldh, int F,
                                                  int rows) {
  pdl_launch_dependents();
  pdl_wait();
  const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= (int64_t)rows * (F / 2)) return;
  const int r = (int)(idx / (F / 2)), f = (int)(idx % (F / 2)) * 2;
  const float2 g = *reinterpret_cast<const float2*>(gu + r * ldg + f);
  const float2 u = *reinterpret_cast<const float2*>(gu + r * ldg + F + f);
  *reinterpret_cast<uint32_t*>(h + r * ldh + f) = swiglu_bf16x2(g.x, u.x, g.y, u.y);
}

// out[t][n] = bf16( sum_j w[t][j] * d[pos(t, j)][n] + g_t * d[T*topk + t][n] ), fixed order,
// four features per thread (g_t: the shared expert's sigmoid gate, or 1); every load of a
// thread is issued before the first multiply-add.
__global__ void __launch_bounds__(256) finish_kernel(const float* d, int64_t ldd, const float* w, const int* pair_pos,
                                                     int T, int topk, int has_shared, const float* shared_gate,
                                                     int64_t H, __nv_bfloat16* out, int64_t ldo) {
  pdl_launch_dependents();
  pdl_wait();
  const int64_t H4 = H / 4;
  const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= (int64_t)T * H4) return;
  const int t = (int)(idx / H4);
  const int64_t n = (idx % H4) * 4;
  int pos[kMaxTopk];
  float p[kMaxTopk];
#pragma unroll
  for (int j = 0; j < kMaxTopk; ++j) {
    pos[j] = j < topk ? pair_pos[t * topk + j] : 0;
    p[j] = j < topk ? w[t * topk + j] : 0.0f;
  }
  float4 v[kMaxTopk];
#pragma unroll
  for (int j = 0; j < kMaxTopk; ++j)
    v[j] = j < topk ? __ldcg(reinterpret_cast<const float4*>(d + (int64_t)pos[j] * ldd + n)) : make_float4(0, 0, 0, 0);
  const float4 sh = has_shared ? __ldcg(reinterpret_cast<const float4*>(d + (int64_t)(T * topk + t) * ldd + n))
                               : make_float4(0, 0, 0, 0);
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int j = 0; j < kMaxTopk; ++j) {
    if (j < topk) {
      acc.x = fmaf(p[j], v[j].x, acc.x);
      acc.y = fmaf(p[j], v[j].y, acc.y);
      acc.z = fmaf(p[j], v[j].z, acc.z);
      acc.w = fmaf(p[j], v[j].w, acc.w);
    }
  }
  if (has_shared) {
    const float g = shared_gate_weight(shared_gate, t);
    acc.x = fmaf(g, sh.x, acc.x);
    acc.y = fmaf(g, sh.y, acc.y);
    acc.z = fmaf(g, sh.z, acc.z);
    acc.w = fmaf(g, sh.w, acc.w);
  }
  const __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y), hi = __floats2bfloat162_rn(acc.z, acc.w);
  uint2 pk;
  pk.x = *reinterpret_cast<const uint32_t*>(&lo);
  pk.y = *reinterpret_cast<const uint32_t*>(&hi);
  *reinterpret_cast<uint2*>(out + (int64_t)t * ldo + n) = pk;
}

// ---------------------------------------------------------------- host side
namespace {
int grouped_stage_bytes(int fmt) {
  switch (fmt) {
    case FMT_MLX: return Stage<FMT_MLX>::bytes(kGC);
    case FMT_MXFP4: return Stage<FMT_MXFP4>::bytes(kGC);
    case FMT_NVFP4: return Stage<FMT_NVFP4>::bytes(kGC);
    default: return Stage<FMT_Q6K>::bytes(kGC);
  }
}
}  // namespace

MoeLayout moe_layout(const Geometry& gu, const Geometry& dn, int64_t T, int E, int topk, int grid) {
  MoeLayout L;
  const int64_t R = T * topk + T;
  size_t o = kWsHeader;
  auto take = [&o](size_t bytes) {
    const size_t at = o;
    o += (bytes + 255) & ~(size_t)255;
    return at;
  };
  // the prefill chain (more than kGMaxRows tokens) fuses the mid into the gate/up GEMM and
  // needs neither the split-K tickets and partials nor the fp32 gate/up rows
  const bool decode = T <= kGMaxRows;
  const int64_t nt_max = std::max(gu.nt, dn.nt);
  L.cnt = take(decode ? (size_t)(E + kGMaxRows) * nt_max * 4 : 0);  // tickets per (group, row tile)
  L.part = take(decode ? (size_t)grid * 2 * kGMaxRows * 128 * 4 : 0);
  L.ld_gu = (gu.n + 7) / 8 * 8;
  L.gu = take(decode ? (size_t)R * L.ld_gu * 4 : 0);
  L.ld_h = (dn.k + 7) / 8 * 8;
  L.h = take(decode ? 0 : (size_t)R * L.ld_h * 2);  // decode: h never leaves the down GEMV
  L.ld_d = (dn.n + 7) / 8 * 8;
  L.d = take((size_t)R * L.ld_d * 4);
  L.total = o;
  return L;
}

static int launch_grouped(int fmt, const GroupedArgs& a0, int nrows, int KG, const DeviceInfo& dev, cudaStream_t s) {
  GroupedArgs a = a0;
  const int sb = grouped_stage_bytes(fmt);
  const size_t fixed = grouped_smem(sb, 0, nrows, KG).total;
  if (fixed + 2 * (size_t)sb + 256 > (size_t)dev.max_smem_optin) return QG_ERR_UNSUPPORTED;
  int S = (int)std::min<size_t>(24, ((size_t)dev.max_smem_optin - fixed - 256) / ((size_t)sb + 16));
  while (S > 2 && grouped_smem(sb, S, nrows, KG).total > (size_t)dev.max_smem_optin) --S;
  a.stages = S;
  a.nrows = nrows;
  const size_t smem = grouped_smem(sb, S, nrows, KG).total;
  static std::atomic<unsigned long long> configured[5];
  int devid = 0;
  if (cudaGetDevice(&devid) != cudaSuccess) return QG_ERR_CUDA;
  const unsigned long long bit = 1ull << (devid & 63);
  const void* fn = nullptr;
  switch (fmt) {
    case FMT_MLX: fn = (const void*)grouped_gemv_kernel<FMT_MLX>; break;
    case FMT_MXFP4: fn = (const void*)grouped_gemv_kernel<FMT_MXFP4>; break;
    case FMT_NVFP4: fn = (const void*)grouped_gemv_kernel<FMT_NVFP4>; break;
    default: fn = (const void*)grouped_gemv_kernel<FMT_Q6K>; break;
  }
  if (!(configured[fmt].load() & bit)) {
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, dev.max_smem_optin) != cudaSuccess)
      return QG_ERR_CUDA;
    configured[fmt].fetch_or(bit);
  }
  const dim3 grid(dev.sms), block(kGThreads);
  cudaError_t e;
  switch (fmt) {
    case FMT_MLX: e = launch_pdl(grouped_gemv_kernel<FMT_MLX>, grid, block, smem, s, a); break;
    case FMT_MXFP4: e = launch_pdl(grouped_gemv_kernel<FMT_MXFP4>, grid, block, smem, s, a); break;
    case FMT_NVFP4: e = launch_pdl(grouped_gemv_kernel<FMT_NVFP4>, grid, block, smem, s, a); break;
    default: e = launch_pdl(grouped_gemv_kernel<FMT_Q6K>, grid, block, smem, s, a); break;
  }
  return (e == cudaSuccess && cudaGetLastError() == cudaSuccess) ? QG_OK : QG_ERR_CUDA;
}

int launch_moe_decode(const qg_moe_layer* m, const Geometry& gu, const Geometry& dn, const void* x, int64_t T,
                      int64_t ldx, int topk, const float* topk_w, const float* shared_gate, const void* route_ws,
                      void* out, int64_t ldo, void* ws, const DeviceInfo& dev, void* stream, int stage) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const RouteView rv = route_view(const_cast<void*>(route_ws), T, m->n_experts, topk);
  const MoeLayout L = moe_layout(gu, dn, T, m->n_experts, topk, dev.sms);
  uint8_t* w = static_cast<uint8_t*>(ws);
  size_t cb = 0, sb = 0, ab = 0;
  qg_packed_sizes(m->fmt, gu.n, gu.k, &cb, &sb, &ab);
  GroupedArgs a{};
  a.codes = static_cast<const uint8_t*>(m->gu_codes);
  a.scales = static_cast<const uint8_t*>(m->gu_scales);
  a.aux = static_cast<const uint8_t*>(m->gu_aux);
  a.cstride = (int64_t)cb;
  a.sstride = (int64_t)sb;
  a.astride = (int64_t)ab;
  a.has_shared = m->has_shared;
  a.sh_codes = m->has_shared ? static_cast<const uint8_t*>(m->shared_gate_up.codes) : nullptr;
  a.sh_scales = m->has_shared ? static_cast<const uint8_t*>(m->shared_gate_up.scales) : nullptr;
  a.sh_aux = m->has_shared ? static_cast<const uint8_t*>(m->shared_gate_up.aux) : nullptr;
  a.ts = (m->fmt == FMT_NVFP4) ? m->tensor_scale : 1.0f;
  a.sh_ts = (m->has_shared && m->fmt == FMT_NVFP4) ? m->shared_gate_up.tensor_scale : 1.0f;
  a.n = gu.n;
  a.k = gu.k;
  a.NT = (int)gu.nt;
  a.KG = (int)gu.kg;
  a.T = (int)T;
  a.topk = topk;
  a.mode = 0;
  a.x = static_cast<const __nv_bfloat16*>(x);
  a.ldx = ldx;
  a.out = reinterpret_cast<float*>(w + L.gu);
  a.ldo = L.ld_gu;
  a.meta = rv.meta;
  a.groups = rv.groups;
  a.ws_part = reinterpret_cast<float*>(w + L.part);
  a.ws_cnt = reinterpret_cast<int*>(w + L.cnt);
  a.status = reinterpret_cast<int*>(w);
  const int rows = (int)(T * topk + (m->has_shared ? T : 0));
  int st = QG_OK;
  if (stage != kMoeDown) {
    st = launch_grouped(m->fmt, a, (int)T, (int)gu.kg, dev, s);
    if (st != QG_OK) return st;
  }
  if (stage == kMoeGateUp) {  // h for the caller: out [rows][ldo] bf16
    const int F = (int)dn.k;
    if (launch_pdl(mid_kernel, dim3((unsigned)(((int64_t)rows * (F / 2) + 255) / 256)), dim3(256), 0, s,
                   (const float*)reinterpret_cast<const float*>(w + L.gu), (int64_t)L.ld_gu,
                   static_cast<__nv_bfloat16*>(out), ldo, F, rows) != cudaSuccess)
      return QG_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? QG_OK : QG_ERR_CUDA;
  }

  qg_packed_sizes(m->fmt, dn.n, dn.k, &cb, &sb, &ab);
  GroupedArgs d = a;
  d.codes = static_cast<const uint8_t*>(m->dn_codes);
  d.scales = static_cast<const uint8_t*>(m->dn_scales);
  d.aux = static_cast<const uint8_t*>(m->dn_aux);
  d.cstride = (int64_t)cb;
  d.sstride = (int64_t)sb;
  d.astride = (int64_t)ab;
  d.sh_codes = m->has_shared ? static_cast<const uint8_t*>(m->shared_down.codes) : nullptr;
  d.sh_scales = m->has_shared ? static_cast<const uint8_t*>(m->shared_down.scales) : nullptr;
  d.sh_aux = m->has_shared ? static_cast<const uint8_t*>(m->shared_down.aux) : nullptr;
  d.sh_ts = (m->has_shared && m->fmt == FMT_NVFP4) ? m->shared_down.tensor_scale : 1.0f;
  d.n = dn.n;
  d.k = dn.k;
  d.NT = (int)dn.nt;
  d.KG = (int)dn.kg;
  d.mode = 1;
  if (stage == kMoeDown) {  // h from the caller's gate/up call
    d.x = static_cast<const __nv_bfloat16*>(x);
    d.ldx = ldx;
    d.gu = nullptr;
  } else {  // fused: SwiGLU of the fp32 gate/up rows while staging
    d.x = nullptr;
    d.gu = reinterpret_cast<const float*>(w + L.gu);
    d.ldg = L.ld_gu;
  }
  d.out = reinterpret_cast<float*>(w + L.d);
  d.ldo = L.ld_d;
  st = launch_grouped(m->fmt, d, rows, (int)dn.kg, dev, s);
  if (st != QG_OK) return st;

  if (launch_pdl(finish_kernel, dim3((unsigned)((T * (dn.n / 4) + 255) / 256)), dim3(256), 0, s,
                 (const float*)reinterpret_cast<const float*>(w + L.d), (int64_t)L.ld_d, topk_w,
                 (const int*)rv.pair_pos, (int)T, topk, (int)m->has_shared, shared_gate, (int64_t)dn.n,
                 static_cast<__nv_bfloat16*>(out), ldo) != cudaSuccess)
    return QG_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? QG_OK : QG_ERR_CUDA;
}

}  // namespace qg
