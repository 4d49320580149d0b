// Mixture-of-experts layer for 1..4 tokens (decode and speculative verify), in the five
// dependent launches of the TurboEXL3 article §4.2: route (route.cu), gate/up, mid, down,
// finish.  The shared expert runs as one more group of the routed gate/up and down launches
// (as §4.2 runs it inside the routed launches).
//
//   gate/up  grouped GEMV: every active expert's 2F x H weights are read from HBM and
//            decoded once for all the tokens that chose it (§4.2), fp32 results per
//            (token, expert)
//   down     grouped GEMV on h = bf16( silu(gate) * up ) (§4.1 "Mid": SwiGLU in 32-bit),
//            which each CTA computes from the fp32 gate/up rows while staging its inputs
//            (only the rows of the experts it works on), so the mid step needs no launch of
//            its own; fp32 results per (token, expert)
//   finish   out[t] = bf16( sum_j p[t, j] * down_{e_j}[t] + shared[t] ) (§4.1 "Finish")
//
// The grouped GEMV runs the dense GEMV's decode (qg_gemv_core.cuh) over the units (group,
// 128-row tile, 64 inputs) of groups = active experts (ascending), then the shared expert as
// one group of all the tokens.  Each CTA takes a contiguous share of the units of equal cost
// (stream-K weighted by unit_cost, so the CTAs finish together whatever the routing); its 12
// consumer warps hand each row tile's partials to two reducer warps (two buffers, so they
// run on).  A row tile cut
// by a share boundary is written as one output part per CTA (parts past the last piece are
// zero), and the parts are summed by whoever reads the output next, in part order.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <type_traits>

#include "qg_common.cuh"
#include "qg_gemv_core.cuh"
#include "qg_internal.h"
#include "qg_route.h"
#include "qg_route_dev.cuh"
#include "qg_sync.cuh"

namespace qg {

constexpr int kGCW = 12;              // consumer warps (128 registers a thread: no spills)
constexpr int kGCT = kGCW * 32;
constexpr int kGC = kGCW / 2;         // units per chunk: two warps per unit, two quarters each
constexpr int kGRW = 2;               // reducer warps
constexpr int kGThreads = kGCT + 32 + 32 * kGRW;  // + the producer warp and the reducer warps
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
  int P;  // output parts: a row tile split over CTAs writes one part per CTA, the rest zero
  int T, topk;
  int mode;  // 0: input rows are tokens (x); 1: input rows are grouped pairs, shared rows
             // after: bf16 rows of x, or (gu non-null) the SwiGLU of the fp32 gate/up rows gu
  const __nv_bfloat16* x;
  int64_t ldx;
  const float* gu;      // gu_parts partial sums of the gate/up rows, gu_pstride floats apart
  int64_t ldg;
  int gu_parts;
  int64_t gu_pstride;
  int gu_nt, gu_kg;     // the gate/up launch's row tiles and 64-input groups (its pieces per tile)
  int nrows;  // input rows (staging slots)
  float* out;  // P partial outputs, out_pstride floats apart
  int64_t ldo;
  int64_t out_pstride;
  const int* meta;
  const int* groups;  // router's group table (kGroupInts ints per active expert)
  // Routing inside the launch (decode gate/up from logits; null: the router's outputs above):
  // every CTA routes the T tokens itself; CTA 0 also stores the router's outputs.
  const float* logits;
  int E;
  int32_t* ids_out;
  float* wts_out;
  RouteView rv;
  int has_shared;
  int stages;
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
  int w;          // cost of one unit (unit_cost(m))
  int cu;         // cost of the groups before this one, per unit of a group
  uint32_t cbase;  // cost of all the units of the groups before this one (units a group x cu)
};
constexpr int kGInfoCache = 8;

// Relative cost of one unit of a group of m rows on the CUDA-core consumer: the decode is
// paid once, the multiply-adds and folds once per row (measured 1 : 1.44 : 1.88 : 2.34 for
// 1..4 rows in the dense GEMV's consume loop).
__host__ __device__ constexpr int unit_cost(int m) { return 2 * m + 3; }

struct GroupedSmem {
  size_t bars, stages, xs, sums, red, lut, misc, ginfo, gpc, route, total;
};
constexpr int kGPcTiles = 64;  // gate/up row tiles a pieces table covers

// Shared memory: mbarriers (full[S], empty[S], rfull[2], rempty[2]), the stage ring, the
// staged activations, two reduction buffers (one per tile piece in flight), the E4M3 table,
// the descriptors of the first groups the CTA touches, the down launch's table of gate/up
// parts per tile, and the routing scratch (group table).
__host__ __device__ inline GroupedSmem grouped_smem(int stage_bytes, int S, int nrows, int KG) {
  GroupedSmem L;
  size_t o = 0;
  L.bars = o;
  o += (size_t)(2 * S + 4) * 8;
  o = (o + 127) & ~(size_t)127;
  L.stages = o;
  o += (size_t)S * stage_bytes;
  o = (o + 127) & ~(size_t)127;
  L.xs = o;
  o += (size_t)nrows * KG * 128;  // f16 activations, all K
  L.sums = o;
  o += (size_t)nrows * KG * 64;   // {scale, Z, X, 0} per 16-input quarter
  L.red = o;
  o += (size_t)2 * kGCW * kGMaxRows * 128 * 4;
  L.lut = o;
  o += 256 * 4;
  L.misc = o;
  o += 64;
  L.ginfo = o;  // descriptors of the first kGInfoCache groups this CTA touches
  o += (size_t)kGInfoCache * sizeof(GroupInfo);
  L.gpc = o;  // down launch: pieces of each gate/up row tile of the cached groups
  o += (size_t)kGInfoCache * kGPcTiles;
  o = (o + 15) & ~(size_t)15;
  L.route = o;  // routing scratch and group table when the launch routes its tokens
  o += sizeof(BlockRouteSmem);
  L.total = o;
  return L;
}

// Descriptor of group g (UG units a group).  The cost before group g in closed form: the
// groups before it hold `first` pairs (rows) between them, so their units cost
// UG * (2 first + 3 g); the shared group follows all T * topk pairs.
__device__ __forceinline__ GroupInfo group_info(const GroupedArgs& a, const int* groups, int g, int n_active, int UG) {
  GroupInfo gi;
  if (g < n_active) {  // one 32-byte entry of the router's group table
    const int4* ge = reinterpret_cast<const int4*>(groups + (size_t)g * kGroupInts);
    const int4 h = ge[0], rows = ge[1];
    const int e = h.x, first = h.y;
    gi.codes = a.codes + (int64_t)e * a.cstride;
    gi.scales = a.scales + (int64_t)e * a.sstride;
    gi.aux = a.aux ? a.aux + (int64_t)e * a.astride : nullptr;
    gi.ts = a.ts;
    gi.m = min(kGMaxRows, h.z);
    gi.w = unit_cost(gi.m);
    gi.cu = 2 * first + 3 * g;
    gi.cbase = (uint32_t)UG * (uint32_t)gi.cu;
    const int tok[kGroupRows] = {rows.x, rows.y, rows.z, rows.w};
#pragma unroll
    for (int i = 0; i < kGMaxRows; ++i) {
      const int j = min(i, gi.m - 1);
      gi.out_row[i] = first + j;
      gi.in_row[i] = a.mode == 0 ? tok[j] : first + j;
    }
  } else {  // the shared expert: one group of all T tokens
    gi.codes = a.sh_codes;
    gi.scales = a.sh_scales;
    gi.aux = a.sh_aux;
    gi.ts = a.sh_ts;
    gi.m = a.T;
    gi.w = unit_cost(a.T);
    gi.cu = 2 * a.T * a.topk + 3 * n_active;
    gi.cbase = (uint32_t)UG * (uint32_t)gi.cu;
#pragma unroll
    for (int i = 0; i < kGMaxRows; ++i) {
      const int t = min(i, a.T - 1);
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

// The CTA's chunks, in order: at most kGC consecutive units of one group (a chunk may span
// row tiles of its group, never two groups, whose weights lie apart).
struct ChunkIter {
  int c0, c1;  // units [c0, c1)
  int g;       // their group
  int gend;    // end of the group's units within the CTA's range
};
__device__ __forceinline__ void chunk_first(ChunkIter& it, int u0, int u1, int UG) {
  it.g = u0 / UG;
  it.gend = min(u1, (it.g + 1) * UG);
  it.c0 = u0;
  it.c1 = min(u0 + kGC, it.gend);
}
__device__ __forceinline__ void chunk_next(ChunkIter& it, int u1, int UG) {
  it.c0 = it.c1;
  if (it.c0 == it.gend) {
    ++it.g;
    it.gend = min(u1, (it.g + 1) * UG);
  }
  it.c1 = min(it.c0 + kGC, it.gend);
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
  uint64_t* rfull = empty + S;  // [2]: every consumer warp's partial of a tile piece is in red[buf]
  uint64_t* rempty = rfull + 2;  // [2]: the reducers have consumed red[buf]
  uint8_t* stages = smem + L.stages;
  uint32_t* xs = reinterpret_cast<uint32_t*>(smem + L.xs);
  float* sums = reinterpret_cast<float*>(smem + L.sums);
  float* red = reinterpret_cast<float*>(smem + L.red);
  float* lut = reinterpret_cast<float*>(smem + L.lut);
  GroupInfo* ginfo = reinterpret_cast<GroupInfo*>(smem + L.ginfo);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  for (int s = tid; s < S; s += blockDim.x) {
    mbar_init(&full[s], 1);
    mbar_init(&empty[s], kGCW);
  }
  if (tid < 2) {
    mbar_init(&rfull[tid], kGCW);
    mbar_init(&rempty[tid], kGRW);
  }
  if (tid < S + 2) fence_mbar_init();
  __syncthreads();
  // The next launch of the chain may start its prologue now; everything below reads the
  // router's (or the previous step's) outputs, so wait for the preceding kernel first.
  if (tid == 0) pdl_launch_dependents();
  pdl_wait();

  // Stage input row `row`, 64-input group sl, quarter kq into xs / sums: bf16 rows of x
  // (mode 0: tokens; mode 1 from the caller: h), or h = bf16( silu(g) * u ) from the fp32
  // gate/up rows, their first npg (gate) and npu (up) parts summed in part order -- every
  // load of a part issued before the first add.
  auto stage_item = [&](int row, int sl, int kq, int npg, int npu) {
    const int64_t k0 = (int64_t)sl * 64 + kq * 16;
    uint32_t u[8];
    if (k0 >= a.k) {
#pragma unroll
      for (int i = 0; i < 8; ++i) u[i] = 0;
    } else if (a.gu == nullptr) {
      const uint4* src = reinterpret_cast<const uint4*>(a.x + (int64_t)row * a.ldx + k0);
      const uint4 r0 = src[0], r1 = src[1];
      u[0] = r0.x; u[1] = r0.y; u[2] = r0.z; u[3] = r0.w;
      u[4] = r1.x; u[5] = r1.y; u[6] = r1.z; u[7] = r1.w;
    } else {
      const float4* gp = reinterpret_cast<const float4*>(a.gu + (int64_t)row * a.ldg + k0);
      const float4* up = reinterpret_cast<const float4*>(a.gu + (int64_t)row * a.ldg + a.k + k0);
      const int64_t ps = a.gu_pstride / 4;
      float4 g4[4], u4[4];
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        g4[q4] = __ldcg(gp + q4);
        u4[q4] = __ldcg(up + q4);
      }
      for (int pp = 1; pp < max(npg, npu); ++pp) {
        float4 gx[4], ux[4];
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          gx[q4] = pp < npg ? __ldcg(gp + pp * ps + q4) : make_float4(0.f, 0.f, 0.f, 0.f);
          ux[q4] = pp < npu ? __ldcg(up + pp * ps + q4) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          if (pp < npg) {
            g4[q4].x += gx[q4].x; g4[q4].y += gx[q4].y; g4[q4].z += gx[q4].z; g4[q4].w += gx[q4].w;
          }
          if (pp < npu) {
            u4[q4].x += ux[q4].x; u4[q4].y += ux[q4].y; u4[q4].z += ux[q4].z; u4[q4].w += ux[q4].w;
          }
        }
      }
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        u[2 * q4] = swiglu_bf16x2(g4[q4].x, u4[q4].x, g4[q4].y, u4[q4].y);
        u[2 * q4 + 1] = swiglu_bf16x2(g4[q4].z, u4[q4].z, g4[q4].w, u4[q4].w);
      }
    }
    const float4 z = stage_quarter<FMT>(u, xs + (size_t)(row * KG + sl) * 32 + kq * 8);
    reinterpret_cast<float4*>(sums)[(size_t)(row * KG + sl) * 4 + kq] = z;
  };
  // Mode 0: every token row, items it0, it0 + step, ...
  auto stage_tokens = [&](int it0, int step) {
    for (int it = it0; it < a.nrows * KG * 4; it += step) {
      const int j = it >> 2, row = j / KG;
      stage_item(row, j - row * KG, it & 3, 1, 1);
    }
  };

  // Groups: the active experts (ascending), then the shared expert as one group of all T
  // tokens.  Routing inside the launch: every CTA routes the T tokens itself (CTA 0 also
  // stores the router's outputs) while its other consumer warps stage the tokens, which do
  // not depend on the routing.
  int n_active;
  const int* groups;
  const bool routed = a.logits != nullptr;
  if (routed) {
    BlockRouteSmem& rs = *reinterpret_cast<BlockRouteSmem*>(smem + L.route);
    n_active = route_decode_block(a.logits, a.T, a.E, a.topk, rs, blockIdx.x == 0, a.ids_out, a.wts_out, a.rv,
                                  [&]() {
                                    if (warp < kGCW) stage_tokens(tid - 32 * a.T, kGCT - 32 * a.T);
                                  });
    groups = rs.groups;
  } else {  // the router's group table into shared memory, every entry it can hold at once
    BlockRouteSmem& rs = *reinterpret_cast<BlockRouteSmem*>(smem + L.route);
    const int nmax = min(a.E, a.T * a.topk);  // <= kBlockRoutePairs for 1..4 tokens
    if (tid < nmax) {
      const int4* src = reinterpret_cast<const int4*>(a.groups + (size_t)tid * kGroupInts);
      int4* dst = reinterpret_cast<int4*>(rs.groups + tid * kGroupInts);
      dst[0] = src[0];
      dst[1] = src[1];
    }
    if (tid == 0) rs.n_active = a.meta[0];
    __syncthreads();
    n_active = rs.n_active;
    groups = rs.groups;
  }

  // The unit range of this CTA: units (group, row tile, 64-input group) in that order, an
  // equal contiguous share of their cost per CTA (stream-K weighted by unit_cost: unit u
  // belongs to CTA floor(C(u) G / Ctot), C(u) the cost of the units before it).  G CTAs take
  // part, few enough that every share holds at least the costliest unit, so none is empty.
  // A row tile cut by a share boundary leaves one piece per CTA, written to output part
  // (CTA - the tile's first CTA).  Costs times G stay below 2^32 (checked on the host), so
  // this is 32-bit arithmetic.
  const int n_groups = n_active + (a.has_shared ? 1 : 0);
  const int UG = NT * KG;  // units per group
  const int wmax = unit_cost(a.T);  // no group has more than T rows
  const uint32_t Csh = (uint32_t)UG * (uint32_t)(2 * a.T * a.topk + 3 * n_active);  // the routed groups
  const uint32_t Ctot = Csh + (a.has_shared ? (uint32_t)(UG * wmax) : 0u);
  const uint32_t G = max(1u, min(gridDim.x, Ctot / (uint32_t)wmax)), b = blockIdx.x;
  if (b >= G) return;
  int u0, u1;
  {  // this warp's lanes hold the cost before groups lane, lane + 32, lane + 64 (<= 65 groups)
    uint32_t cg[3];
    int wg[3];
    bool has[3];
#pragma unroll
    for (int k = 0; k < 3; ++k) {
      const int g = lane + 32 * k;
      cg[k] = 0u;
      wg[k] = 1;
      has[k] = g < n_groups;
      if (g < n_active) {
        const int4 h = reinterpret_cast<const int4*>(groups + (size_t)g * kGroupInts)[0];
        cg[k] = (uint32_t)UG * (uint32_t)(2 * h.y + 3 * g);
        wg[k] = unit_cost(min(kGMaxRows, h.z));
      } else if (g == n_active && a.has_shared) {
        cg[k] = Csh;
        wg[k] = wmax;
      }
    }
    // first unit of share bb: the smallest u with C(u) G >= bb Ctot
    auto share_start = [&](uint32_t bb) -> int {
      if (bb >= G) return n_groups * UG;
      const uint32_t tgt = bb * Ctot;
      int n = 0;  // groups starting at or before the target (C is increasing in g)
#pragma unroll
      for (int k = 0; k < 3; ++k) n += __popc(__ballot_sync(0xFFFFFFFFu, has[k] && cg[k] * G <= tgt));
      const int gs = n - 1, ks = gs >> 5;
      const uint32_t c = __shfl_sync(0xFFFFFFFFu, ks == 0 ? cg[0] : ks == 1 ? cg[1] : cg[2], gs & 31);
      const uint32_t wG = (uint32_t)__shfl_sync(0xFFFFFFFFu, ks == 0 ? wg[0] : ks == 1 ? wg[1] : wg[2], gs & 31) * G;
      const uint32_t j = (tgt - c * G + wG - 1) / wG;
      return (int)min((uint32_t)(gs * UG) + j, (uint32_t)((gs + 1) * UG));
    };
    u0 = share_start(b);
    u1 = share_start(b + 1);
  }
  const int t0 = u0 / KG;                     // first row tile (g * NT + q) of the range
  const int npieces = (u1 - 1) / KG - t0 + 1;  // row tiles it touches
  const int g_first = u0 / UG;
  const int g_span = (u1 - 1) / UG - g_first + 1;

  if (warp == kGCW) {  // producer: the range's chunks
    if (lane == 0) {
      const uint64_t pol = l2_evict_first();  // every weight is read once per call
      int s = 0;
      uint32_t ph = 0;
      int j = 0, pg = -1;
      const uint8_t *bc = nullptr, *bs = nullptr, *ba = nullptr;
      ChunkIter it;
      for (chunk_first(it, u0, u1, UG); it.c0 < u1; chunk_next(it, u1, UG), ++j) {
        if (it.g != pg) {
          pg = it.g;
          if (it.g < n_active) {
            const int e = groups[(size_t)it.g * kGroupInts];
            bc = a.codes + (int64_t)e * a.cstride;
            bs = a.scales + (int64_t)e * a.sstride;
            ba = a.aux ? a.aux + (int64_t)e * a.astride : nullptr;
          } else {
            bc = a.sh_codes;
            bs = a.sh_scales;
            ba = a.sh_aux;
          }
        }
        if (j >= S && !mbar_wait_bounded(&empty[s], ph ^ 1u, a.status)) break;
        const int l0 = it.c0 - it.g * UG;  // unit index within the group
        const int nu = it.c1 - it.c0;
        uint8_t* dst = stages + (size_t)s * SBY;
        uint32_t bytes = (uint32_t)nu * (SG::CODE + SG::SCALE);
        int aux_a = 0, aux_n = 0;
        if (SG::AUX) {
          aux_a = l0 >> 2;
          aux_n = ((l0 + nu - 1) >> 2) - aux_a + 1;
          bytes += (uint32_t)aux_n * SG::AUX;
        }
        mbar_arrive_expect_tx(&full[s], bytes);
        bulk_g2s_hint(dst, bc + (size_t)l0 * SG::CODE, (uint32_t)nu * SG::CODE, &full[s], pol);
        bulk_g2s_hint(dst + kGC * SG::CODE, bs + (size_t)l0 * SG::SCALE, (uint32_t)nu * SG::SCALE, &full[s], pol);
        if (SG::AUX)
          bulk_g2s_hint(dst + kGC * (SG::CODE + SG::SCALE), ba + (size_t)aux_a * SG::AUX,
                        (uint32_t)aux_n * SG::AUX, &full[s], pol);
        if (++s == S) {
          s = 0;
          ph ^= 1u;
        }
      }
    }
    return;
  }

  // The groups this CTA touches: their descriptors are read once here.
  if (tid < kGInfoCache && tid < g_span) ginfo[tid] = group_info(a, groups, g_first + tid, n_active, UG);
  // Down launch: how many parts each gate/up row tile of those groups was written in -- the
  // gate/up launch's weighted split over the same groups (same routing, same grid), redone.
  uint8_t* gpc = smem + L.gpc;
  const bool use_gpc = a.mode == 1 && a.gu != nullptr && g_span <= kGInfoCache && a.gu_nt <= kGPcTiles;
  for (int i = tid; use_gpc && tid < kGCT && i < g_span * a.gu_nt; i += kGCT) {  // consumer threads
    const int gs = i / a.gu_nt, tg = i - gs * a.gu_nt;
    const GroupInfo gg = group_info(a, groups, g_first + gs, n_active, 1);
    const uint32_t ug = (uint32_t)(a.gu_nt * a.gu_kg);
    const uint32_t ctot = ug * (uint32_t)(2 * a.T * a.topk + 3 * n_active + (a.has_shared ? wmax : 0));
    const uint32_t gn = max(1u, min(gridDim.x, ctot / (uint32_t)wmax));
    const uint32_t ct = ug * (uint32_t)gg.cu + (uint32_t)(tg * a.gu_kg * gg.w);
    const uint32_t f = ct * gn / ctot, l = (ct + (uint32_t)((a.gu_kg - 1) * gg.w)) * gn / ctot;
    gpc[gs * kGPcTiles + tg] = (uint8_t)min((uint32_t)a.gu_parts, l - f + 1u);
  }

  if (warp > kGCW) {  // reducers: each tile piece's 12 warp partials, summed in warp order
    const int rl = (warp - kGCW - 1) * 32 + lane;  // float4 column of the piece's rows
    __syncwarp();
    named_sync(2, kGCT + 32 * kGRW);  // descriptors ready
    bool ok = true;
    for (int i = 0; i < npieces; ++i) {
      const int buf = i & 1;
      if (ok && !mbar_try_wait(&rfull[buf], (uint32_t)(i >> 1) & 1u) &&
          !mbar_wait_bounded(&rfull[buf], (uint32_t)(i >> 1) & 1u, a.status))
        ok = false;
      if (ok) {
        const int tile = t0 + i, g = tile / NT, q = tile - g * NT;
        const GroupInfo gi = (g - g_first < kGInfoCache) ? ginfo[g - g_first] : group_info(a, groups, g, n_active, UG);
        const uint32_t ct = gi.cbase + (uint32_t)((tile - g * NT) * KG * gi.w);  // cost before the tile
        const int part = (int)(b - ct * G / Ctot);
        const bool last = (ct + (uint32_t)((KG - 1) * gi.w)) * G / Ctot == b;
        const int pend = last ? a.P : part + 1;  // the tile's last piece zeroes the parts after it
        if (part >= a.P && lane == 0) atomicExch(a.status, kStatusUnsupported);  // more pieces than parts
        const float4* rb = reinterpret_cast<const float4*>(red + (size_t)buf * kGCW * kGMaxRows * 128);
        for (int e4 = rl; part < a.P && e4 < gi.m * 32; e4 += 32 * kGRW) {
          float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
          for (int w2 = 0; w2 < kGCW; ++w2) {
            const float4 x = rb[w2 * kGMaxRows * 32 + e4];
            v.x += x.x;
            v.y += x.y;
            v.z += x.z;
            v.w += x.w;
          }
          v = make_float4(v.x * gi.ts, v.y * gi.ts, v.z * gi.ts, v.w * gi.ts);
          const int64_t n = (int64_t)q * 128 + (e4 & 31) * 4;
          float* o = a.out + (int64_t)gi.out_row[e4 >> 5] * a.ldo + n;
          for (int p = part; p < pend; ++p) {
            const float4 x = p == part ? v : make_float4(0.f, 0.f, 0.f, 0.f);
            float* op = o + (int64_t)p * a.out_pstride;
            if (n + 3 < a.n) {
              *reinterpret_cast<float4*>(op) = x;
            } else {
              if (n < a.n) op[0] = x.x;
              if (n + 1 < a.n) op[1] = x.y;
              if (n + 2 < a.n) op[2] = x.z;
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&rempty[buf]);  // also on failure, so no consumer waits forever
    }
    return;
  }

  if (FMT == FMT_NVFP4 && tid < 128) {
    const float2 v = e4m3x2_f32<0>((uint32_t)(2 * tid) | ((uint32_t)(2 * tid + 1) << 8));
    lut[2 * tid] = v.x;
    lut[2 * tid + 1] = v.y;
  }
  named_sync(2, kGCT + 32 * kGRW);  // descriptors ready (consumers and reducers)
  // Stage the input rows over all of K (mode 0 routed here: staged during the routing).
  // Mode 1: the rows of the groups this CTA touches (all rows if it touches more than
  // kGInfoCache groups).
  if (a.mode == 0) {
    if (!routed) stage_tokens(tid, kGCT);
  } else if (g_span <= kGInfoCache && a.gu != nullptr) {
    // h = bf16( silu(g) * u ) of the groups' rows, four features a thread item (every thread
    // busy however few rows), written as bf16 into the rows' staging slots; then each
    // 16-input quarter is staged in place.
    int nsr = 0;  // staged rows: the rows of the CTA's groups, in group order
    for (int gs = 0; gs < g_span; ++gs) nsr += ginfo[gs].m;
    auto row_of = [&](int r, int& gs) {
      gs = 0;
      while (r >= ginfo[gs].m) r -= ginfo[gs++].m;
      return ginfo[gs].in_row[r];
    };
    const int F4 = KG * 16;  // float4 columns of a row padded to whole 64-input groups
    const int64_t ps = a.gu_pstride / 4;
    for (int it = tid; it < nsr * F4; it += kGCT) {
      const int r = it / F4, c4 = it - r * F4, f = 4 * c4;
      int gs;
      const int row = row_of(r, gs);
      uint2 hv = make_uint2(0u, 0u);
      if (f < a.k) {
        int npg = a.gu_parts, npu = a.gu_parts;
        if (use_gpc) {
          npg = gpc[gs * kGPcTiles + f / 128];
          npu = gpc[gs * kGPcTiles + (int)((a.k + f) / 128)];
        }
        const float4* gp = reinterpret_cast<const float4*>(a.gu + (int64_t)row * a.ldg + f);
        const float4* up = reinterpret_cast<const float4*>(a.gu + (int64_t)row * a.ldg + a.k + f);
        float4 g4 = __ldcg(gp), u4 = __ldcg(up);
        float4 g1 = make_float4(0.f, 0.f, 0.f, 0.f), u1 = g1;
        if (npg > 1) g1 = __ldcg(gp + ps);
        if (npu > 1) u1 = __ldcg(up + ps);
        if (npg > 1) { g4.x += g1.x; g4.y += g1.y; g4.z += g1.z; g4.w += g1.w; }
        if (npu > 1) { u4.x += u1.x; u4.y += u1.y; u4.z += u1.z; u4.w += u1.w; }
        for (int pp = 2; pp < max(npg, npu); ++pp) {  // more parts (few tiles, or one token)
          if (pp < npg) {
            const float4 x = __ldcg(gp + pp * ps);
            g4.x += x.x; g4.y += x.y; g4.z += x.z; g4.w += x.w;
          }
          if (pp < npu) {
            const float4 x = __ldcg(up + pp * ps);
            u4.x += x.x; u4.y += x.y; u4.z += x.z; u4.w += x.w;
          }
        }
        hv = make_uint2(swiglu_bf16x2(g4.x, u4.x, g4.y, u4.y), swiglu_bf16x2(g4.z, u4.z, g4.w, u4.w));
      }
      *reinterpret_cast<uint2*>(xs + (size_t)(row * KG + (f >> 6)) * 32 + ((f & 63) >> 1)) = hv;
    }
    named_sync(1, kGCT);
    for (int it = tid; it < nsr * KG * 4; it += kGCT) {
      const int r = it / (KG * 4), rem = it - r * (KG * 4);
      int gs;
      const int row = row_of(r, gs), sl = rem >> 2, kq = rem & 3;
      uint32_t* dst = xs + (size_t)(row * KG + sl) * 32 + kq * 8;
      const uint4 v0 = reinterpret_cast<const uint4*>(dst)[0], v1 = reinterpret_cast<const uint4*>(dst)[1];
      const uint32_t u[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
      const float4 z = stage_quarter<FMT>(u, dst);
      reinterpret_cast<float4*>(sums)[(size_t)(row * KG + sl) * 4 + kq] = z;
    }
  } else if (g_span <= kGInfoCache) {
    for (int it = tid; it < g_span * kGMaxRows * KG * 4; it += kGCT) {
      const int kq = it & 3, sl = (it >> 2) % KG, slot = (it >> 2) / KG;
      const GroupInfo& gs = ginfo[slot / kGMaxRows];
      if (slot % kGMaxRows >= gs.m) continue;
      int npg = a.gu_parts, npu = a.gu_parts;
      if (use_gpc) {
        const int k0 = sl * 64 + kq * 16;
        const uint8_t* pc = gpc + (slot / kGMaxRows) * kGPcTiles;
        npg = k0 < a.k ? pc[k0 / 128] : 1;
        npu = k0 < a.k ? pc[(a.k + k0) / 128] : 1;
      }
      stage_item(gs.in_row[slot % kGMaxRows], sl, kq, npg, npu);
    }
  } else {
    for (int it = tid; it < a.nrows * KG * 4; it += kGCT) {
      const int j = it >> 2, row = j / KG;
      stage_item(row, j - row * KG, it & 3, a.gu_parts, a.gu_parts);
    }
  }
  named_sync(1, kGCT);

  // Warp w takes unit w / 2 of every chunk, quarters 2 (w % 2) and 2 (w % 2) + 1 of it,
  // accumulating one tile piece at a time; a piece's partial goes to the reducer once the
  // warp's chunks have moved past it (zeros for a piece it had no unit of).
  const int ug = warp >> 1, kh = warp & 1;
  bool ok = true;
  int s = 0;
  uint32_t ph = 0;
  int cur = 0;  // the piece being accumulated
  float acc[4][kGMaxRows];
#pragma unroll
  for (int rt = 0; rt < 4; ++rt)
#pragma unroll
    for (int m = 0; m < kGMaxRows; ++m) acc[rt][m] = 0.0f;
  auto flush = [&](int i) {
    const int buf = i & 1;
    if (i >= 2 && ok && !mbar_wait_bounded(&rempty[buf], (uint32_t)((i >> 1) - 1) & 1u, a.status)) ok = false;
    float* rb = red + ((size_t)buf * kGCW + warp) * kGMaxRows * 128;
#pragma unroll
    for (int rt = 0; rt < 4; ++rt)
#pragma unroll
      for (int m = 0; m < kGMaxRows; ++m) {
        if (ok) rb[m * 128 + rt * 32 + lane] = acc[rt][m];  // after a timed-out wait: leave it
        acc[rt][m] = 0.0f;
      }
    __syncwarp();
    if (lane == 0) mbar_arrive(&rfull[buf]);
  };
  // One loop per run of chunks of a group, compiled for the group's row count: the loop the
  // warps spin in holds one consume variant, so it stays in the instruction cache.
  ChunkIter it;
  chunk_first(it, u0, u1, UG);
  while (it.c0 < u1) {
    const int g = it.g;
    const GroupInfo gi = (g - g_first < kGInfoCache) ? ginfo[g - g_first] : group_info(a, groups, g, n_active, UG);
    auto run = [&](auto rows) {
      constexpr int M = decltype(rows)::value;
      for (; it.c0 < u1 && it.g == g; chunk_next(it, u1, UG)) {
        // Hand over every piece before this warp's unit (or before the chunk, without one)
        // before waiting for the chunk: a warp with no unit for a while must not hold back
        // the reducers, which the other warps wait for.
        const int uw = it.c0 + ug;
        const int tile = (uw < it.c1 ? uw : it.c0) / KG;
        while (cur < tile - t0) flush(cur++);
        if (ok && !mbar_try_wait(&full[s], ph) && !mbar_wait_bounded(&full[s], ph, a.status)) ok = false;
        if (ok && uw < it.c1) {
          const int l = uw - g * UG, l0 = it.c0 - g * UG;  // units within the group
          const int kg = uw - tile * KG;
          const uint8_t* st = stages + (size_t)s * SBY;
          const uint8_t* cst = st + ug * SG::CODE;
          const uint8_t* sst = st + kGC * SG::CODE + ug * SG::SCALE;
          const uint8_t* aux = st + kGC * (SG::CODE + SG::SCALE) + ((l >> 2) - (l0 >> 2)) * SG::AUX;
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int kq = 2 * kh + h;
            const uint32_t* xr[kGMaxRows];
            const float* zr[kGMaxRows];
#pragma unroll
            for (int m = 0; m < kGMaxRows; ++m) {
              const int r = gi.in_row[m < M ? m : 0];
              xr[m] = xs + (size_t)(r * KG + kg) * 32 + kq * 8;
              zr[m] = sums + ((size_t)(r * KG + kg) * 4 + kq) * 4;
            }
            consume<FMT, M, kGMaxRows>(cst, sst, aux, xr, zr, lut, kq, lane, acc);
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
        if (++s == S) {
          s = 0;
          ph ^= 1u;
        }
      }
    };
    switch (gi.m) {
      case 1: run(std::integral_constant<int, 1>{}); break;
      case 2: run(std::integral_constant<int, 2>{}); break;
      case 3: run(std::integral_constant<int, 3>{}); break;
      default: run(std::integral_constant<int, 4>{}); break;
    }
  }
  while (cur < npieces) flush(cur++);
  // the reducer still reads red: it returns on its own; nothing here waits for it
}

// h[r][f] = bf16( silu(gu[r][f]) * gu[r][F + f] ) for every row (the staged gate/up call
// writes h for the caller; the fused chain computes it inside the down GEMV instead).
__global__ void __launch_bounds__(256) mid_kernel(const float* gu, int64_t ldg, int parts, int64_t pstride,
                                                  __nv_bfloat16* h, int64_t ldh, int F, int rows) {
  pdl_launch_dependents();
  pdl_wait();
  const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= (int64_t)rows * (F / 2)) return;
  const int r = (int)(idx / (F / 2)), f = (int)(idx % (F / 2)) * 2;
  float2 g = *reinterpret_cast<const float2*>(gu + r * ldg + f);
  float2 u = *reinterpret_cast<const float2*>(gu + r * ldg + F + f);
  for (int p = 1; p < parts; ++p) {  // the gate/up GEMV's input parts, summed in order
    const float2 gp = *reinterpret_cast<const float2*>(gu + p * pstride + r * ldg + f);
    const float2 up = *reinterpret_cast<const float2*>(gu + p * pstride + r * ldg + F + f);
    g.x += gp.x;
    g.y += gp.y;
    u.x += up.x;
    u.y += up.y;
  }
  *reinterpret_cast<uint32_t*>(h + r * ldh + f) = swiglu_bf16x2(g.x, u.x, g.y, u.y);
}

// out[t][n] = bf16( sum_j w[t][j] * d[pos(t, j)][n] + g_t * d[T*topk + t][n] ), fixed order,
// four features per thread (g_t: the shared expert's sigmoid gate, or 1); every load of a
// thread is issued before the first multiply-add.
__global__ void __launch_bounds__(256) finish_kernel(const float* d, int64_t ldd, int parts, int64_t pstride,
                                                     const float* w, const int* pair_pos,
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
  float4 sh = has_shared ? __ldcg(reinterpret_cast<const float4*>(d + (int64_t)(T * topk + t) * ldd + n))
                         : make_float4(0, 0, 0, 0);
  for (int p = 1; p < parts; ++p) {  // the down GEMV's input parts, summed in order
    const float* dp = d + p * pstride;
#pragma unroll
    for (int j = 0; j < kMaxTopk; ++j) {
      if (j < topk) {
        const float4 x = __ldcg(reinterpret_cast<const float4*>(dp + (int64_t)pos[j] * ldd + n));
        v[j].x += x.x;
        v[j].y += x.y;
        v[j].z += x.z;
        v[j].w += x.w;
      }
    }
    if (has_shared) {
      const float4 x = __ldcg(reinterpret_cast<const float4*>(dp + (int64_t)(T * topk + t) * ldd + n));
      sh.x += x.x;
      sh.y += x.y;
      sh.z += x.z;
      sh.w += x.w;
    }
  }
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

// Output parts of a decode GEMV: the most CTA shares one row tile of kg units can meet.  A
// share spans at least Ctot / grid of cost, a tile at most kg * unit_cost(T); the least total
// cost the routing can produce is that of topk groups (a token's experts are distinct) holding
// all T * topk rows: nt * kg * (2 T topk + 3 topk).
static int grouped_parts(int64_t T, int64_t topk, int64_t nt, int64_t kg, int grid) {
  const int64_t cmin = nt * kg * (2 * T * topk + 3 * topk);
  const int64_t span = kg * unit_cost((int)T) * grid;  // tile cost x grid
  return (int)std::min<int64_t>(kg, (span + cmin - 1) / cmin + 1);
}

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
  // needs no fp32 gate/up rows; its down outputs are one part, in bf16
  const bool decode = T <= kGMaxRows;
  L.p_gu = decode ? grouped_parts(T, topk, gu.nt, gu.kg, grid) : 1;
  L.p_dn = decode ? grouped_parts(T, topk, dn.nt, dn.kg, grid) : 1;
  L.ld_gu = (gu.n + 7) / 8 * 8;
  L.pst_gu = R * L.ld_gu;
  L.gu = take(decode ? (size_t)L.p_gu * R * L.ld_gu * 4 : 0);
  L.ld_h = (dn.k + 7) / 8 * 8;
  L.h = take(decode ? 0 : (size_t)R * L.ld_h * 2);  // decode: h never leaves the down GEMV
  L.ld_d = (dn.n + 7) / 8 * 8;
  L.pst_dn = R * L.ld_d;
  L.d = take((size_t)L.p_dn * R * L.ld_d * (decode ? 4 : 2));
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
  static std::atomic<unsigned long long> configured[8];
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
                      void* out, int64_t ldo, void* ws, const DeviceInfo& dev, void* stream, int stage,
                      const float* logits, int32_t* topk_ids_out, float* topk_w_out) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // the grouped GEMV splits work by cost in 32-bit arithmetic: (cost of every unit) x CTAs
  const int64_t cu_max = 2 * T * topk + 3 * std::min<int64_t>(m->n_experts, T * topk) + unit_cost((int)T) + 1;
  for (const Geometry* g : {&gu, &dn})
    if (g->nt * g->kg * cu_max * dev.sms >= ((int64_t)1 << 32)) return QG_ERR_UNSUPPORTED;
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
  a.E = m->n_experts;
  a.mode = 0;
  a.x = static_cast<const __nv_bfloat16*>(x);
  a.ldx = ldx;
  a.out = reinterpret_cast<float*>(w + L.gu);
  a.ldo = L.ld_gu;
  a.P = L.p_gu;
  a.out_pstride = L.pst_gu;
  a.meta = rv.meta;
  a.groups = rv.groups;
  if (logits) {  // the gate/up launch routes the tokens and stores the router's outputs
    a.logits = logits;
    a.E = m->n_experts;
    a.ids_out = topk_ids_out;
    a.wts_out = topk_w_out;
    a.rv = rv;
    topk_w = topk_w_out;
  }
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
                   (const float*)reinterpret_cast<const float*>(w + L.gu), (int64_t)L.ld_gu, L.p_gu, L.pst_gu,
                   static_cast<__nv_bfloat16*>(out), ldo, F, rows) != cudaSuccess)
      return QG_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? QG_OK : QG_ERR_CUDA;
  }

  qg_packed_sizes(m->fmt, dn.n, dn.k, &cb, &sb, &ab);
  GroupedArgs d = a;
  d.logits = nullptr;  // the down launch reads the routing the gate/up launch stored
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
    d.gu_parts = L.p_gu;
    d.gu_pstride = L.pst_gu;
    d.gu_nt = (int)gu.nt;
    d.gu_kg = (int)gu.kg;
  }
  d.out = reinterpret_cast<float*>(w + L.d);
  d.ldo = L.ld_d;
  d.P = L.p_dn;
  d.out_pstride = L.pst_dn;
  st = launch_grouped(m->fmt, d, rows, (int)dn.kg, dev, s);
  if (st != QG_OK) return st;

  if (launch_pdl(finish_kernel, dim3((unsigned)((T * (dn.n / 4) + 255) / 256)), dim3(256), 0, s,
                 (const float*)reinterpret_cast<const float*>(w + L.d), (int64_t)L.ld_d, L.p_dn, L.pst_dn, topk_w,
                 (const int*)rv.pair_pos, (int)T, topk, (int)m->has_shared, shared_gate, (int64_t)dn.n,
                 static_cast<__nv_bfloat16*>(out), ldo) != cudaSuccess)
    return QG_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? QG_OK : QG_ERR_CUDA;
}

}  // namespace qg
