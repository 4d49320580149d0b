// Mixture-of-experts layer for 1..4 tokens (decode and speculative verify), in the five
// dependent launches of the TurboEXL3 article §4.2: route (route.cu), gate/up, mid, down,
// finish.  The shared expert runs as extra groups of the routed gate/up and down launches
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
// The grouped GEMV runs the dense GEMV's decode (qg_gemv_core.cuh) over segments (group,
// 128-row tile, 1/P of the inputs) with groups = active experts (ascending) then the shared
// expert once per token; each CTA takes an equal share of whole segments, its 12 consumer
// warps hand each segment's partials to a reducer warp (two buffers, so they run on), and
// the P parts of an output are summed by whoever reads it next, in part order.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>

#include "qg_common.cuh"
#include "qg_gemv_core.cuh"
#include "qg_internal.h"
#include "qg_route.h"
#include "qg_route_dev.cuh"
#include "qg_sync.cuh"

namespace qg {

constexpr int kGCW = 12;              // consumer warps (3 units per chunk, 128 registers a thread: no spills)
constexpr int kGCT = kGCW * 32;
constexpr int kGC = kGCW / 4;         // units per chunk
constexpr int kGThreads = kGCT + 64;  // + the producer warp and the reducer warp
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
  int P;  // input parts: a segment is (group, 128-row tile, 1/P of the inputs)
  int T, topk;
  int mode;  // 0: input rows are tokens (x); 1: input rows are grouped pairs, shared rows
             // after: bf16 rows of x, or (gu non-null) the SwiGLU of the fp32 gate/up rows gu
  const __nv_bfloat16* x;
  int64_t ldx;
  const float* gu;      // gu_parts partial sums of the gate/up rows, gu_pstride floats apart
  int64_t ldg;
  int gu_parts;
  int64_t gu_pstride;
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
};
constexpr int kGInfoCache = 8;

struct GroupedSmem {
  size_t bars, stages, xs, sums, red, lut, misc, ginfo, route, total;
};

// Shared memory: mbarriers (full[S], empty[S], rfull[2], rempty[2]), the stage ring, the
// staged activations, two reduction buffers (one per segment in flight), the E4M3 table
// and the descriptors of the first groups the CTA touches.
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
  o = (o + 15) & ~(size_t)15;
  L.route = o;  // routing scratch and group table when the launch routes its tokens
  o += sizeof(BlockRouteSmem);
  L.total = o;
  return L;
}

__device__ __forceinline__ GroupInfo group_info(const GroupedArgs& a, const int* groups, int g, int n_active) {
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
  const int S = a.stages, KG = a.KG, NT = a.NT, P = a.P;
  const int SBY = SG::bytes(kGC);
  const GroupedSmem L = grouped_smem(SBY, S, a.nrows, KG);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bars);
  uint64_t* empty = full + S;
  uint64_t* rfull = empty + S;  // [2]: a segment's 12 partials are in red[buf]
  uint64_t* rempty = rfull + 2;  // [2]: the reducer has consumed red[buf]
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
    mbar_init(&rempty[tid], 1);
  }
  if (tid < S + 2) fence_mbar_init();
  __syncthreads();
  // The next launch of the chain may start its prologue now; everything below reads the
  // router's (or the previous step's) outputs, so wait for the preceding kernel first.
  if (tid == 0) pdl_launch_dependents();
  pdl_wait();

  // Segments: (group, row tile q, input part p), p-major inside a row tile; groups are the
  // active experts, then the shared expert once per token.  Each CTA takes a contiguous,
  // equal share of whole segments: no row tile is split across CTAs, so there are no
  // tickets or partials to combine here -- the P parts are summed by the consumer of the
  // outputs (the down GEMV's staging, the mid, the finish), in part order.
  int n_active;
  const int* groups;
  if (a.logits) {  // route the T tokens here (every CTA the same table; CTA 0 stores it)
    BlockRouteSmem& rs = *reinterpret_cast<BlockRouteSmem*>(smem + L.route);
    n_active = route_decode_block(a.logits, a.T, a.E, a.topk, rs, blockIdx.x == 0, a.ids_out, a.wts_out, a.rv);
    groups = rs.groups;
  } else {
    n_active = a.meta[0];
    groups = a.groups;
  }
  const int n_groups = n_active + (a.has_shared ? a.T : 0);
  const int spg = NT * P;
  const int64_t n_seg = (int64_t)n_groups * spg;
  const int64_t G = min((int64_t)gridDim.x, n_seg), b = blockIdx.x;
  if (b >= G) return;
  const int sg0 = (int)(b * n_seg / G), sg1 = (int)((b + 1) * n_seg / G);
  const int nck = (KG + kGC - 1) / kGC;  // chunks per row tile; part p takes chunks [p*nck/P, (p+1)*nck/P)
  auto seg_units = [&](int sg, int& g, int& q, int& p, int& k0, int& k1) {
    g = sg / spg;
    const int r = sg - g * spg;
    q = r / P;
    p = r - q * P;
    k0 = kGC * (p * nck / P);
    k1 = min(KG, kGC * ((p + 1) * nck / P));
  };

  if (warp == kGCW) {  // producer: the segments' units, chunks never span two segments
    if (lane == 0) {
      int s = 0, j = 0;
      uint32_t ph = 0;
      bool ok = true;
      for (int sg = sg0; ok && sg < sg1; ++sg) {
        int g, q, p, k0, k1;
        seg_units(sg, g, q, p, k0, k1);
        const uint8_t *bc, *bs, *ba;
        if (g < n_active) {
          const int e = groups[(size_t)g * kGroupInts];
          bc = a.codes + (int64_t)e * a.cstride;
          bs = a.scales + (int64_t)e * a.sstride;
          ba = a.aux ? a.aux + (int64_t)e * a.astride : nullptr;
        } else {
          bc = a.sh_codes;
          bs = a.sh_scales;
          ba = a.sh_aux;
        }
        for (int kc = k0; kc < k1; kc += kGC, ++j) {
          if (j >= S && !mbar_wait_bounded(&empty[s], ph ^ 1u, a.status)) {
            ok = false;
            break;
          }
          const int l0 = q * KG + kc;  // unit index within the group
          const int nu = min(kGC, k1 - kc);
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
    }
    return;
  }

  // The groups this CTA touches: their descriptors are read once here.
  const int g_first = sg0 / spg;
  const int g_span = (sg1 - 1) / spg - g_first + 1;
  if (tid < kGInfoCache && g_first + tid < n_groups) ginfo[tid] = group_info(a, groups, g_first + tid, n_active);

  if (warp == kGCW + 1) {  // reducer: each segment's 12 warp partials, summed in warp order
    __syncwarp();
    named_sync(2, kGCT + 32);  // descriptors ready
    bool ok = true;
    for (int sg = sg0; sg < sg1; ++sg) {
      const int i = sg - sg0, buf = i & 1;
      if (ok && !mbar_wait_bounded(&rfull[buf], (uint32_t)(i >> 1) & 1u, a.status)) ok = false;
      if (ok) {
        int g, q, p, k0, k1;
        seg_units(sg, g, q, p, k0, k1);
        const GroupInfo gi = (g - g_first < kGInfoCache) ? ginfo[g - g_first] : group_info(a, groups, g, n_active);
        const float* rb = red + (size_t)buf * kGCW * kGMaxRows * 128;
        float* outp = a.out + (int64_t)p * a.out_pstride;
        for (int e = lane; e < gi.m * 128; e += 32) {
          float v = 0.0f;
#pragma unroll
          for (int w2 = 0; w2 < kGCW; ++w2) v += rb[w2 * kGMaxRows * 128 + e];
          const int64_t n = (int64_t)q * 128 + (e & 127);
          if (n < a.n) outp[(int64_t)gi.out_row[e >> 7] * a.ldo + n] = v * gi.ts;
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
  named_sync(2, kGCT + 32);  // descriptors ready (consumers and reducer)
  // Stage the input rows over all of K.  Mode 0: every token row of x.  Mode 1: the rows of
  // the groups this CTA touches (all rows if it touches more than kGInfoCache groups), each
  // computed as h = bf16( silu(g) * u ) from the fp32 gate/up outputs (their parts summed).
  const bool by_group = a.mode == 1 && g_span <= kGInfoCache;
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
      const float* gp = a.gu + (int64_t)row * a.ldg + k0;
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        float4 g4 = __ldcg(reinterpret_cast<const float4*>(gp) + q4);
        float4 u4 = __ldcg(reinterpret_cast<const float4*>(gp + a.k) + q4);
        for (int pp = 1; pp < a.gu_parts; ++pp) {
          const float4 gx = __ldcg(reinterpret_cast<const float4*>(gp + pp * a.gu_pstride) + q4);
          const float4 ux = __ldcg(reinterpret_cast<const float4*>(gp + pp * a.gu_pstride + a.k) + q4);
          g4.x += gx.x; g4.y += gx.y; g4.z += gx.z; g4.w += gx.w;
          u4.x += ux.x; u4.y += ux.y; u4.z += ux.z; u4.w += ux.w;
        }
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
  int s = 0;
  uint32_t ph = 0;
  for (int sg = sg0; sg < sg1; ++sg) {
    int g, q, p, k0, k1;
    seg_units(sg, g, q, p, k0, k1);
    const GroupInfo gi = (g - g_first < kGInfoCache) ? ginfo[g - g_first] : group_info(a, groups, g, n_active);
    float acc[4][kGMaxRows];
#pragma unroll
    for (int rt = 0; rt < 4; ++rt)
#pragma unroll
      for (int m = 0; m < kGMaxRows; ++m) acc[rt][m] = 0.0f;
    const uint32_t* xr[kGMaxRows];
    const float* zr[kGMaxRows];
    for (int kc = k0; kc < k1; kc += kGC) {
      if (ok && !mbar_wait_bounded(&full[s], ph, a.status)) ok = false;
      const int kg = kc + ug;
      if (ok && kg < k1) {
        const int ul = q * KG + kg;  // unit within the group
        const uint8_t* st = stages + (size_t)s * SBY;
        const int l0 = q * KG + kc;  // first unit of this chunk
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
    // Hand the warp's partial to the reducer (two buffers: the warps run on into the next
    // segment while the reducer sums this one).
    const int i = sg - sg0, buf = i & 1;
    if (i >= 2 && ok && !mbar_wait_bounded(&rempty[buf], (uint32_t)((i >> 1) - 1) & 1u, a.status)) ok = false;
    float* rb = red + ((size_t)buf * kGCW + warp) * kGMaxRows * 128;
    if (ok) {  // after a timed-out wait the reducer may still read this buffer: leave it
#pragma unroll
      for (int rt = 0; rt < 4; ++rt)
#pragma unroll
        for (int m = 0; m < kGMaxRows; ++m) rb[m * 128 + rt * 32 + lane] = acc[rt][m];
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&rfull[buf]);
  }
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

// Input parts of a decode GEMV: the fewest that give every CTA about four whole segments
// (group, row tile, part) at the most groups the routing can produce, so equal shares of
// whole segments stay balanced; parts are whole chunks of kGC units, so at most one part
// per row tile -- the last -- leaves warps idle in its last chunk.
static int grouped_parts(int64_t max_groups, int64_t nt, int64_t kg, int sms) {
  const int64_t nck = (kg + kGC - 1) / kGC;
  int64_t p = (4 * (int64_t)sms + max_groups * nt - 1) / (max_groups * nt);
  return (int)std::max<int64_t>(1, std::min<int64_t>(p, nck));
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
  // needs no fp32 gate/up rows; its down outputs are one part
  const bool decode = T <= kGMaxRows;
  const int64_t max_groups = std::min<int64_t>(E, T * topk) + T;
  L.p_gu = decode ? grouped_parts(max_groups, gu.nt, gu.kg, grid) : 1;
  L.p_dn = decode ? grouped_parts(max_groups, dn.nt, dn.kg, grid) : 1;
  L.ld_gu = (gu.n + 7) / 8 * 8;
  L.pst_gu = R * L.ld_gu;
  L.gu = take(decode ? (size_t)L.p_gu * R * L.ld_gu * 4 : 0);
  L.ld_h = (dn.k + 7) / 8 * 8;
  L.h = take(decode ? 0 : (size_t)R * L.ld_h * 2);  // decode: h never leaves the down GEMV
  L.ld_d = (dn.n + 7) / 8 * 8;
  L.pst_dn = R * L.ld_d;
  L.d = take((size_t)L.p_dn * R * L.ld_d * 4);
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
