// Mixture-of-experts router (TurboEXL3 article §4.1 "Route": count each expert's tokens,
// group the tokens by expert, build the table of tiles -- one pass instead of a sort;
// §4.2: the router's top-k and softmax).
//
// Per token: the top-k experts by fp32 logit (ties to the lower expert index) and the
// softmax of the k kept logits.  Then every (token, slot) pair p = t*k + j is placed in
// grouped order -- experts ascending, tokens ascending within an expert -- giving
// counts[e], offsets[e] (exclusive prefix), pair_list[pos] = p, pair_pos[p] = pos, the
// ascending list of active experts, and a tile table of (expert, first position, count)
// with at most kRouteTile pairs per tile for the grouped prefill GEMM.  Everything is
// deterministic: ranks come from ordered scans, never from atomic arrival order.
#include <cuda_runtime.h>

#include "qg_internal.h"
#include "qg_route.h"
#include "qg_route_dev.cuh"
#include "qg_sync.cuh"

namespace qg {

constexpr int kRouteBlock = 1024;  // pairs per grouping block (one thread per pair)

__global__ void __launch_bounds__(256) route_topk_kernel(const float* logits, int64_t T, int E, int k, int32_t* ids,
                                                         float* wts) {
  const int64_t t = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (t >= T) return;
  warp_topk(logits + t * E, E, k, ids + t * k, wts + t * k);
}

// Clear a shared array with 16-byte stores (bytes a multiple of 16, 16-byte aligned).
__device__ __forceinline__ void zero_shared(void* p, int bytes) {
  uint4* q = static_cast<uint4*>(p);
  for (int i = threadIdx.x; i < bytes / 16; i += blockDim.x) q[i] = make_uint4(0, 0, 0, 0);
}

// Per-block histogram of the experts of pairs [b*kRouteBlock, ...).
__device__ void block_count(const int32_t* ids, int64_t P, int E, int b, int* out) {
  __shared__ int hist[kMaxExperts];
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
  __syncthreads();
  const int64_t p = (int64_t)b * kRouteBlock + threadIdx.x;
  if (threadIdx.x < kRouteBlock && p < P) atomicAdd(&hist[ids[p]], 1);  // integer counts: order-free
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) out[e] = hist[e];
  __syncthreads();
}

// Block-wide exclusive scan of three counters (every thread of the block calls it;
// blockDim.x a multiple of 32, <= 1024); the totals go to *tot (shared memory).
__device__ __forceinline__ int3 block_scan3(int3 x, int3* tot) {
  __shared__ int3 wsum[32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int3 inc = x;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int a = __shfl_up_sync(0xFFFFFFFFu, inc.x, off), b = __shfl_up_sync(0xFFFFFFFFu, inc.y, off),
              c = __shfl_up_sync(0xFFFFFFFFu, inc.z, off);
    if (lane >= off) {
      inc.x += a;
      inc.y += b;
      inc.z += c;
    }
  }
  if (lane == 31) wsum[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    const int3 w = lane < nw ? wsum[lane] : make_int3(0, 0, 0);
    int3 wi = w;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int a = __shfl_up_sync(0xFFFFFFFFu, wi.x, off), b = __shfl_up_sync(0xFFFFFFFFu, wi.y, off),
                c = __shfl_up_sync(0xFFFFFFFFu, wi.z, off);
      if (lane >= off) {
        wi.x += a;
        wi.y += b;
        wi.z += c;
      }
    }
    if (lane < nw) wsum[lane] = make_int3(wi.x - w.x, wi.y - w.y, wi.z - w.z);  // exclusive, per warp
    if (lane == 31) *tot = wi;
  }
  __syncthreads();
  const int3 base = wsum[warp];
  __syncthreads();
  return make_int3(base.x + inc.x - x.x, base.y + inc.y - x.y, base.z + inc.z - x.z);
}

// Sum of n counters strided by E (per-block expert counts), loads batched for overlap.
__device__ __forceinline__ int strided_sum(const int* p, int E, int n) {
  int s = 0, b = 0;
  for (; b + 8 <= n; b += 8) {
    int t[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) t[i] = p[(size_t)(b + i) * E];
#pragma unroll
    for (int i = 0; i < 8; ++i) s += t[i];
  }
  for (; b < n; ++b) s += p[(size_t)b * E];
  return s;
}

// Totals, exclusive offsets, per-block starting positions, active list and tile table,
// one thread per expert and block-wide scans (blockDim.x >= E).
__device__ void scan_groups(const RouteView& r, int E, int nblocks, int tile) {
  __shared__ int3 totals;
  const int e = threadIdx.x;
  const int tot = e < E ? strided_sum(r.block_counts + e, E, nblocks) : 0;
  const int3 x = make_int3(tot, (tot + tile - 1) / tile, tot > 0 ? 1 : 0);
  const int3 ex = block_scan3(x, &totals);
  if (e < E) {
    r.counts[e] = tot;
    r.offsets[e] = ex.x;
    if (tot > 0) {
      r.active[ex.z] = e;
      r.zidx[e] = ex.z;
      int4* g = reinterpret_cast<int4*>(r.groups + (size_t)ex.z * kGroupInts);
      g[0] = make_int4(e, ex.x, tot, 0);
    }
    for (int s = 0; s < x.y; ++s) {
      r.tiles[3 * (ex.y + s)] = e;
      r.tiles[3 * (ex.y + s) + 1] = ex.x + s * tile;
      r.tiles[3 * (ex.y + s) + 2] = min(tile, tot - s * tile);
    }
    // starting position of block b's pairs of expert e
    int run = ex.x, b = 0;
    for (; b + 8 <= nblocks; b += 8) {
      int t[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) t[i] = r.block_counts[(size_t)(b + i) * E + e];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        r.block_start[(size_t)(b + i) * E + e] = run;
        run += t[i];
      }
    }
    for (; b < nblocks; ++b) {
      const int c = r.block_counts[(size_t)b * E + e];
      r.block_start[(size_t)b * E + e] = run;
      run += c;
    }
  }
  if (threadIdx.x == 0) {
    r.offsets[E] = totals.x;
    r.meta[0] = totals.z;
    r.meta[1] = totals.y;
  }
  __syncthreads();
}

// Stable placement of the pairs of block b: rank among equal experts = earlier pairs of
// the block with the same expert (warp match + per-warp counts), in pair order.
__device__ void block_scatter(const int32_t* ids, int64_t P, int E, int k, int b, const RouteView& r) {
  __shared__ __align__(16) unsigned short wc[kRouteBlock / 32][kMaxExperts];  // pairs per (warp, expert)
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t p = (int64_t)b * kRouteBlock + tid;
  const bool valid = tid < kRouteBlock && p < P;
  const int e = valid ? ids[p] : -1;
  zero_shared(&wc[0][0], sizeof(wc));
  __syncthreads();
  const unsigned mask = __match_any_sync(0xFFFFFFFFu, e);
  const int rank_in_warp = __popc(mask & ((1u << lane) - 1u));
  if (valid && rank_in_warp == 0) wc[warp][e] = (unsigned short)__popc(mask);
  __syncthreads();
  if (valid) {
    int before = 0;
    for (int w = 0; w < warp; ++w) before += wc[w][e];
    const int pos = r.block_start[(size_t)b * E + e] + before + rank_in_warp;
    r.pair_list[pos] = (int)p;
    r.pair_pos[p] = pos;
    const int rank = pos - r.offsets[e];
    if (rank < kGroupRows) r.groups[(size_t)r.zidx[e] * kGroupInts + 4 + rank] = (int)(p / k);
  }
  __syncthreads();
}

__global__ void __launch_bounds__(kRouteBlock) route_count_kernel(const int32_t* ids, int64_t P, int E, RouteView r) {
  block_count(ids, P, E, blockIdx.x, r.block_counts + (size_t)blockIdx.x * E);
}
__global__ void __launch_bounds__(kRouteBlock) route_scan_kernel(int E, int nblocks, int tile, RouteView r) {
  scan_groups(r, E, nblocks, tile);
}
__global__ void __launch_bounds__(kRouteBlock) route_scatter_kernel(const int32_t* ids, int64_t P, int E, int k,
                                                                    RouteView r) {
  block_scatter(ids, P, E, k, blockIdx.x, r);
}

// Decode-sized routing (T*k <= kRouteBlock, T <= 32): every phase in one CTA, with the
// histogram, the scan and the placement in shared memory; only the results go to device
// memory.
__global__ void __launch_bounds__(kRouteBlock) route_small_kernel(const float* logits, int T, int E, int k,
                                                                  int32_t* ids, float* wts, int tile, RouteView r) {
  __shared__ int s_ids[kRouteBlock];
  __shared__ int hist[kMaxExperts];
  __shared__ int off[kMaxExperts];
  __shared__ int zid[kMaxExperts];
  __shared__ int3 totals;
  __shared__ __align__(16) unsigned short wc[kRouteBlock / 32][kMaxExperts];  // pairs per (warp, expert)
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // The consumers of the routing wait for this grid to complete before reading it; the
  // logits may come from the preceding kernel.
  if (tid == 0) pdl_launch_dependents();
  for (int e = tid; e < E; e += blockDim.x) hist[e] = 0;
  zero_shared(&wc[0][0], sizeof(wc));
  pdl_wait();
  if (warp < T) warp_topk(logits + (int64_t)warp * E, E, k, ids + warp * k, wts + warp * k, s_ids + warp * k);
  __syncthreads();
  // pairs p = t*k + j: histogram (order-free integer counts) and rank within the warp
  const int P = T * k;
  const bool valid = tid < P;
  const int e = valid ? s_ids[tid] : -1;
  if (valid) atomicAdd(&hist[e], 1);
  const unsigned mask = __match_any_sync(0xFFFFFFFFu, e);
  const int rank_in_warp = __popc(mask & ((1u << lane) - 1u));
  if (valid && rank_in_warp == 0) wc[warp][e] = (unsigned short)__popc(mask);
  __syncthreads();
  // totals, exclusive offsets, active list and tile table (one thread per expert)
  const int tot = tid < E ? hist[tid] : 0;
  const int3 ex = block_scan3(make_int3(tot, (tot + tile - 1) / tile, tot > 0 ? 1 : 0), &totals);
  if (tid < E) {
    r.counts[tid] = tot;
    r.offsets[tid] = ex.x;
    off[tid] = ex.x;
    zid[tid] = ex.z;
    if (tot > 0) {
      r.active[ex.z] = tid;
      r.zidx[tid] = ex.z;
      reinterpret_cast<int4*>(r.groups + (size_t)ex.z * kGroupInts)[0] = make_int4(tid, ex.x, tot, 0);
    }
    for (int s = 0; s * tile < tot; ++s) {
      r.tiles[3 * (ex.y + s)] = tid;
      r.tiles[3 * (ex.y + s) + 1] = ex.x + s * tile;
      r.tiles[3 * (ex.y + s) + 2] = min(tile, tot - s * tile);
    }
  }
  if (tid == 0) {
    r.offsets[E] = totals.x;
    r.meta[0] = totals.z;
    r.meta[1] = totals.y;
  }
  __syncthreads();
  // stable placement: experts ascending, pairs ascending within an expert
  if (valid) {
    int before = 0;
    for (int w = 0; w < warp; ++w) before += wc[w][e];
    const int pos = off[e] + before + rank_in_warp;
    r.pair_list[pos] = tid;
    r.pair_pos[tid] = pos;
    const int rank = before + rank_in_warp;
    if (rank < kGroupRows) r.groups[(size_t)zid[e] * kGroupInts + 4 + rank] = tid / k;
  }
}

RouteView route_view(void* ws, int64_t T, int E, int k) {
  const RouteLayout L = route_layout(T, E, k);
  uint8_t* b = static_cast<uint8_t*>(ws);
  RouteView v;
  v.meta = reinterpret_cast<int*>(b + L.meta);
  v.counts = reinterpret_cast<int*>(b + L.counts);
  v.offsets = reinterpret_cast<int*>(b + L.offsets);
  v.active = reinterpret_cast<int*>(b + L.active);
  v.pair_list = reinterpret_cast<int*>(b + L.pair_list);
  v.pair_pos = reinterpret_cast<int*>(b + L.pair_pos);
  v.tiles = reinterpret_cast<int*>(b + L.tiles);
  v.groups = reinterpret_cast<int*>(b + L.groups);
  v.zidx = reinterpret_cast<int*>(b + L.zidx);
  v.block_counts = reinterpret_cast<int*>(b + L.block_counts);
  v.block_start = reinterpret_cast<int*>(b + L.block_start);
  return v;
}

int launch_route(const float* logits, int64_t T, int E, int k, int32_t* ids, float* wts, void* ws, void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  RouteView r = route_view(ws, T, E, k);
  const int64_t P = T * k;
  if (P <= kRouteBlock && T <= 32) {
    if (launch_pdl(route_small_kernel, dim3(1), dim3(kRouteBlock), 0, s, logits, (int)T, E, k, ids, wts,
                   (int)kRouteTile, r) != cudaSuccess)
      return QG_ERR_CUDA;
  } else {
    const int64_t nb = (P + kRouteBlock - 1) / kRouteBlock;
    route_topk_kernel<<<(unsigned)((T + 7) / 8), 256, 0, s>>>(logits, T, E, k, ids, wts);
    route_count_kernel<<<(unsigned)nb, kRouteBlock, 0, s>>>(ids, P, E, r);
    route_scan_kernel<<<1, kRouteBlock, 0, s>>>(E, (int)nb, kRouteTile, r);
    route_scatter_kernel<<<(unsigned)nb, kRouteBlock, 0, s>>>(ids, P, E, k, r);
  }
  return cudaGetLastError() == cudaSuccess ? QG_OK : QG_ERR_CUDA;
}

}  // namespace qg
