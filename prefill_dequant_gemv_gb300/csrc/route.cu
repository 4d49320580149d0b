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

namespace qg {

constexpr int kRouteBlock = 1024;  // pairs per grouping block (one thread per pair)

// Warp-level top-k of one token's logits; lane l holds logits l, l+32, ... (<= 32 each).
__device__ void warp_topk(const float* lg, int E, int k, int32_t* ids, float* wts) {
  const int lane = threadIdx.x & 31;
  float v[32];
  uint32_t taken = 0;
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = (lane + 32 * i < E) ? lg[lane + 32 * i] : 0.0f;
  float sel[16];
  int sid[16];
  for (int j = 0; j < k; ++j) {
    // lane-local best: largest value, lowest index on ties
    float bv = 0.0f;
    int bi = 0x7FFFFFFF;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const int e = lane + 32 * i;
      if (e < E && !((taken >> i) & 1u) && (bi == 0x7FFFFFFF || v[i] > bv || (v[i] == bv && e < bi))) {
        bv = v[i];
        bi = e;
      }
    }
#pragma unroll
    for (int off = 16; off; off >>= 1) {
      const float ov = __shfl_xor_sync(0xFFFFFFFFu, bv, off);
      const int oi = __shfl_xor_sync(0xFFFFFFFFu, bi, off);
      if (oi != 0x7FFFFFFF && (bi == 0x7FFFFFFF || ov > bv || (ov == bv && oi < bi))) {
        bv = ov;
        bi = oi;
      }
    }
    if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
    sel[j] = bv;
    sid[j] = bi;
  }
  if (lane == 0) {
    // softmax over the k kept logits, in selection (descending) order
    float z[16], sum = 0.0f;
    for (int j = 0; j < k; ++j) {
      z[j] = expf(sel[j] - sel[0]);
      sum += z[j];
    }
    for (int j = 0; j < k; ++j) {
      ids[j] = sid[j];
      wts[j] = z[j] / sum;
    }
  }
}

__global__ void __launch_bounds__(256) route_topk_kernel(const float* logits, int64_t T, int E, int k, int32_t* ids,
                                                         float* wts) {
  const int64_t t = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (t >= T) return;
  warp_topk(logits + t * E, E, k, ids + t * k, wts + t * k);
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

// Totals, exclusive offsets, per-block starting positions, active list, tile table.
__device__ void scan_groups(const RouteView& r, int E, int nblocks, int tile) {
  __shared__ int tot[kMaxExperts];
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int s = 0;
    for (int b = 0; b < nblocks; ++b) s += r.block_counts[(size_t)b * E + e];
    tot[e] = s;
    r.counts[e] = s;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int off = 0, na = 0, nt = 0;
    for (int e = 0; e < E; ++e) {
      r.offsets[e] = off;
      if (tot[e] > 0) {
        r.active[na++] = e;
        for (int s = 0; s < tot[e]; s += tile) {
          r.tiles[3 * nt] = e;
          r.tiles[3 * nt + 1] = off + s;
          r.tiles[3 * nt + 2] = min(tile, tot[e] - s);
          ++nt;
        }
      }
      off += tot[e];
    }
    r.offsets[E] = off;
    r.meta[0] = na;
    r.meta[1] = nt;
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int run = r.offsets[e];
    for (int b = 0; b < nblocks; ++b) {
      const int c = r.block_counts[(size_t)b * E + e];
      r.block_start[(size_t)b * E + e] = run;
      run += c;
    }
  }
  __syncthreads();
}

// Stable placement of the pairs of block b: rank among equal experts = earlier pairs of
// the block with the same expert (warp match + per-warp counts), in pair order.
__device__ void block_scatter(const int32_t* ids, int64_t P, int E, int b, const RouteView& r) {
  __shared__ unsigned short wc[kRouteBlock / 32][kMaxExperts];  // pairs per (warp, expert)
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t p = (int64_t)b * kRouteBlock + tid;
  const bool valid = tid < kRouteBlock && p < P;
  const int e = valid ? ids[p] : -1;
  for (int i = tid; i < (kRouteBlock / 32) * E; i += blockDim.x) wc[i / E][i % E] = 0;
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
  }
  __syncthreads();
}

__global__ void __launch_bounds__(kRouteBlock) route_count_kernel(const int32_t* ids, int64_t P, int E, RouteView r) {
  block_count(ids, P, E, blockIdx.x, r.block_counts + (size_t)blockIdx.x * E);
}
__global__ void __launch_bounds__(kRouteBlock) route_scan_kernel(int E, int nblocks, int tile, RouteView r) {
  scan_groups(r, E, nblocks, tile);
}
__global__ void __launch_bounds__(kRouteBlock) route_scatter_kernel(const int32_t* ids, int64_t P, int E,
                                                                    RouteView r) {
  block_scatter(ids, P, E, blockIdx.x, r);
}

// Decode-sized routing (T*k <= kRouteBlock, T <= 32): every phase in one CTA.
__global__ void __launch_bounds__(kRouteBlock) route_small_kernel(const float* logits, int T, int E, int k,
                                                                  int32_t* ids, float* wts, int tile, RouteView r) {
  const int warp = threadIdx.x >> 5;
  for (int t = warp; t < T; t += kRouteBlock / 32) warp_topk(logits + (int64_t)t * E, E, k, ids + t * k, wts + t * k);
  __threadfence_block();
  __syncthreads();
  const int64_t P = (int64_t)T * k;
  block_count(ids, P, E, 0, r.block_counts);
  scan_groups(r, E, 1, tile);
  block_scatter(ids, P, E, 0, r);
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
  v.block_counts = reinterpret_cast<int*>(b + L.block_counts);
  v.block_start = reinterpret_cast<int*>(b + L.block_start);
  return v;
}

int launch_route(const float* logits, int64_t T, int E, int k, int32_t* ids, float* wts, void* ws, void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  RouteView r = route_view(ws, T, E, k);
  const int64_t P = T * k;
  if (P <= kRouteBlock && T <= 32) {
    route_small_kernel<<<1, kRouteBlock, 0, s>>>(logits, (int)T, E, k, ids, wts, kRouteTile, r);
  } else {
    const int64_t nb = (P + kRouteBlock - 1) / kRouteBlock;
    route_topk_kernel<<<(unsigned)((T + 7) / 8), 256, 0, s>>>(logits, T, E, k, ids, wts);
    route_count_kernel<<<(unsigned)nb, kRouteBlock, 0, s>>>(ids, P, E, r);
    route_scan_kernel<<<1, kRouteBlock, 0, s>>>(E, (int)nb, kRouteTile, r);
    route_scatter_kernel<<<(unsigned)nb, kRouteBlock, 0, s>>>(ids, P, E, r);
  }
  return cudaGetLastError() == cudaSuccess ? QG_OK : QG_ERR_CUDA;
}

}  // namespace qg
