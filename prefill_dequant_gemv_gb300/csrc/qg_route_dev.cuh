// Router device functions shared by the router kernels and the decode chain's gate/up
// launch, which routes its tokens itself (TurboEXL3 article §4.2: the router's top-k and
// softmax run inside an FFN launch).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "qg_route.h"

namespace qg {

// Order-preserving 32-bit key of an fp32 logit: larger logit, larger key; -0 ties with +0
// and NaN sorts below every number (a stable descending sort of the values puts NaN last)
// but above key 0, which marks padding and experts already taken.
__device__ __forceinline__ uint32_t order_key(float v) {
  uint32_t u = __float_as_uint(v);
  if (u == 0x80000000u) u = 0u;
  if ((u & 0x7FFFFFFFu) > 0x7F800000u) return 1u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_value(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k ^ 0x80000000u) : ~k);
}

// Largest key of a lane's 16 (ties to the lower slot, i.e. the lower expert index): a
// 4-level tree over fixed register indices.
__device__ __forceinline__ void lane_best(const uint32_t (&key)[16], uint32_t& bk, int& bi) {
  uint32_t k8[8];
  int i8[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const bool hi = key[2 * i + 1] > key[2 * i];
    k8[i] = hi ? key[2 * i + 1] : key[2 * i];
    i8[i] = hi ? 2 * i + 1 : 2 * i;
  }
#pragma unroll
  for (int w = 4; w >= 1; w >>= 1)
#pragma unroll
    for (int i = 0; i < w; ++i) {
      const bool hi = k8[i + w] > k8[i] || (k8[i + w] == k8[i] && i8[i + w] < i8[i]);
      k8[i] = hi ? k8[i + w] : k8[i];
      i8[i] = hi ? i8[i + w] : i8[i];
    }
  bk = k8[0];
  bi = i8[0];
}

// Warp-level top-k of one token's logits (E <= 512): lane l holds the keys of logits l,
// l+32, ... (16 registers; the expert of slot i is l + 32 i).  Each of k rounds takes the
// warp maximum of the lanes' best keys and the warp minimum of the experts holding it (two
// single-instruction warp reductions); the winner's lane clears that slot and finds its
// next best.  Lane j keeps the j-th winner and the k lanes compute the softmax over the kept
// logits in parallel.
__device__ __forceinline__ void warp_topk(const float* lg, int E, int k, int32_t* ids, float* wts, int* ids_copy = nullptr) {
  const int lane = threadIdx.x & 31;
  uint32_t key[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const int e = lane + 32 * i;
    key[i] = e < E ? order_key(lg[e]) : 0u;
  }
  uint32_t bk;
  int bi;
  lane_best(key, bk, bi);
  uint32_t mine = 0u, top = 0u;
  int mine_id = 0;
  for (int j = 0; j < k; ++j) {
    const uint32_t kmax = __reduce_max_sync(0xFFFFFFFFu, bk);
    const int win = (int)__reduce_min_sync(0xFFFFFFFFu, bk == kmax ? (uint32_t)(lane + 32 * bi) : 0xFFFFFFFFu);
    if (j == 0) top = kmax;
    if (lane == j) {
      mine = kmax;
      mine_id = win;
    }
    if ((win & 31) == lane) {  // the winner's lane takes the slot out and finds its next best
#pragma unroll
      for (int i = 0; i < 16; ++i) key[i] = (i == (win >> 5)) ? 0u : key[i];
      lane_best(key, bk, bi);
    }
  }
  // softmax over the k kept logits (descending order), shifted by the largest
  const float z = lane < k ? expf(key_value(mine) - key_value(top)) : 0.0f;
  float sum = z;
#pragma unroll
  for (int off = 16; off; off >>= 1) sum += __shfl_xor_sync(0xFFFFFFFFu, sum, off);
  if (lane < k) {
    ids[lane] = mine_id;
    wts[lane] = z / sum;
    if (ids_copy) ids_copy[lane] = mine_id;
  }
}

// Shared-memory scratch of route_decode_block.
struct BlockRouteSmem {
  int ids[kBlockRoutePairs];
  float wts[kBlockRoutePairs];
  int rank[kBlockRoutePairs];   // pairs of the same expert before this one
  int groups[kBlockRoutePairs * kGroupInts];
  int n_active;
};

// Routing of T tokens (P = T*k <= kBlockRoutePairs pairs) by one CTA: warps 0..T-1 take one
// token each (warp_topk), then threads 0..P-1 place the pairs -- experts ascending, pairs
// ascending within an expert -- by counting (P is small), not sorting.  Every CTA that calls
// it builds the same group table in shared memory (sm.groups, kGroupInts ints per active
// expert; returns the number of active experts).  The CTA with `write` set also stores the
// router's outputs, the same values qmoe_route stores for these tokens: ids, wts, counts,
// offsets, active, zidx, groups, tiles (one per active expert: a decode expert has at most
// T < tile pairs), pair_list, pair_pos and meta.  Every thread of the CTA must call it.
__device__ __forceinline__ int route_decode_block(const float* logits, int T, int E, int k, BlockRouteSmem& sm,
                                                  bool write, int32_t* ids, float* wts, const RouteView& r) {
  const int tid = threadIdx.x, warp = tid >> 5;
  const int P = T * k;
  if (warp < T) warp_topk(logits + (int64_t)warp * E, E, k, sm.ids + warp * k, sm.wts + warp * k);
  __syncthreads();
  int e = -1, rank = 0, first = 0, cnt = 0;
  if (tid < P) {
    e = sm.ids[tid];
    for (int q = 0; q < P; ++q) {
      const int eq = sm.ids[q];
      first += eq < e;
      cnt += eq == e;
      rank += (eq == e) && (q < tid);
    }
    sm.rank[tid] = rank;
  }
  __syncthreads();
  int z = 0, n_active = 0;
  if (tid < P) {
    for (int q = 0; q < P; ++q) {
      const bool lead = sm.rank[q] == 0;  // the first pair of its expert
      n_active += lead;
      z += lead && sm.ids[q] < e;
    }
    if (rank == 0) {
      int* g = sm.groups + z * kGroupInts;
      g[0] = e;
      g[1] = first;
      g[2] = cnt;
      g[3] = 0;
    }
    if (rank < kGroupRows) sm.groups[z * kGroupInts + 4 + rank] = tid / k;
    if (tid == 0) sm.n_active = n_active;
  }
  __syncthreads();
  if (write) {
    if (tid < P) {
      ids[tid] = e;
      wts[tid] = sm.wts[tid];
      const int pos = first + rank;
      r.pair_list[pos] = tid;
      r.pair_pos[tid] = pos;
      if (rank == 0) {
        r.active[z] = e;
        r.zidx[e] = z;
        r.tiles[3 * z] = e;
        r.tiles[3 * z + 1] = first;
        r.tiles[3 * z + 2] = cnt;
        reinterpret_cast<int4*>(r.groups + (size_t)z * kGroupInts)[0] = make_int4(e, first, cnt, 0);
      }
      if (rank < kGroupRows) r.groups[(size_t)z * kGroupInts + 4 + rank] = tid / k;
    }
    for (int x = tid; x < E; x += blockDim.x) {
      int c = 0, f = 0;
      for (int q = 0; q < P; ++q) {
        c += sm.ids[q] == x;
        f += sm.ids[q] < x;
      }
      r.counts[x] = c;
      r.offsets[x] = f;
    }
    if (tid == 0) {
      r.offsets[E] = P;
      r.meta[0] = sm.n_active;
      r.meta[1] = sm.n_active;
    }
  }
  return sm.n_active;
}

}  // namespace qg
