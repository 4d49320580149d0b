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
// l+32, ... (16 registers; the expert of slot i is l + 32 i).  Each lane first extracts its
// three best keys in order (ties to the lower slot, i.e. the lower expert).  Each of k rounds
// then takes the warp maximum of the lanes' current heads and the warp minimum of the experts
// holding it (two single-instruction warp reductions), and the winner's lane steps to its
// next key with three selects -- no search on the rounds' serial path.  A lane that has won
// three times before the last round has no extracted key left: the rounds are then redone
// from all 16 keys, the winner's lane searching its next best each time (the same result,
// only slower; the fast rounds never pick a wrong key before that point).  Lane
// j keeps the j-th winner and the k lanes compute the softmax over the kept logits in parallel.
__device__ __forceinline__ void warp_topk(const float* lg, int E, int k, int32_t* ids, float* wts, int* ids_copy = nullptr) {
  const int lane = threadIdx.x & 31;
  uint32_t key[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const int e = lane + 32 * i;
    key[i] = e < E ? order_key(lg[e]) : 0u;
  }
  uint32_t h0, h1, h2;  // the lane's three best keys, descending, and their experts
  int e0, e1, e2;
  {
    uint32_t kk[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) kk[i] = key[i];
    int bi;
    lane_best(kk, h0, bi);
    e0 = lane + 32 * bi;
#pragma unroll
    for (int i = 0; i < 16; ++i) kk[i] = (i == bi) ? 0u : kk[i];
    lane_best(kk, h1, bi);
    e1 = lane + 32 * bi;
#pragma unroll
    for (int i = 0; i < 16; ++i) kk[i] = (i == bi) ? 0u : kk[i];
    lane_best(kk, h2, bi);
    e2 = lane + 32 * bi;
  }
  uint32_t mine = 0u, top = 0u;
  int mine_id = 0, taken = 0;
  bool short_of_keys = false;
  for (int j = 0; j < k; ++j) {
    const uint32_t kmax = __reduce_max_sync(0xFFFFFFFFu, h0);
    const int win = (int)__reduce_min_sync(0xFFFFFFFFu, h0 == kmax ? (uint32_t)e0 : 0xFFFFFFFFu);
    if (j == 0) top = kmax;
    if (lane == j) {
      mine = kmax;
      mine_id = win;
    }
    const bool w = (win & 31) == lane;
    taken += w;
    short_of_keys |= taken == 3 && j + 1 < k;  // its head is now empty though rounds remain
    h0 = w ? h1 : h0;
    e0 = w ? e1 : e0;
    h1 = w ? h2 : h1;
    e1 = w ? e2 : e1;
    h2 = w ? 0u : h2;
  }
  if (__any_sync(0xFFFFFFFFu, short_of_keys)) {  // a lane may have needed a fourth key: redo from all 16
    uint32_t bk;
    int bi;
    lane_best(key, bk, bi);
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

// Shared-memory scratch of route_decode_block: each token's experts as a bit set over the
// (at most kMaxExperts) experts, their union in row kRouteTokens, and per row and 32-bit
// word the number of set bits in the words before it.
constexpr int kRouteTokens = 4;
constexpr int kRouteWords = kMaxExperts / 32;
struct BlockRouteSmem {
  int ids[kBlockRoutePairs];
  float wts[kBlockRoutePairs];
  uint32_t mask[kRouteTokens + 1][kRouteWords];
  int before[kRouteTokens + 1][kRouteWords];
  int groups[kBlockRoutePairs * kGroupInts];
  int n_active;
};

// Routing of T <= kRouteTokens tokens (P = T*k <= kBlockRoutePairs pairs) by one CTA: warps
// 0..T-1 take one token each (warp_topk); then every pair is placed -- experts ascending,
// pairs ascending within an expert -- from the tokens' expert bit sets, in constant work a
// pair: a token's experts are distinct, so the pairs of expert e before pair (t, j) are the
// tokens before t that chose e; the pairs of smaller experts are the set bits below e of
// every token; the active experts below e, the set bits below e of the union.  Every CTA
// that calls it builds the same group table in shared memory (sm.groups, kGroupInts ints per
// active expert; returns the number of active experts).  The CTA with `write` set also
// stores the router's outputs, the same values qmoe_route stores for these tokens: ids,
// wts, counts, offsets, active, zidx, groups, tiles (one per active expert: a decode expert
// has at most T < tile pairs), pair_list, pair_pos and meta.  Every thread of the CTA must
// call it; the threads of warps T and above run `idle()` (work that does not depend on the
// routing) while warps 0..T-1 take the top-k.
template <class Idle>
__device__ __forceinline__ int route_decode_block(const float* logits, int T, int E, int k, BlockRouteSmem& sm,
                                                  bool write, int32_t* ids, float* wts, const RouteView& r,
                                                  Idle&& idle) {
  const int tid = threadIdx.x, warp = tid >> 5;
  const int P = T * k;
  constexpr int kRows = kRouteTokens + 1, kU = kRouteTokens;  // row kU: the union
  if (tid < kRouteTokens * kRouteWords && tid / kRouteWords >= T) (&sm.mask[0][0])[tid] = 0u;  // no token
  if (warp < T) {  // the token's top-k, then its expert set, one word a lane (warp reductions)
    const int lane = tid & 31;
    warp_topk(logits + (int64_t)warp * E, E, k, sm.ids + warp * k, sm.wts + warp * k);
    __syncwarp();
    const int ex = lane < k ? sm.ids[warp * k + lane] : -1;
    uint32_t word = 0u;
#pragma unroll
    for (int w = 0; w < kRouteWords; ++w) {
      const uint32_t v = __reduce_or_sync(0xFFFFFFFFu, (ex >> 5) == w ? 1u << (ex & 31) : 0u);
      if (lane == w) word = v;
    }
    if (lane < kRouteWords) sm.mask[warp][lane] = word;
  } else {
    idle();
  }
  __syncthreads();
  int e = -1, t = 0;
  if (tid < P) {
    e = sm.ids[tid];
    t = tid / k;
  }
  if (tid < 3 * 32) {  // rows in half-warps: word prefix counts by an inclusive scan of 16
    const int row = tid >> 4, w = tid & 15;
    uint32_t bits = 0u;
    if (row < kRouteTokens) {
      bits = sm.mask[row][w];
    } else if (row == kU) {
#pragma unroll
      for (int tt = 0; tt < kRouteTokens; ++tt) bits |= sm.mask[tt][w];
      sm.mask[kU][w] = bits;
    }
    const int v = __popc(bits);
    int sc = v;
#pragma unroll
    for (int d = 1; d < 16; d <<= 1) {
      const int n = __shfl_up_sync(0xFFFFFFFFu, sc, d, 16);
      if (w >= d) sc += n;
    }
    if (row < kRows) sm.before[row][w] = sc - v;
  }
  __syncthreads();
  int rank = 0, first = 0, cnt = 0, z = 0;
  if (tid < P) {
    const int w = e >> 5, b = e & 31;
    const uint32_t low = (1u << b) - 1u;
    for (int tt = 0; tt < T; ++tt) {
      const uint32_t mw = sm.mask[tt][w];
      const int bit = (int)((mw >> b) & 1u);
      cnt += bit;
      rank += tt < t ? bit : 0;
      first += sm.before[tt][w] + __popc(mw & low);
    }
    z = sm.before[kU][w] + __popc(sm.mask[kU][w] & low);
    if (rank == 0) {
      int* g = sm.groups + z * kGroupInts;
      g[0] = e;
      g[1] = first;
      g[2] = cnt;
      g[3] = 0;
    }
    if (rank < kGroupRows) sm.groups[z * kGroupInts + 4 + rank] = t;
  }
  const int n_active = sm.before[kU][kRouteWords - 1] + __popc(sm.mask[kU][kRouteWords - 1]);
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
      if (rank < kGroupRows) r.groups[(size_t)z * kGroupInts + 4 + rank] = t;
    }
    for (int x = tid; x < E; x += blockDim.x) {  // pairs of expert x, and of the experts below it
      const int w = x >> 5, b = x & 31;
      const uint32_t low = (1u << b) - 1u;
      int c = 0, f = 0;
      for (int tt = 0; tt < T; ++tt) {
        const uint32_t mw = sm.mask[tt][w];
        c += (int)((mw >> b) & 1u);
        f += sm.before[tt][w] + __popc(mw & low);
      }
      r.counts[x] = c;
      r.offsets[x] = f;
    }
    if (tid == 0) {
      r.offsets[E] = P;
      r.meta[0] = n_active;
      r.meta[1] = n_active;
    }
  }
  return n_active;
}

}  // namespace qg
