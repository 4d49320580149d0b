// Router workspace layout (host and device).
#pragma once

#include <stddef.h>
#include <stdint.h>

namespace qg {

constexpr int kMaxExperts = 512;
constexpr int kMaxTopk = 16;
constexpr int kRouteTile = 192;  // pairs per grouped-prefill tile (the tensor-core N)

// Group table entry (8 ints) of active expert z (ascending experts): expert, first grouped
// position, pair count, 0, then the tokens of its first kGroupRows pairs.
constexpr int kGroupRows = 4;
constexpr int kGroupInts = 8;
// Pairs one CTA routes in the decode chain's gate/up launch (T <= 4 tokens, k <= 16).
constexpr int kBlockRoutePairs = 64;

struct RouteLayout {
  size_t meta, counts, offsets, active, pair_list, pair_pos, tiles, groups, zidx, block_counts, block_start, total;
  int64_t max_tiles, nblocks;
};

__host__ __device__ inline RouteLayout route_layout(int64_t T, int E, int k) {
  RouteLayout L;
  const int64_t P = T * k;
  L.nblocks = (P + 1023) / 1024;
  L.max_tiles = (P + kRouteTile - 1) / kRouteTile + E;
  size_t o = 0;
  auto take = [&o](size_t bytes) {
    const size_t at = o;
    o += (bytes + 255) & ~(size_t)255;
    return at;
  };
  L.meta = take(64);                      // [0] active experts, [1] tiles
  L.counts = take((size_t)E * 4);
  L.offsets = take((size_t)(E + 1) * 4);
  L.active = take((size_t)E * 4);
  L.pair_list = take((size_t)P * 4);      // grouped position -> pair t*k + j
  L.pair_pos = take((size_t)P * 4);       // pair -> grouped position
  L.tiles = take((size_t)L.max_tiles * 12);  // (expert, first position, count)
  L.groups = take((size_t)E * kGroupInts * 4);  // group table, one entry per active expert
  L.zidx = take((size_t)E * 4);                 // expert -> its index in the active list
  L.block_counts = take((size_t)L.nblocks * E * 4);
  L.block_start = take((size_t)L.nblocks * E * 4);
  L.total = o;
  return L;
}

struct RouteView {
  int* meta;
  int* counts;
  int* offsets;
  int* active;
  int* pair_list;
  int* pair_pos;
  int* tiles;
  int* groups;
  int* zidx;
  int* block_counts;
  int* block_start;
};

RouteView route_view(void* ws, int64_t T, int E, int k);
int launch_route(const float* logits, int64_t T, int E, int k, int32_t* ids, float* wts, void* ws, void* stream);

}  // namespace qg
