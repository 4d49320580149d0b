// Tensor-core GEMM for small token counts (5..128 rows): Y[t, n] = bf16( sum_k W[n, k] X[t, k]
// (+ R[t, n]) ) -- the prefill GEMM's decode-once-multiply-many scheme (TurboEXL3 article
// §4.1) shaped for few tokens, where the 256-token tile of the large-batch kernel would leave
// most of each MMA empty and its one accumulator chain over all of K would set the pace.
//
// One CTA computes a 128-row tile of W against NB <= 128 tokens over a K range; a cluster of
// ks CTAs (the grid's z) splits K when there are too few row x token tiles to fill the GPU.
//   warp 0      producer: per 64-deep stage, bulk-copies the packed weight tile and TMA-loads
//               the NB x 64 activation tile (128-byte swizzle) into an 8-stage ring
//   warp 1      allocates the 512 TMEM columns and issues tcgen05.mma M=128 N=NB K=16 (A from
//               TMEM, B from shared memory) into one accumulator, with every operand prepared
//               ahead (one thread issues an MMA every ~48 cycles at best)
//   warps 2-9   decode in two groups of four, alternate pairs of stages, each row's 64 inputs
//               per stage written with one 32-column tcgen05.st; then the epilogue
// With few tokens the MMAs are short and the MMA thread's own instruction stream sets the
// pace, so stages travel in pairs -- one readiness wait and one commit (freeing both stages'
// buffers and A slots) per pair -- and the descriptors are prepared outside the issue.
// Epilogue: every thread of warps 2-5 scales its row of the accumulator into a token-major
// fp32 tile in its CTA's idle stage buffers; after a cluster barrier each
// CTA takes every ks-th group of 8 rows of one token, adds the ks partial tiles in rank order
// (distributed shared memory), the residual, rounds to bf16 once and writes 16 bytes.  No
// workspace, no atomics: results are deterministic.  Every wait is bounded (QG_ERR_TIMEOUT in
// the workspace status word) and TMEM is freed on every path.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>

#include "qg_common.cuh"
#include "qg_decode_tile.cuh"
#include "qg_internal.h"
#include "qg_sync.cuh"
#include "qg_tc.cuh"

namespace qg {

constexpr int kSmThreads = 320;
constexpr int kSmRawMax = 7168;  // >= Q6_K tile 6144 + 512 + 256
constexpr uint32_t kSmA0 = 256;  // accumulators in TMEM columns [0, 256), A ring in [256, 512)
constexpr int kSmAS = 8;         // A ring stages of 32 columns

template <int NB>
struct SmCfg {
  static constexpr int B = NB * 128;                                 // NB token rows x 64 bf16
  static constexpr int STAGE = ((B + kSmRawMax) + 1023) & ~1023;     // B tile 1024-byte aligned
  static constexpr int S = kSmAS;  // stage ring = A ring: stage j uses buffer and A slot j % 8
  static constexpr int SMEM = 1024 + S * STAGE + 1024;
  static_assert(NB <= (int)kSmA0, "accumulator");
  static_assert(NB * 128 * 4 <= S * STAGE, "epilogue tile fits in the stage buffers");
  static_assert(SMEM <= 232448, "shared memory");
};

struct SmallArgs {
  const uint8_t* codes;
  const uint8_t* scales;
  const uint8_t* aux;
  const __nv_bfloat16* res;
  __nv_bfloat16* y;
  int64_t ldr, ldy;
  int64_t n, t;
  int KG;
  int ks;  // CTAs per cluster splitting K
  float ts;
  int* status;
};

__device__ __forceinline__ float4 ld_cluster_f32x4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0,%1,%2,%3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr) : "memory");
  return v;
}

template <int FMT, int NB>
__global__ void __launch_bounds__(kSmThreads, 1)
    gemm_small_kernel(const __grid_constant__ CUtensorMap tmx, const SmallArgs a) {
  using F = Fmt<FMT>;
  using C = SmCfg<NB>;
  constexpr int kRaw = F::TB + 128 * F::SB + fmt_aux(FMT);  // tile, scales, aux of its 256 inputs
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  // full[s]: stage s landed; pair barriers (pair q = stages 2q, 2q+1 uses index q % 4):
  // afull[]: the pair's A operand is in TMEM, empty[]: the pair's MMAs completed
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::S * C::STAGE);
  uint64_t* afull = full + C::S;
  uint64_t* empty = afull + C::S / 2;
  uint64_t* done = empty + C::S / 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int tile_n = blockIdx.x;
  const int t0 = blockIdx.y * NB;
  const int ks = a.ks;
  const int rank = ks > 1 ? (int)cluster_rank() : 0;
  const int kt0 = (int)((int64_t)rank * a.KG / ks), kt1 = (int)((int64_t)(rank + 1) * a.KG / ks);
  const int nst = kt1 - kt0;  // stages of this CTA (>= 1: the host keeps ks <= KG)

  if (tid == 0) {
    for (int s = 0; s < C::S; ++s) mbar_init(&full[s], 1);
    for (int q = 0; q < C::S / 2; ++q) {
      mbar_init(&afull[q], 4);  // the four decode warps of the pair's group
      mbar_init(&empty[q], 1);
    }
    mbar_init(done, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {  // producer
      int issued = 0;
      for (int j = 0; j < nst; ++j) {
        const int s = j % C::S;
        if (j >= C::S && !mbar_wait_bounded(&empty[s >> 1], (uint32_t)((j / C::S) & 1) ^ 1u, a.status)) break;
        uint8_t* st = smem + s * C::STAGE;
        const int kt = kt0 + j;
        const int64_t tile = (int64_t)tile_n * a.KG + kt;
        mbar_arrive_expect_tx(&full[s], kRaw + C::B);
        bulk_g2s(st + C::B, a.codes + tile * F::TB, F::TB, &full[s]);
        bulk_g2s(st + C::B + F::TB, a.scales + tile * (128 * F::SB), 128 * F::SB, &full[s]);
        if (fmt_aux(FMT))
          bulk_g2s(st + C::B + F::TB + 128 * F::SB,
                   a.aux + ((int64_t)tile_n * (a.KG / 4) + kt / 4) * fmt_aux(FMT), fmt_aux(FMT), &full[s]);
        tma_load_2d(st, &tmx, kt * 64, t0, &full[s]);
        ++issued;
      }
      // do not leave copies in flight into this CTA's shared memory
      for (int j = (issued > C::S ? issued - C::S : 0); j < issued; ++j)
        mbar_wait_bounded(&full[j % C::S], (uint32_t)(j / C::S) & 1u, a.status);
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {  // MMA issuer
      constexpr uint32_t idesc = idesc_bf16_f32(128, NB);
      const uint32_t lo0 = sw128_desc_lo(smem_u32(smem));  // stage s: lo0 + s * STAGE / 16
      // the decoders waited for each stage's landing before arriving on afull, so one wait
      // per pair covers both its A and its B
      for (int q = 0; 2 * q < nst; ++q) {
        const int pq = q % (C::S / 2);
        if (!mbar_wait_bounded(&afull[pq], (uint32_t)(q / (C::S / 2)) & 1u, a.status)) break;
        tc_fence_after();
        const uint32_t s0 = 2u * (uint32_t)pq;  // the pair's stages s0, s0 + 1
        const uint32_t ta = tmem + kSmA0 + 32u * s0, lo = lo0 + s0 * (uint32_t)(C::STAGE / 16);
        if (q == 0) mma_bf16_ts_fast<false>(tmem, ta, lo, idesc);
        else mma_bf16_ts_fast<true>(tmem, ta, lo, idesc);
#pragma unroll
        for (int kk = 1; kk < 4; ++kk) mma_bf16_ts_fast<true>(tmem, ta + 8u * kk, lo + 2u * kk, idesc);
        if (2 * q + 1 < nst) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_bf16_ts_fast<true>(tmem, ta + 32u + 8u * kk, lo + (uint32_t)(C::STAGE / 16) + 2u * kk, idesc);
        }
        mma_commit(&empty[pq]);
      }
      mma_commit(done);  // also drains whatever was issued if the loop stopped early
    }
    __syncwarp();
  }

  bool ok = true;
  if (warp >= 2) {
    // decode: group g = (warp - 2) / 4 takes the pairs q = g, g + 2, ... (stages 2q, 2q+1);
    // warp w touches TMEM lanes 32*(w%4).. only: rows 32*(w%4)+lane, all 64 inputs
    const int r = (warp & 3) * 32 + lane, grp = (warp - 2) >> 2;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    for (int q = grp; 2 * q < nst && ok; q += 2) {
      const int pq = q % (C::S / 2);
      // the pair's buffers and A slots were last used 4 pairs ago: their MMAs completed
      if (q >= C::S / 2 && !mbar_wait_bounded(&empty[pq], (uint32_t)((q / (C::S / 2)) & 1) ^ 1u, a.status)) {
        ok = false;
        break;
      }
      for (int j = 2 * q; j < 2 * q + 2 && j < nst; ++j) {
        const int s = j % C::S;
        if (!mbar_wait_bounded(&full[s], (uint32_t)(j / C::S) & 1u, a.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint8_t* raw = smem + s * C::STAGE + C::B;
        uint32_t o[32];
        decode_regs<FMT>(raw, r, 0, *reinterpret_cast<uint32_t(*)[16]>(o));
        decode_regs<FMT>(raw, r, 1, *reinterpret_cast<uint32_t(*)[16]>(o + 16));
        tmem_st32(tmem + lane_base + kSmA0 + 32u * (uint32_t)s, o);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0 && ok) mbar_arrive(&afull[pq]);
    }
    // Phase 1 (warps 2-5): this row of the accumulator, scaled by the tensor scale, into the
    // token-major fp32 tile [NB tokens][128 rows].
    const bool go = mbar_wait_bounded(done, 0, a.status);
    float* sF = reinterpret_cast<float*>(smem);
    if (go && warp < 6) {
      tc_fence_after();
#pragma unroll 1
      for (int c = 0; c < NB; c += 16) {
        uint32_t v[16];
        tmem_ld16(tmem + lane_base + (uint32_t)c, v);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 16; ++i) sF[(c + i) * 128 + r] = a.ts * __uint_as_float(v[i]);
      }
    }
  }
  // Every thread of every CTA of the cluster reaches these barriers, after a failed wait too.
  __syncwarp();
  if (ks > 1) cluster_sync_all();
  else __syncthreads();
  if (warp >= 2 && ok) {
    // Phase 2 (warps 2-9): item = (token, group of 8 rows); this CTA takes every ks-th item
    // and sums the ks partial tiles in rank order.
    float* sF = reinterpret_cast<float*>(smem);
    const int e = tid - 64;
    const int64_t nb = (int64_t)tile_n * 128;
    for (int item = rank + ks * e; item < NB * 16; item += ks * 256) {
      const int tok = item >> 4, f8 = (item & 15) * 8;
      const int64_t t = t0 + tok, n = nb + f8;
      if (t >= a.t || n >= a.n) continue;
      float o[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      for (int q = 0; q < ks; ++q) {
        float4 p0, p1;
        if (ks > 1) {
          const uint32_t ad = cluster_map(sF + tok * 128 + f8, (uint32_t)q);
          p0 = ld_cluster_f32x4(ad);
          p1 = ld_cluster_f32x4(ad + 16);
        } else {
          p0 = *reinterpret_cast<const float4*>(sF + tok * 128 + f8);
          p1 = *reinterpret_cast<const float4*>(sF + tok * 128 + f8 + 4);
        }
        o[0] += p0.x; o[1] += p0.y; o[2] += p0.z; o[3] += p0.w;
        o[4] += p1.x; o[5] += p1.y; o[6] += p1.z; o[7] += p1.w;
      }
      if (n + 8 <= a.n) {
        if (a.res) {
          const uint4 rv = *reinterpret_cast<const uint4*>(a.res + t * a.ldr + n);
          const uint32_t rw[4] = {rv.x, rv.y, rv.z, rv.w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            o[2 * i] += __uint_as_float(rw[i] << 16);
            o[2 * i + 1] += __uint_as_float(rw[i] & 0xFFFF0000u);
          }
        }
        uint32_t pk[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const __nv_bfloat162 b2 = __floats2bfloat162_rn(o[2 * i], o[2 * i + 1]);
          pk[i] = *reinterpret_cast<const uint32_t*>(&b2);
        }
        *reinterpret_cast<uint4*>(a.y + t * a.ldy + n) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
      } else {  // the matrix's last rows
        for (int i = 0; i < 8 && n + i < a.n; ++i) {
          float v = o[i];
          if (a.res) v += __bfloat162float(a.res[t * a.ldr + n + i]);
          a.y[t * a.ldy + n + i] = __float2bfloat16_rn(v);
        }
      }
    }
  }
  // the other CTAs of the cluster may still read this CTA's tile
  if (ks > 1) cluster_sync_all();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ---------------------------------------------------------------- host side
namespace {

template <int FMT, int NB>
int launch_small_t(const CUtensorMap& map, const SmallArgs& a, dim3 grid, cudaStream_t s) {
  using C = SmCfg<NB>;
  static std::atomic<unsigned long long> configured{0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return QG_ERR_CUDA;
  const unsigned long long bit = 1ull << (dev & 63);
  if (!(configured.load() & bit)) {
    if (cudaFuncSetAttribute((const void*)gemm_small_kernel<FMT, NB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             C::SMEM) != cudaSuccess)
      return QG_ERR_CUDA;
    configured.fetch_or(bit);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kSmThreads);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  cfg.attrs = attr;
  cfg.numAttrs = 0;
  if (a.ks > 1) {
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = (unsigned)a.ks;
    cfg.numAttrs = 1;
  }
  if (cudaLaunchKernelEx(&cfg, gemm_small_kernel<FMT, NB>, map, a) != cudaSuccess) return QG_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? QG_OK : QG_ERR_CUDA;
}

template <int NB>
int launch_small_nb(int fmt, const CUtensorMap& map, const SmallArgs& a, dim3 grid, cudaStream_t s) {
  switch (fmt) {
    case FMT_MLX: return launch_small_t<FMT_MLX, NB>(map, a, grid, s);
    case FMT_MXFP4: return launch_small_t<FMT_MXFP4, NB>(map, a, grid, s);
    case FMT_NVFP4: return launch_small_t<FMT_NVFP4, NB>(map, a, grid, s);
    case FMT_Q50: return launch_small_t<FMT_Q50, NB>(map, a, grid, s);
    case FMT_Q51: return launch_small_t<FMT_Q51, NB>(map, a, grid, s);
    case FMT_Q5K: return launch_small_t<FMT_Q5K, NB>(map, a, grid, s);
    default: return launch_small_t<FMT_Q6K, NB>(map, a, grid, s);
  }
}

}  // namespace

int launch_gemm_small(const Geometry& g, const qg_weight* w, const void* x, int64_t t, int64_t ldx, const void* res,
                      int64_t ldr, void* y, int64_t ldy, void* ws, const DeviceInfo& dev, void* stream) {
  const int nb = t <= 16 ? 16 : t <= 32 ? 32 : t <= 64 ? 64 : 128;
  const int64_t tt = (t + nb - 1) / nb;
  const int64_t tiles = g.nt * tt;
  // split K over a cluster when the tiles fill less than half of the GPU
  int ks = 1;
  if (tiles * 2 <= dev.sms) ks = (int)std::min<int64_t>(std::min<int64_t>(8, dev.sms / tiles), g.kg);
  if (tt > 65535 || ks < 1) return QG_ERR_UNSUPPORTED;
  CUtensorMap map;
  if (!encode_token_rows(&map, x, t, g.k, ldx, nb)) return QG_ERR_CUDA;
  SmallArgs a;
  a.codes = static_cast<const uint8_t*>(w->codes);
  a.scales = static_cast<const uint8_t*>(w->scales);
  a.aux = static_cast<const uint8_t*>(w->aux);
  a.res = static_cast<const __nv_bfloat16*>(res);
  a.y = static_cast<__nv_bfloat16*>(y);
  a.ldr = ldr;
  a.ldy = ldy;
  a.n = g.n;
  a.t = t;
  a.KG = (int)g.kg;
  a.ks = ks;
  a.ts = (g.fmt == FMT_NVFP4) ? w->tensor_scale : 1.0f;
  a.status = static_cast<int*>(ws);
  const dim3 grid((unsigned)g.nt, (unsigned)tt, (unsigned)ks);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  switch (nb) {
    case 16: return launch_small_nb<16>(g.fmt, map, a, grid, s);
    case 32: return launch_small_nb<32>(g.fmt, map, a, grid, s);
    case 64: return launch_small_nb<64>(g.fmt, map, a, grid, s);
    default: return launch_small_nb<128>(g.fmt, map, a, grid, s);
  }
}

}  // namespace qg
