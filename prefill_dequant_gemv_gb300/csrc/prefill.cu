// Prefill GEMM on GB300 tensor cores: Y[t, n] = bf16( sum_k W[n, k] X[t, k] (+ R[t, n]) )
// for quantized W and bf16 X with many tokens (TurboEXL3 article §4.1, "decode once,
// multiply many times": each 64-deep slice of the weights is decoded once into on-chip
// memory and multiplied against up to 256 tokens; the decoded weights never reach device
// memory and no 16-bit copy is written).
//
// One CTA computes a 128-row x 256-token output tile over the whole K:
//   warp 0      producer: per 64-deep stage, bulk-copies the packed weight tile (codes,
//               scales, Q6_K d) and TMA-loads the 256 x 64 activation tile (128-byte swizzle)
//   warps 2..9  decode the stage's 128 x 64 weights to bf16 (E2M1 x block scale is exact in
//               bf16) straight into tensor memory (tcgen05.st: row r -> TMEM lane r), the
//               MMA's A operand, then run the epilogue (TMEM -> registers -> bf16 output,
//               tensor scale and residual)
//   warp 1      allocates all 512 TMEM columns (accumulator 0-255, A ring 256-415) and
//               issues tcgen05.mma (M=128, N=256, K=16, A from TMEM, B from shared memory,
//               fp32 accumulate) from one lane; completion is committed to mbarriers.
// With A in tensor memory the decoded weights cost no shared-memory bandwidth; one
// accumulator chain at N = 256 can keep the tensor pipe full when the issuing thread has its
// operands ready (its MMA descriptors are prepared outside the issue).
// Every wait is bounded (QG_ERR_TIMEOUT in the workspace status word) and TMEM is freed
// on every path.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <mutex>

#include "qg_common.cuh"
#include "qg_decode_tile.cuh"
#include "qg_internal.h"
#include "qg_sync.cuh"
#include "qg_tc.cuh"

namespace qg {

constexpr int kPfBN = 256;                                   // tokens per tile (MMA N)
constexpr int kPfStages = 5;
constexpr int kPfDeqWarps = 8;                               // epilogue warps (and Q6_K decoders)
__host__ __device__ constexpr int pf_decoders(int fmt) { return fmt == FMT_Q6K || fmt_q5(fmt) ? 8 : 4; }
constexpr int kPfThreads = (2 + kPfDeqWarps) * 32;           // 320
constexpr int kBTile = kPfBN * 128;                          // 256 tokens x 64 bf16
constexpr int kRawMax = 7168;                                // >= Q6_K tile 6144 + 512 + 256
constexpr int kPfStageBytes = kBTile + kRawMax;              // 39936, a multiple of 1024
constexpr int kPfSmem = 1024 + kPfStages * kPfStageBytes + 256;
constexpr uint32_t kPfTmemCols = 512;
constexpr uint32_t kPfA0 = 256;                              // A stage s at columns 256 + 32 s
static_assert(kPfA0 + 32 * kPfStages <= kPfTmemCols, "tensor memory");
static_assert(kPfBN * 128 * 4 <= kPfStages * kPfStageBytes, "epilogue tile fits in the stage buffers");

struct PrefillArgs {
  const uint8_t* codes;
  const uint8_t* scales;
  const uint8_t* aux;
  const __nv_bfloat16* res;
  __nv_bfloat16* y;
  int64_t ldr, ldy;
  int64_t n, t;
  int KG;
  float ts;
  int ks;  // CTAs per cluster splitting K (1: no split)
  int* status;
};

__device__ __forceinline__ float4 ld_cluster_f32x4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0,%1,%2,%3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr) : "memory");
  return v;
}

template <int FMT>
__global__ void __launch_bounds__(kPfThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tmx, const PrefillArgs a) {
  using F = Fmt<FMT>;
  constexpr int kRaw = F::TB + 128 * F::SB + fmt_aux(FMT);  // tile, scales, aux of its 256 inputs
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kPfStages * kPfStageBytes);
  uint64_t* full = bars;
  uint64_t* afull = bars + kPfStages;
  uint64_t* empty = bars + 2 * kPfStages;
  uint64_t* done = bars + 3 * kPfStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 3 * kPfStages + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int tile_n = blockIdx.x;
  const int t0 = blockIdx.y * kPfBN;
  const int KG = a.KG;
  // split K: this CTA's 64-deep stages [kt0, kt1) (the host keeps ks <= KG)
  const int ks = a.ks;
  const int rank = ks > 1 ? (int)cluster_rank() : 0;
  const int kt0 = (int)((int64_t)rank * KG / ks), kt1 = (int)((int64_t)(rank + 1) * KG / ks);
  const int nst = kt1 - kt0;

  if (tid == 0) {
    for (int s = 0; s < kPfStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&afull[s], 4);  // the four decode warps of the stage's group
      mbar_init(&empty[s], 1);
    }
    mbar_init(done, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kPfTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {  // producer
      int s = 0;
      uint32_t ph = 0;
      int issued = 0;
      for (int kt = kt0; kt < kt1; ++kt) {
        if (kt - kt0 >= kPfStages && !mbar_wait_bounded(&empty[s], ph ^ 1u, a.status)) break;
        uint8_t* st = smem + s * kPfStageBytes;
        const int64_t tile = (int64_t)tile_n * KG + kt;
        mbar_arrive_expect_tx(&full[s], kRaw + kBTile);
        bulk_g2s(st + kBTile, a.codes + tile * F::TB, F::TB, &full[s]);
        bulk_g2s(st + kBTile + F::TB, a.scales + tile * (128 * F::SB), 128 * F::SB, &full[s]);
        if (fmt_aux(FMT))
          bulk_g2s(st + kBTile + F::TB + 128 * F::SB,
                   a.aux + ((int64_t)tile_n * (KG / 4) + kt / 4) * fmt_aux(FMT), fmt_aux(FMT), &full[s]);
        tma_load_2d(st, &tmx, kt * 64, t0, &full[s]);
        ++issued;
        if (++s == kPfStages) {
          s = 0;
          ph ^= 1u;
        }
      }
      // do not leave copies in flight into this CTA's shared memory
      for (int i = (issued > kPfStages ? issued - kPfStages : 0); i < issued; ++i)
        mbar_wait_bounded(&full[i % kPfStages], (uint32_t)(i / kPfStages) & 1u, a.status);
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {  // MMA issuer
      constexpr uint32_t idesc = idesc_bf16_f32(128, kPfBN);
      const uint32_t lo0 = sw128_desc_lo(smem_u32(smem));  // stage s: lo0 + s * kPfStageBytes / 16
      int s = 0;
      uint32_t ph = 0;
      // the decoders waited for the stage's landing before arriving on afull, so this one
      // wait covers both operands; the MMAs' operands are prepared outside the issue
      for (int kt = kt0; kt < kt1; ++kt) {
        if (!mbar_wait_bounded(&afull[s], ph, a.status)) break;
        tc_fence_after();
        const uint32_t ta = tmem + kPfA0 + 32u * (uint32_t)s;
        const uint32_t lo = lo0 + (uint32_t)s * (uint32_t)(kPfStageBytes / 16);
        if (kt == kt0) mma_bf16_ts_fast<false>(tmem, ta, lo, idesc);
        else mma_bf16_ts_fast<true>(tmem, ta, lo, idesc);
#pragma unroll
        for (int kk = 1; kk < 4; ++kk) mma_bf16_ts_fast<true>(tmem, ta + 8u * kk, lo + 2u * kk, idesc);
        mma_commit(&empty[s]);
        if (++s == kPfStages) {
          s = 0;
          ph ^= 1u;
        }
      }
      mma_commit(done);  // also drains whatever was issued if the loop stopped early
    }
    __syncwarp();
  }
  bool go = false;  // decode warps: every wait succeeded and the accumulator is complete
  float* sF = reinterpret_cast<float*>(smem);  // epilogue tile, 128 KB inside stages 0..3
  if (warp >= 2) {
    // decode warps: warp w may only touch TMEM lanes 32*(w%4)..; it decodes rows
    // 32*(w%4)+lane, all 64 inputs of a stage, stored with one 32-column tensor-memory write
    // (fewer, wider writes contend less with the MMAs).  4-bit formats: warps 2-5 take every
    // stage; Q6_K (heavier extraction): warps 2-5 the even stages, warps 6-9 the odd ones.
    constexpr int kGroups = pf_decoders(FMT) / 4;
    const int r = (warp & 3) * 32 + lane, grp = (warp - 2) >> 2;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    bool ok = true;
    for (int j = grp < kGroups ? grp : nst; j < nst; j += kGroups) {
      const int s = j % kPfStages;
      const uint32_t ph = (uint32_t)(j / kPfStages) & 1u;
      if (!mbar_wait_bounded(&full[s], ph, a.status)) {
        ok = false;
        break;
      }
      // slot s's previous A was read by MMAs that completed before the producer refilled the
      // slot (empty -> producer -> full): order this thread's TMEM writes after them
      tc_fence_after();
      uint8_t* st = smem + s * kPfStageBytes;
      uint32_t o[32];
      decode_regs<FMT>(st + kBTile, r, 0, *reinterpret_cast<uint32_t(*)[16]>(o));
      decode_regs<FMT>(st + kBTile, r, 1, *reinterpret_cast<uint32_t(*)[16]>(o + 16));
      tmem_st32(tmem + lane_base + kPfA0 + 32u * (uint32_t)s, o);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&afull[s]);
    }
    // Epilogue, two phases over the (now idle) stage buffers.  Phase 1: TMEM lanes
    // 32*(warp%4).. hold output rows; warps 2-5 take tokens 0..127, warps 6-9 tokens
    // 128..255; each thread scales its row's accumulators by the tensor scale into a
    // token-major fp32 tile [256 tokens][128 rows] (a warp writes 128 contiguous bytes per
    // token).  Phase 2 (below, after a barrier of the CTA or, with K split, of the cluster):
    // each thread takes 8 consecutive rows of one token -- sums the K-split partial tiles in
    // rank order, adds the residual, rounds to bf16 once and writes 16 bytes.  The barriers
    // are reached by every thread, also after a failed wait.
    go = mbar_wait_bounded(done, 0, a.status) && ok;
    if (go) {
      tc_fence_after();
      const int quarter = warp & 3;
      const int col0 = ((warp - 2) >> 2) * (kPfBN / 2);
      const int row = quarter * 32 + lane;
      for (int c = 0; c < kPfBN / 2; c += 32) {
        uint32_t v[32];
        tmem_ld32(tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(col0 + c), v);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 32; ++j) sF[(col0 + c + j) * 128 + row] = a.ts * __uint_as_float(v[j]);
      }
    }
  }
  __syncwarp();
  if (ks > 1) cluster_sync_all();
  else __syncthreads();
  if (go) {
    const int e = tid - 64;  // 0..255
    const int64_t nb = (int64_t)tile_n * 128;
    for (int item = rank + ks * e; item < kPfBN * 16; item += ks * kPfDeqWarps * 32) {
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
          for (int q = 0; q < 4; ++q) {
            o[2 * q] += __uint_as_float(rw[q] << 16);
            o[2 * q + 1] += __uint_as_float(rw[q] & 0xFFFF0000u);
          }
        }
        uint32_t pk[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const __nv_bfloat162 b2 = __floats2bfloat162_rn(o[2 * q], o[2 * q + 1]);
          pk[q] = *reinterpret_cast<const uint32_t*>(&b2);
        }
        *reinterpret_cast<uint4*>(a.y + t * a.ldy + n) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
      } else {  // the matrix's last rows
        for (int q = 0; q < 8 && n + q < a.n; ++q) {
          float v = o[q];
          if (a.res) v += __bfloat162float(a.res[t * a.ldr + n + q]);
          a.y[t * a.ldy + n + q] = __float2bfloat16_rn(v);
        }
      }
    }
  }
  // with K split, the other CTAs of the cluster may still read this CTA's tile
  __syncwarp();
  if (ks > 1) cluster_sync_all();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kPfTmemCols);
  }
}

// ---------------------------------------------------------------- host side
namespace {
using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                              const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                              CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
std::once_flag g_encode_once;
EncodeFn g_encode = nullptr;

EncodeFn encode_fn() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<EncodeFn>(fn);
  });
  return g_encode;
}
}  // namespace

bool encode_token_rows(CUtensorMap* map, const void* x, int64_t rows, int64_t k, int64_t ldx, int box_rows) {
  EncodeFn enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)k, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)ldx * 2};
  const cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(x), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int launch_prefill(const Geometry& g, const qg_weight* w, const void* x, int64_t t, int64_t ldx, const void* res,
                   int64_t ldr, void* y, int64_t ldy, void* ws, void* stream) {
  EncodeFn enc = encode_fn();
  if (!enc) return QG_ERR_CUDA;
  CUtensorMap map;
  const cuuint64_t dims[2] = {(cuuint64_t)g.k, (cuuint64_t)t};
  const cuuint64_t strides[1] = {(cuuint64_t)ldx * 2};
  const cuuint32_t box[2] = {64, (cuuint32_t)kPfBN};
  const cuuint32_t estr[2] = {1, 1};
  if (enc(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(x), dims, strides, box, estr,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return QG_ERR_CUDA;
  PrefillArgs a;
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
  a.ts = (g.fmt == FMT_NVFP4) ? w->tensor_scale : 1.0f;
  a.status = static_cast<int*>(ws);
  DeviceInfo info;
  int devid = 0;
  if (cudaGetDevice(&devid) != cudaSuccess || !device_info(devid, &info)) return QG_ERR_CUDA;
  const int64_t tt = (t + kPfBN - 1) / kPfBN;
  if (tt > 65535) return QG_ERR_UNSUPPORTED;
  // split K over a cluster of up to 8 CTAs when the output tiles fill less than half the GPU
  a.ks = 1;
  if (g.nt * tt * 2 <= info.sms) a.ks = (int)std::min<int64_t>(std::min<int64_t>(8, info.sms / (g.nt * tt)), g.kg);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  static std::atomic<unsigned long long> configured[8];
  const unsigned long long bit = 1ull << (devid & 63);
  const void* fn = nullptr;
  switch (g.fmt) {
    case FMT_MLX: fn = (const void*)prefill_kernel<FMT_MLX>; break;
    case FMT_MXFP4: fn = (const void*)prefill_kernel<FMT_MXFP4>; break;
    case FMT_NVFP4: fn = (const void*)prefill_kernel<FMT_NVFP4>; break;
    case FMT_Q50: fn = (const void*)prefill_kernel<FMT_Q50>; break;
    case FMT_Q51: fn = (const void*)prefill_kernel<FMT_Q51>; break;
    case FMT_Q5K: fn = (const void*)prefill_kernel<FMT_Q5K>; break;
    default: fn = (const void*)prefill_kernel<FMT_Q6K>; break;
  }
  if (!(configured[g.fmt].load() & bit)) {
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kPfSmem) != cudaSuccess)
      return QG_ERR_CUDA;
    configured[g.fmt].fetch_or(bit);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)g.nt, (unsigned)tt, (unsigned)a.ks);
  cfg.blockDim = dim3(kPfThreads);
  cfg.dynamicSmemBytes = kPfSmem;
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
  cudaError_t e;
  switch (g.fmt) {
    case FMT_MLX: e = cudaLaunchKernelEx(&cfg, prefill_kernel<FMT_MLX>, map, a); break;
    case FMT_MXFP4: e = cudaLaunchKernelEx(&cfg, prefill_kernel<FMT_MXFP4>, map, a); break;
    case FMT_NVFP4: e = cudaLaunchKernelEx(&cfg, prefill_kernel<FMT_NVFP4>, map, a); break;
    case FMT_Q50: e = cudaLaunchKernelEx(&cfg, prefill_kernel<FMT_Q50>, map, a); break;
    case FMT_Q51: e = cudaLaunchKernelEx(&cfg, prefill_kernel<FMT_Q51>, map, a); break;
    case FMT_Q5K: e = cudaLaunchKernelEx(&cfg, prefill_kernel<FMT_Q5K>, map, a); break;
    default: e = cudaLaunchKernelEx(&cfg, prefill_kernel<FMT_Q6K>, map, a); break;
  }
  if (e != cudaSuccess) return QG_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? QG_OK : QG_ERR_CUDA;
}

}  // namespace qg
