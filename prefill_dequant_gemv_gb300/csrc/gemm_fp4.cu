// W4A4 GEMM on the block-scaled FP4 tensor cores (TurboEXL3 article §2.2, W4A4: activations
// quantised to NVFP4 on the fly, weights NVFP4, the FP4 x FP4 products on the tensor cores):
//   Y[t, n] = bf16( ts_w * ts_a * sum_k (S_w[n, k/16] E2M1_w[n, k]) (S_a[t, k/16] E2M1_a[t, k])
//                   (+ R[t, n]) )
// with tcgen05.mma kind::mxf4nvf4 (E2M1 operands, one E4M3 scale per 16 inputs of either
// operand, fp32 accumulation in tensor memory).  Nothing is decoded: the packed codes are the
// MMA's operands and the block scales its scale factors.
//
// One CTA computes a 128-row x 256-token output tile over the whole K, in stages of four
// 64-deep K steps:
//   warp 0      producer: per stage, the four packed weight tiles (4 x 4 KB) by one 4-D TMA
//               that lays them out as the tensor cores' no-swizzle K-major operand (the packed
//               tile keeps 8-row x 16-byte core matrices contiguous, 32-row groups apart:
//               the TMA's dimensions (128-byte core matrix, 2 K-halves, 4 row blocks, group)
//               make the row-block stride uniform), the tiles' E4M3 scales (bulk copy), the 256 x 256
//               activation codes (2-D TMA, 128-byte swizzle) and their E4M3 scales (2-D TMA)
//   warps 2..5  write the stage's scale factors into tensor memory (tcgen05.st; each warp its
//               lane quarter, every quarter the same copy: row r's four scales of a K step in
//               lane r % 32, column r / 32, byte = 16-block -- weights in 4 columns per K step,
//               tokens in 8)
//   warp 1      allocates the 512 TMEM columns (accumulator 0-255, scale-factor ring
//               256-447) and issues the block-scaled MMAs (M=128, N=256, K=64) from one lane
//   warps 2..9  epilogue: tensor scales, residual, bf16 once.
// Every wait is bounded (QG_ERR_TIMEOUT in the workspace status word); TMEM is freed on every
// path.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>

#include "qg_common.cuh"
#include "qg_internal.h"
#include "qg_sync.cuh"
#include "qg_tc.cuh"

namespace qg {

namespace {

constexpr int kF4BN = 256;                       // tokens per tile (MMA N)
constexpr int kF4KS = 4;                         // 64-deep K steps per stage
constexpr int kF4Stages = 4;
constexpr int kF4Threads = 320;
constexpr int kF4A = kF4KS * 4096;               // weight codes per stage (no-swizzle layout)
constexpr int kF4B = kF4BN * 128;                // activation codes: 256 tokens x 128 bytes (256 FP4)
constexpr int kF4SA = kF4KS * 512;               // weight scales: 128 rows x 4 per K step
constexpr int kF4SB = kF4BN * 16;                // activation scales: 256 tokens x 16
constexpr int kF4Stage = kF4B + kF4A + kF4SA + kF4SB;  // B first: its 128-byte swizzle wants 1024 alignment
constexpr int kF4Smem = 1024 + kF4Stages * kF4Stage + 256;
constexpr uint32_t kF4SfCols = kF4KS * 4 + kF4KS * (kF4BN / 32);  // 48 TMEM columns per stage
constexpr uint32_t kF4Sf0 = 256;
static_assert(kF4Stage % 1024 == 0, "stage alignment");
static_assert(kF4Smem <= 232448, "shared memory");
static_assert(kF4Sf0 + kF4Stages * kF4SfCols <= 512, "tensor memory");
static_assert(kF4BN * 128 * 4 <= kF4Stages * kF4Stage, "epilogue tile fits in the stage buffers");

// Instruction descriptor, kind::mxf4nvf4: A and B E2M1, K-major, UE4M3 scale factors (scale
// factor ids 0: a K step's four scales fill each 32-bit cell), shape M x N.
constexpr uint32_t idesc_fp4(int M, int N) {
  return (1u << 7)                     // A format: E2M1
         | (1u << 10)                  // B format: E2M1
         | ((uint32_t)(N >> 3) << 17)  // N / 8
         | (0u << 23)                  // scale factor format: UE4M3
         | ((uint32_t)(M >> 4) << 24); // M / 16
}

// No-swizzle K-major shared-memory descriptor: 8-row x 16-byte core matrices, K-adjacent ones
// 128 bytes apart (leading byte offset), row-block-adjacent ones 256 bytes apart (stride byte
// offset).
__device__ __forceinline__ uint64_t noswz_desc(uint32_t addr) {
  uint64_t d = 0;
  d |= (uint64_t)((addr & 0x3FFFFu) >> 4);
  d |= (uint64_t)(128 >> 4) << 16;
  d |= (uint64_t)(256 >> 4) << 32;
  d |= (uint64_t)1 << 46;
  return d;
}

// D[tmem] (+)= (SFA . A[smem]) * (SFB . B[smem])^T with E4M3 scale factors per 16 inputs.
__device__ __forceinline__ void mma_fp4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                        uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
          d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* map, int c3, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5}], "
      "[%6];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(0), "r"(0), "r"(0), "r"(c3), "r"(smem_u32(bar))
      : "memory");
}

struct Fp4Args {
  const uint8_t* scales;  // weight E4M3 scales, packed layout
  const __nv_bfloat16* res;
  __nv_bfloat16* y;
  int64_t ldr, ldy;
  int64_t n, t;
  int KG;
  float ts;  // weight tensor scale x activation tensor scale
  int* status;
};

__global__ void __launch_bounds__(kF4Threads, 1)
    gemm_fp4_kernel(const __grid_constant__ CUtensorMap tmw, const __grid_constant__ CUtensorMap tmx,
                    const __grid_constant__ CUtensorMap tms, const Fp4Args a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kF4Stages * kF4Stage);
  uint64_t* full = bars;                    // stage landed
  uint64_t* sfull = bars + kF4Stages;       // its scale factors are in tensor memory
  uint64_t* empty = bars + 2 * kF4Stages;   // its MMAs completed
  uint64_t* done = bars + 3 * kF4Stages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 3 * kF4Stages + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int tile_n = blockIdx.x;
  const int t0 = blockIdx.y * kF4BN;
  const int KG = a.KG;
  const int nst = (KG + kF4KS - 1) / kF4KS;

  if (tid == 0) {
    for (int s = 0; s < kF4Stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&sfull[s], 4);  // the four scale-factor warps
      mbar_init(&empty[s], 1);
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
      int s = 0;
      uint32_t ph = 0;
      int issued = 0;
      for (int j = 0; j < nst; ++j) {
        if (j >= kF4Stages && !mbar_wait_bounded(&empty[s], ph ^ 1u, a.status)) break;
        uint8_t* st = smem + s * kF4Stage;
        const int kt = j * kF4KS, nk = min(kF4KS, KG - kt);
        const int64_t tile = (int64_t)tile_n * KG + kt;
        mbar_arrive_expect_tx(&full[s], kF4A + nk * 512 + kF4B + kF4SB);
        tma_load_4d(st + kF4B, &tmw, (int)(tile * 4), &full[s]);
        bulk_g2s(st + kF4B + kF4A, a.scales + tile * 512, nk * 512, &full[s]);
        if (j == 0) pdl_wait();  // the quantised activations come from the preceding kernel
        tma_load_2d(st, &tmx, kt * 32, t0, &full[s]);
        tma_load_2d(st + kF4B + kF4A + kF4SA, &tms, kt * 4, t0, &full[s]);
        ++issued;
        if (++s == kF4Stages) {
          s = 0;
          ph ^= 1u;
        }
      }
      // no copies left in flight into this CTA's shared memory
      for (int i = (issued > kF4Stages ? issued - kF4Stages : 0); i < issued; ++i)
        mbar_wait_bounded(&full[i % kF4Stages], (uint32_t)(i / kF4Stages) & 1u, a.status);
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {  // MMA issuer
      constexpr uint32_t idesc = idesc_fp4(128, kF4BN);
      int s = 0;
      uint32_t ph = 0;
      for (int j = 0; j < nst; ++j) {
        if (!mbar_wait_bounded(&sfull[s], ph, a.status)) break;  // scale-factor warps saw the landing
        tc_fence_after();
        const uint32_t stb = smem_u32(smem + s * kF4Stage);
        const uint32_t sf = tmem + kF4Sf0 + (uint32_t)s * kF4SfCols;
        const int nk = min(kF4KS, KG - j * kF4KS);
        for (int kk = 0; kk < nk; ++kk)
          mma_fp4(tmem, noswz_desc(stb + kF4B + 4096u * kk), sw128_desc(stb + 32u * kk), idesc, sf + 4u * kk,
                  sf + kF4KS * 4 + (kF4BN / 32) * kk, (j | kk) ? 1u : 0u);
        mma_commit(&empty[s]);
        if (++s == kF4Stages) {
          s = 0;
          ph ^= 1u;
        }
      }
      mma_commit(done);
    }
    __syncwarp();
  }
  bool go = false;
  float* sF = reinterpret_cast<float*>(smem);  // epilogue tile [256 tokens][128 rows] in the stage buffers
  if (warp >= 2) {
    bool ok = true;
    if (warp < 6) {
      // scale factors of each stage into tensor memory, this warp's lane quarter
      const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
      for (int j = 0; j < nst; ++j) {
        const int s = j % kF4Stages;
        if (!mbar_wait_bounded(&full[s], (uint32_t)(j / kF4Stages) & 1u, a.status)) {
          ok = false;
          break;
        }
        // slot s's previous scale factors were read by MMAs that completed before the producer
        // refilled the stage (empty -> producer -> full): order these writes after them
        tc_fence_after();
        const uint8_t* st = smem + s * kF4Stage;
        const uint8_t* sa = st + kF4B + kF4A;
        const uint8_t* sb = sa + kF4SA;
        uint32_t va[kF4KS * 4], vb[kF4KS * (kF4BN / 32)];
#pragma unroll
        for (int kk = 0; kk < kF4KS; ++kk)
#pragma unroll
          for (int c = 0; c < 4; ++c)  // weight row lane + 32 c, K step kk
            va[kk * 4 + c] = *reinterpret_cast<const uint32_t*>(sa + kk * 512 + (lane + 32 * c) * 4);
#pragma unroll
        for (int c = 0; c < kF4BN / 32; ++c) {  // token lane + 32 c, all four K steps
          const uint4 v = *reinterpret_cast<const uint4*>(sb + (lane + 32 * c) * 16);
          vb[0 * (kF4BN / 32) + c] = v.x;
          vb[1 * (kF4BN / 32) + c] = v.y;
          vb[2 * (kF4BN / 32) + c] = v.z;
          vb[3 * (kF4BN / 32) + c] = v.w;
        }
        const uint32_t sf = tmem + lane_base + kF4Sf0 + (uint32_t)s * kF4SfCols;
        tmem_st16(sf, va);
        tmem_st32(sf + kF4KS * 4, vb);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sfull[s]);
      }
    }
    // Epilogue, two phases over the idle stage buffers (as the bf16 prefill GEMM): phase 1,
    // each thread scales its TMEM row into a token-major fp32 tile; phase 2 (after the CTA
    // barrier) each thread takes 8 consecutive rows of one token, adds the residual, rounds to
    // bf16 once and writes 16 bytes.
    go = mbar_wait_bounded(done, 0, a.status) && ok;
    if (go) {
      tc_fence_after();
      const int quarter = warp & 3;
      const int col0 = ((warp - 2) >> 2) * (kF4BN / 2);
      const int row = quarter * 32 + lane;
      for (int c = 0; c < kF4BN / 2; c += 32) {
        uint32_t v[32];
        tmem_ld32(tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(col0 + c), v);
        tmem_ld_wait();
#pragma unroll
        for (int q = 0; q < 32; ++q) sF[(col0 + c + q) * 128 + row] = a.ts * __uint_as_float(v[q]);
      }
    }
  }
  __syncwarp();
  __syncthreads();
  if (go) {
    pdl_wait();  // the residual may come from the preceding kernel, which may also read y
    const int e = tid - 64;  // 0..255
    const int64_t nb = (int64_t)tile_n * 128;
    for (int item = e; item < kF4BN * 16; item += 8 * 32) {
      const int tok = item >> 4, f8 = (item & 15) * 8;
      const int64_t t = t0 + tok, n = nb + f8;
      if (t >= a.t || n >= a.n) continue;
      const float4 p0 = *reinterpret_cast<const float4*>(sF + tok * 128 + f8);
      const float4 p1 = *reinterpret_cast<const float4*>(sF + tok * 128 + f8 + 4);
      float o[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
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
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                              const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                              CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

}  // namespace

int launch_gemm_fp4(const Geometry& g, const qg_weight* w, float act_scale, const uint8_t* xcodes, int64_t ldc,
                    const uint8_t* xscales, int64_t lds, int64_t t, const void* res, int64_t ldr, void* y, int64_t ldy,
                    void* ws, void* stream) {
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult qr;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &qr) != cudaSuccess ||
      qr != cudaDriverEntryPointSuccess || !fn)
    return QG_ERR_CUDA;
  EncodeFn enc = reinterpret_cast<EncodeFn>(fn);
  const cuuint32_t e1[5] = {1, 1, 1, 1, 1};
  // weight codes: (one 8-row x 16-byte core matrix = 128 contiguous bytes, 2 K halves, 4 row
  // blocks, 32-row group over all tiles)
  CUtensorMap tmw, tmx, tms;
  {
    const cuuint64_t dims[4] = {128, 2, 4, (cuuint64_t)(g.nt * g.kg * 4)};
    const cuuint64_t strides[3] = {512, 128, 1024};
    const cuuint32_t box[4] = {128, 2, 4, (cuuint32_t)(kF4KS * 4)};
    if (enc(&tmw, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(w->codes), dims, strides, box, e1,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return QG_ERR_CUDA;
  }
  {  // activation codes: k / 2 bytes per token row
    const cuuint64_t dims[2] = {(cuuint64_t)(g.k / 2), (cuuint64_t)t};
    const cuuint64_t strides[1] = {(cuuint64_t)ldc};
    const cuuint32_t box[2] = {128, (cuuint32_t)kF4BN};
    if (enc(&tmx, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(xcodes), dims, strides, box, e1,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return QG_ERR_CUDA;
  }
  {  // activation scales: k / 16 bytes per token row
    const cuuint64_t dims[2] = {(cuuint64_t)(g.k / 16), (cuuint64_t)t};
    const cuuint64_t strides[1] = {(cuuint64_t)lds};
    const cuuint32_t box[2] = {16, (cuuint32_t)kF4BN};
    if (enc(&tms, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(xscales), dims, strides, box, e1,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return QG_ERR_CUDA;
  }
  Fp4Args a;
  a.scales = static_cast<const uint8_t*>(w->scales);
  a.res = static_cast<const __nv_bfloat16*>(res);
  a.y = static_cast<__nv_bfloat16*>(y);
  a.ldr = ldr;
  a.ldy = ldy;
  a.n = g.n;
  a.t = t;
  a.KG = (int)g.kg;
  a.ts = w->tensor_scale * act_scale;
  a.status = static_cast<int*>(ws);
  const int64_t tt = (t + kF4BN - 1) / kF4BN;
  if (tt > 65535 || g.nt > 0x7FFFFFFF) return QG_ERR_UNSUPPORTED;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return QG_ERR_CUDA;
  static std::atomic<unsigned long long> configured{0};
  const unsigned long long bit = 1ull << (dev & 63);
  if (!(configured.load() & bit)) {
    if (cudaFuncSetAttribute(gemm_fp4_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kF4Smem) != cudaSuccess)
      return QG_ERR_CUDA;
    configured.fetch_or(bit);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)g.nt, (unsigned)tt, 1);
  cfg.blockDim = dim3(kF4Threads);
  cfg.dynamicSmemBytes = kF4Smem;
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, gemm_fp4_kernel, tmw, tmx, tms, a) != cudaSuccess) return QG_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? QG_OK : QG_ERR_CUDA;
}

}  // namespace qg
