// Mixture-of-experts layer for many tokens (TurboEXL3 article §4.1, "Prefill: decode once,
// multiply many times"): after the route (route.cu) groups every (token, expert) pair by
// expert and cuts each expert's run into tiles of at most 192 pairs,
//
//   gate/up  one grouped tensor-core GEMM over the tile table: each work item is (tile,
//            128 features); it decodes the expert's gate rows f.. and up rows F+f.. of every
//            64-deep stage once into tensor memory, multiplies both by the tile's tokens
//            gathered straight from x (no grouped copy of x is written), and its epilogue
//            runs the mid step -- h = bf16(silu(gate) * up) in fp32 (§4.1 "Mid") -- so the
//            gate/up outputs never reach device memory
//   down     the same GEMM body on h (rows already in grouped order), fp32 outputs per pair
//   finish   out[t] = bf16( sum_j p[t, j] * down[pos(t, j)] + shared[t] ) (§4.1 "Finish")
//
// The shared expert runs as extra tiles of both GEMMs (every token, in 192-token tiles).
// Tile widths are ragged: the MMA's N is the tile's pair count rounded up to 16, so an
// expert with 160 tokens costs 160 columns, not 192.
//
// The GEMM is persistent (one CTA per SM walks the work items) and warp-specialised:
//   warp 0       raw-weight producer: bulk copies of the packed tiles into a deep ring
//   warp 1       TMEM allocation and the tcgen05.mma issuer (one lane)
//   warps 2-9    decode a stage's tiles into the bf16 A operand ring in tensor memory
//                (tcgen05.st), so the decoded weights cost no shared-memory bandwidth
//   warps 10-17  epilogue: TMEM -> registers -> h (bf16) or per-pair outputs (fp32)
//   warps 18-21  gather: cp.async of the tile's activation rows, by row index, into the
//                128-byte swizzled operand ring; each thread's copies arrive on the
//                stage's mbarrier when they land, and the MMA thread fences the generic
//                proxy writes before the tensor cores read them
// The three rings (raw, decoded A, gathered B) have their own full/empty mbarriers, so HBM
// latency on the weights, L2 latency on the gathers and the decode overlap one another and
// the tensor cores.  The down GEMM double-buffers its accumulator in TMEM so an item's
// epilogue overlaps the next item's main loop.  Every wait is bounded (QG_ERR_TIMEOUT in
// the workspace status word) and TMEM is freed on every path.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>

#include "qg_common.cuh"
#include "qg_decode_tile.cuh"
#include "qg_internal.h"
#include "qg_route.h"
#include "qg_sync.cuh"
#include "qg_tc.cuh"

namespace qg {

constexpr int kMpDecWarps = 8;  // two per TMEM lane quarter, one per half of a stage's 64 inputs
constexpr int kMpEpiWarps = 8;  // two per TMEM lane quarter, alternate 16-column chunks
constexpr int kMpGatWarps = 4;
constexpr int kMpGatThreads = kMpGatWarps * 32;
constexpr int kMpWarps = 2 + kMpDecWarps + kMpEpiWarps + kMpGatWarps;  // 22
constexpr int kMpThreads = kMpWarps * 32;                               // 704
constexpr int kMpEpiWarp0 = 2 + kMpDecWarps;                            // 10
constexpr int kMpGatWarp0 = kMpEpiWarp0 + kMpEpiWarps;                  // 18
constexpr int kMpTile = kRouteTile;  // pairs per tile = largest MMA N
constexpr int kMpSmemCap = 232448;   // opt-in shared memory per block on sm_100-family GPUs

// Tensor memory (512 columns x 128 lanes of 32 bits) holds the accumulators and the decoded
// weight operand A:
//   gate/up: gate accumulator [0, 192), up accumulator [192, 384), A ring of 2 stages x 64
//            columns (gate rows' 64 inputs in 32 columns, then the up rows')
//   down:    two accumulators [0, 192) and [192, 384), A ring of 4 stages x 32 columns
// so shared memory holds only the raw packed tiles and the gathered activation rows.
template <int FMT, bool DUAL>
struct MpCfg {
  using F = Fmt<FMT>;
  static constexpr int RAW1 = F::TB + 128 * F::SB + (FMT == FMT_Q6K ? 256 : 0);  // one packed tile
  static constexpr int RAWB = (DUAL ? 2 : 1) * RAW1;
  static constexpr int B = kMpTile * 128;      // gathered rows, 128-byte swizzled
  static constexpr int BS = 6;
  static constexpr int ACC = DUAL ? 1 : 2;      // accumulator buffers
  static constexpr uint32_t ACC_COLS = DUAL ? 2 * kMpTile : kMpTile;
  static constexpr int AS = DUAL ? 2 : 4;       // A stages in TMEM
  static constexpr uint32_t A_COLS = DUAL ? 64 : 32;
  static constexpr uint32_t A0 = 2 * kMpTile;  // first A column
  static_assert(A0 + AS * A_COLS <= 512, "tensor memory");
  static constexpr int FIT = (kMpSmemCap - 1024 - 512 - BS * B) / RAWB;
  static constexpr int RS = FIT > 16 ? 16 : FIT;
  static constexpr int OFF_RAW = BS * B;
  static constexpr int OFF_BAR = OFF_RAW + RS * RAWB;
  static constexpr int NBAR = 2 * RS + 2 * AS + 2 * BS + 2 * 2 + 1;
  static constexpr int SMEM = 1024 + OFF_BAR + NBAR * 8 + 16;
  static_assert(RS >= 4, "raw ring too shallow");
  static_assert(SMEM <= kMpSmemCap, "shared memory");
};

struct MpArgs {
  const uint8_t* codes;  // routed experts, concatenated (stride per expert below)
  const uint8_t* scales;
  const uint8_t* aux;
  int64_t cstride, sstride, astride;
  const uint8_t* sh_codes;  // shared expert (used when n_sh_tiles > 0)
  const uint8_t* sh_scales;
  const uint8_t* sh_aux;
  float ts, sh_ts;
  const __nv_bfloat16* in;  // gate/up: x [T][ldi]; down: h [R][ldi]
  int64_t ldi;
  int64_t K;
  int KG;
  void* out;  // gate/up: h bf16 [R][ldo]; down: d fp32 [R][ldo]
  int64_t ldo;
  int64_t n_out;  // features of the output (F for gate/up, H for down)
  int QN;         // 128-feature blocks per tile (gate/up: F/128; down: ceil(H/128))
  int T, topk, n_sh_tiles;
  const int* meta;
  const int* tiles;
  const int* pair_list;
  int* status;
};

struct MpItem {
  const uint8_t* codes;
  const uint8_t* scales;
  const uint8_t* aux;
  const int* in_list;  // routed gate/up: grouped position -> pair; row = pair / topk
  float ts;
  int q, count, in_base, out_base;
};

template <bool DUAL>
__device__ __forceinline__ MpItem mp_item(const MpArgs& a, int n_rt, int i) {
  MpItem it;
  const int ti = i / a.QN;
  it.q = i - ti * a.QN;
  if (ti < n_rt) {
    const int e = a.tiles[3 * ti], first = a.tiles[3 * ti + 1];
    it.count = a.tiles[3 * ti + 2];
    it.codes = a.codes + (int64_t)e * a.cstride;
    it.scales = a.scales + (int64_t)e * a.sstride;
    it.aux = a.aux ? a.aux + (int64_t)e * a.astride : nullptr;
    it.ts = a.ts;
    it.out_base = first;
    it.in_list = DUAL ? a.pair_list + first : nullptr;
    it.in_base = first;
  } else {
    const int t0 = (ti - n_rt) * kMpTile;
    it.count = min(kMpTile, a.T - t0);
    it.codes = a.sh_codes;
    it.scales = a.sh_scales;
    it.aux = a.sh_aux;
    it.ts = a.sh_ts;
    it.out_base = a.T * a.topk + t0;
    it.in_list = nullptr;
    it.in_base = DUAL ? t0 : a.T * a.topk + t0;
  }
  return it;
}

template <int FMT>
__device__ __forceinline__ void mp_load_tile(uint8_t* dst, const MpItem& it, int row_tile, int KG, int kt,
                                             uint64_t* bar) {
  using F = Fmt<FMT>;
  const int64_t tile = (int64_t)row_tile * KG + kt;
  bulk_g2s(dst, it.codes + tile * F::TB, F::TB, bar);
  bulk_g2s(dst + F::TB, it.scales + tile * (128 * F::SB), 128 * F::SB, bar);
  if (FMT == FMT_Q6K)
    bulk_g2s(dst + F::TB + 128 * F::SB, it.aux + ((int64_t)row_tile * (KG / 4) + kt / 4) * 256, 256, bar);
}

template <int FMT, bool DUAL>
__global__ void __launch_bounds__(kMpThreads, 1) moe_gemm_kernel(const MpArgs a) {
  using C = MpCfg<FMT, DUAL>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sB = smem;
  uint8_t* sR = smem + C::OFF_RAW;
  uint64_t* r_full = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* r_empty = r_full + C::RS;
  uint64_t* a_full = r_empty + C::RS;
  uint64_t* a_empty = a_full + C::AS;
  uint64_t* b_full = a_empty + C::AS;
  uint64_t* b_empty = b_full + C::BS;
  uint64_t* t_full = b_empty + C::BS;
  uint64_t* t_empty = t_full + 2;
  uint64_t* fin = t_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(fin + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n_rt = a.meta[1];
  const int n_items = (n_rt + a.n_sh_tiles) * a.QN;
  const int G = gridDim.x, b = blockIdx.x;
  const int KG = a.KG;

  if (tid == 0) {
    for (int s = 0; s < C::RS; ++s) {
      mbar_init(&r_full[s], 1);
      mbar_init(&r_empty[s], kMpDecWarps);
    }
    for (int s = 0; s < C::AS; ++s) {
      mbar_init(&a_full[s], kMpDecWarps);
      mbar_init(&a_empty[s], 1);
    }
    for (int s = 0; s < C::BS; ++s) {
      mbar_init(&b_full[s], kMpGatThreads);  // one cp.async completion arrival per gather thread
      mbar_init(&b_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&t_full[s], 1);
      mbar_init(&t_empty[s], kMpEpiWarps);
    }
    mbar_init(fin, 1);
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
    // ------------------------------------------------------------ raw-weight producer
    if (lane == 0) {
      uint32_t gs = 0;
      bool ok = true;
      for (int i = b; ok && i < n_items; i += G) {
        const MpItem it = mp_item<DUAL>(a, n_rt, i);
        for (int kt = 0; kt < KG; ++kt, ++gs) {
          const uint32_t s = gs % C::RS;
          if (gs >= (uint32_t)C::RS && !mbar_wait_bounded(&r_empty[s], ((gs / C::RS) & 1u) ^ 1u, a.status)) {
            ok = false;
            break;
          }
          uint8_t* dst = sR + s * C::RAWB;
          mbar_arrive_expect_tx(&r_full[s], C::RAWB);
          mp_load_tile<FMT>(dst, it, it.q, KG, kt, &r_full[s]);
          if (DUAL) mp_load_tile<FMT>(dst + C::RAW1, it, it.q + a.QN, KG, kt, &r_full[s]);
        }
      }
      // leave no copy in flight into this CTA's shared memory
      for (uint32_t g2 = gs > (uint32_t)C::RS ? gs - C::RS : 0; g2 < gs; ++g2)
        mbar_wait_bounded(&r_full[g2 % C::RS], (g2 / C::RS) & 1u, a.status);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      uint32_t gs = 0, itc = 0;
      bool ok = true;
      for (int i = b; ok && i < n_items; i += G, ++itc) {
        const MpItem it = mp_item<DUAL>(a, n_rt, i);
        const int N = (it.count + 15) & ~15;
        const uint32_t idesc = idesc_bf16_f32(128, N);
        const uint32_t acc = DUAL ? 0u : (itc & 1u);
        if (itc >= (uint32_t)C::ACC &&
            !mbar_wait_bounded(&t_empty[acc], ((itc / C::ACC) & 1u) ^ 1u, a.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d0 = tmem + acc * C::ACC_COLS;
        for (int kt = 0; kt < KG; ++kt, ++gs) {
          const uint32_t sa = gs % C::AS, sb = gs % C::BS;
          if (!mbar_wait_bounded(&a_full[sa], (gs / C::AS) & 1u, a.status) ||
              !mbar_wait_bounded(&b_full[sb], (gs / C::BS) & 1u, a.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          // the gathered rows were written by cp.async (generic proxy); order them before
          // the tensor cores' (async proxy) reads of this stage
          fence_proxy_async_smem();
          const uint32_t ta = tmem + C::A0 + sa * C::A_COLS;
          const uint32_t bbase = smem_u32(sB + sb * C::B);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint32_t accum = (kt | kk) ? 1u : 0u;
            const uint64_t bd = sw128_desc(bbase + kk * 32);
            mma_bf16_ts(d0, ta + kk * 8, bd, idesc, accum);
            if (DUAL) mma_bf16_ts(tmem + kMpTile, ta + 32 + kk * 8, bd, idesc, accum);
          }
          mma_commit(&a_empty[sa]);
          mma_commit(&b_empty[sb]);
        }
        if (!ok) break;
        mma_commit(&t_full[acc]);
      }
      mma_commit(fin);  // every MMA issued so far is complete when this arrives
      mbar_wait_bounded(fin, 0, a.status);
    }
    __syncwarp();
  } else if (warp < kMpEpiWarp0) {
    // ------------------------------------------------------------ decode
    // Warp w may only touch TMEM lanes 32*(w%4)..: it decodes rows 32*(w%4)+lane, inputs
    // 32h..32h+31 of each 64-deep stage (h = 0 for warps 2-5, 1 for warps 6-9).
    const int r = (warp & 3) * 32 + lane, h = (warp - 2) >> 2;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    uint32_t gs = 0;
    bool ok = true;
    for (int i = b; ok && i < n_items; i += G) {
      for (int kt = 0; kt < KG; ++kt, ++gs) {
        const uint32_t sr = gs % C::RS, sa = gs % C::AS;
        if (!mbar_wait_bounded(&r_full[sr], (gs / C::RS) & 1u, a.status) ||
            (gs >= (uint32_t)C::AS && !mbar_wait_bounded(&a_empty[sa], ((gs / C::AS) & 1u) ^ 1u, a.status))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint8_t* raw = sR + sr * C::RAWB;
        const uint32_t ta = tmem + lane_base + C::A0 + sa * C::A_COLS + 16 * h;
        uint32_t o[16];
        decode_regs<FMT>(raw, r, h, o);
        tmem_st16(ta, o);
        if (DUAL) {
          decode_regs<FMT>(raw + C::RAW1, r, h, o);
          tmem_st16(ta + 32, o);
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&a_full[sa]);
          mbar_arrive(&r_empty[sr]);
        }
      }
    }
  } else if (warp < kMpGatWarp0) {
    // ------------------------------------------------------------ epilogue
    const int quarter = warp & 3, half = (warp - kMpEpiWarp0) >> 2;
    const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
    uint32_t itc = 0;
    for (int i = b; i < n_items; i += G, ++itc) {
      const MpItem it = mp_item<DUAL>(a, n_rt, i);
      const int N = (it.count + 15) & ~15;
      const uint32_t acc = DUAL ? 0u : (itc & 1u);
      if (!mbar_wait_bounded(&t_full[acc], (itc / C::ACC) & 1u, a.status)) break;
      tc_fence_after();
      const int64_t n = (int64_t)it.q * 128 + quarter * 32 + lane;
      for (int c = 16 * half; c < N; c += 32) {
        uint32_t v[16];
        tmem_ld16(tmem + lane_base + acc * C::ACC_COLS + (uint32_t)c, v);
        if (DUAL) {
          uint32_t u[16];
          tmem_ld16(tmem + lane_base + kMpTile + (uint32_t)c, u);
          tmem_ld_wait();
          __nv_bfloat16* hout = static_cast<__nv_bfloat16*>(a.out) + (int64_t)(it.out_base + c) * a.ldo + n;
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            if (c + j < it.count) {
              const float g = it.ts * __uint_as_float(v[j]);
              const float up = it.ts * __uint_as_float(u[j]);
              // silu(g) = g / (1 + e^-g); e^-g capped at e^80 keeps the quotient finite
              const float silu = __fdividef(g, 1.0f + __expf(-fmaxf(g, -80.0f)));
              hout[(int64_t)j * a.ldo] = __float2bfloat16_rn(silu * up);
            }
          }
        } else {
          tmem_ld_wait();
          if (n < a.n_out) {
            float* dout = static_cast<float*>(a.out) + (int64_t)(it.out_base + c) * a.ldo + n;
#pragma unroll
            for (int j = 0; j < 16; ++j)
              if (c + j < it.count) dout[(int64_t)j * a.ldo] = it.ts * __uint_as_float(v[j]);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&t_empty[acc]);
    }
  } else {
    // ------------------------------------------------------------ activation gather
    // Each thread copies 16-byte chunks of the stage's rows and arrives on the stage's
    // barrier when its copies land (cp.async.mbarrier.arrive.noinc), so the gather runs up
    // to BS stages ahead without waiting on its own loads.
    const int gt = tid - kMpGatWarp0 * 32;
    const int c8 = gt & 7, rs = gt >> 3;  // 16-byte chunk of a 128-byte row; row within 16
    uint32_t gs = 0;
    bool ok = true;
    for (int i = b; ok && i < n_items; i += G) {
      const MpItem it = mp_item<DUAL>(a, n_rt, i);
      const int N = (it.count + 15) & ~15;
      int row[kMpTile / 16];
#pragma unroll
      for (int ii = 0; ii < kMpTile / 16; ++ii) {
        const int j = rs + 16 * ii;
        row[ii] = j < it.count ? (it.in_list ? it.in_list[j] / a.topk : it.in_base + j) : -1;
      }
      for (int kt = 0; kt < KG; ++kt, ++gs) {
        const uint32_t s = gs % C::BS;
        if (gs >= (uint32_t)C::BS && !mbar_wait_bounded(&b_empty[s], ((gs / C::BS) & 1u) ^ 1u, a.status)) {
          ok = false;
          break;
        }
        uint8_t* dst = sB + s * C::B;
        const int64_t k0 = (int64_t)kt * 64 + c8 * 8;
        const uint32_t kb = k0 + 8 <= a.K ? 16u : (k0 < a.K ? (uint32_t)(a.K - k0) * 2u : 0u);
#pragma unroll
        for (int ii = 0; ii < kMpTile / 16; ++ii) {
          const int j = rs + 16 * ii;
          if (j < N) {
            const bool live = row[ii] >= 0 && kb > 0;
            const __nv_bfloat16* src = live ? a.in + (int64_t)row[ii] * a.ldi + k0 : a.in;
            cp_async16(dst + (j >> 3) * 1024 + (j & 7) * 128 + ((c8 ^ (j & 7)) << 4), src, live ? kb : 0u);
          }
        }
        cp_async_arrive_noinc(&b_full[s]);
      }
    }
    cp_async_wait_all();  // no copy in flight into shared memory past this point
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// out[t][n] = bf16( sum_j w[t][j] * d[pos(t, j)][n] + d[T*topk + t][n] ), fixed order, four
// features per thread.
__global__ void __launch_bounds__(256) moe_finish4_kernel(const float* d, int64_t ldd, const float* w,
                                                          const int* pair_pos, int T, int topk, int has_shared,
                                                          int64_t H, __nv_bfloat16* out, int64_t ldo) {
  const int64_t H4 = H / 4;
  const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= (int64_t)T * H4) return;
  const int t = (int)(idx / H4);
  const int64_t n = (idx % H4) * 4;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int j = 0; j < topk; ++j) {
    const float p = w[(int64_t)t * topk + j];
    const float4 v = __ldcs(reinterpret_cast<const float4*>(d + (int64_t)pair_pos[(int64_t)t * topk + j] * ldd + n));
    acc.x = fmaf(p, v.x, acc.x);
    acc.y = fmaf(p, v.y, acc.y);
    acc.z = fmaf(p, v.z, acc.z);
    acc.w = fmaf(p, v.w, acc.w);
  }
  if (has_shared) {
    const float4 v = __ldcs(reinterpret_cast<const float4*>(d + (int64_t)(T * topk + t) * ldd + n));
    acc.x += v.x;
    acc.y += v.y;
    acc.z += v.z;
    acc.w += v.w;
  }
  __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y), hi = __floats2bfloat162_rn(acc.z, acc.w);
  uint2 pk;
  pk.x = *reinterpret_cast<uint32_t*>(&lo);
  pk.y = *reinterpret_cast<uint32_t*>(&hi);
  *reinterpret_cast<uint2*>(out + (int64_t)t * ldo + n) = pk;
}

// ---------------------------------------------------------------- host side
namespace {

template <int FMT, bool DUAL>
int launch_mp(const MpArgs& a, const DeviceInfo& dev, cudaStream_t s) {
  using C = MpCfg<FMT, DUAL>;
  static std::atomic<unsigned long long> configured{0};
  if (C::SMEM > dev.max_smem_optin) return QG_ERR_UNSUPPORTED;
  int devid = 0;
  if (cudaGetDevice(&devid) != cudaSuccess) return QG_ERR_CUDA;
  const unsigned long long bit = 1ull << (devid & 63);
  if (!(configured.load() & bit)) {
    if (cudaFuncSetAttribute((const void*)moe_gemm_kernel<FMT, DUAL>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             C::SMEM) != cudaSuccess)
      return QG_ERR_CUDA;
    configured.fetch_or(bit);
  }
  moe_gemm_kernel<FMT, DUAL><<<dev.sms, kMpThreads, C::SMEM, s>>>(a);
  return cudaGetLastError() == cudaSuccess ? QG_OK : QG_ERR_CUDA;
}

template <bool DUAL>
int launch_mp_fmt(int fmt, const MpArgs& a, const DeviceInfo& dev, cudaStream_t s) {
  switch (fmt) {
    case FMT_MLX: return launch_mp<FMT_MLX, DUAL>(a, dev, s);
    case FMT_MXFP4: return launch_mp<FMT_MXFP4, DUAL>(a, dev, s);
    case FMT_NVFP4: return launch_mp<FMT_NVFP4, DUAL>(a, dev, s);
    default: return launch_mp<FMT_Q6K, DUAL>(a, dev, s);
  }
}

}  // namespace

int launch_moe_prefill(const qg_moe_layer* m, const Geometry& gu, const Geometry& dn, const void* x, int64_t T,
                       int64_t ldx, int topk, const float* topk_w, const void* route_ws, void* out, int64_t ldo,
                       void* ws, const DeviceInfo& dev, void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const RouteView rv = route_view(const_cast<void*>(route_ws), T, m->n_experts, topk);
  const MoeLayout L = moe_layout(gu, dn, T, m->n_experts, topk, dev.sms);
  uint8_t* w = static_cast<uint8_t*>(ws);
  const int F = (int)dn.k;
  size_t cb = 0, sb = 0, ab = 0;
  qg_packed_sizes(m->fmt, gu.n, gu.k, &cb, &sb, &ab);

  MpArgs a{};
  a.codes = static_cast<const uint8_t*>(m->gu_codes);
  a.scales = static_cast<const uint8_t*>(m->gu_scales);
  a.aux = static_cast<const uint8_t*>(m->gu_aux);
  a.cstride = (int64_t)cb;
  a.sstride = (int64_t)sb;
  a.astride = (int64_t)ab;
  a.n_sh_tiles = m->has_shared ? (int)((T + kMpTile - 1) / kMpTile) : 0;
  a.sh_codes = m->has_shared ? static_cast<const uint8_t*>(m->shared_gate_up.codes) : nullptr;
  a.sh_scales = m->has_shared ? static_cast<const uint8_t*>(m->shared_gate_up.scales) : nullptr;
  a.sh_aux = m->has_shared ? static_cast<const uint8_t*>(m->shared_gate_up.aux) : nullptr;
  a.ts = (m->fmt == FMT_NVFP4) ? m->tensor_scale : 1.0f;
  a.sh_ts = (m->has_shared && m->fmt == FMT_NVFP4) ? m->shared_gate_up.tensor_scale : 1.0f;
  a.in = static_cast<const __nv_bfloat16*>(x);
  a.ldi = ldx;
  a.K = gu.k;
  a.KG = (int)gu.kg;
  a.out = w + L.h;
  a.ldo = L.ld_h;
  a.n_out = F;
  a.QN = F / 128;
  a.T = (int)T;
  a.topk = topk;
  a.meta = rv.meta;
  a.tiles = rv.tiles;
  a.pair_list = rv.pair_list;
  a.status = reinterpret_cast<int*>(w);
  int st = launch_mp_fmt<true>(m->fmt, a, dev, s);
  if (st != QG_OK) return st;

  qg_packed_sizes(m->fmt, dn.n, dn.k, &cb, &sb, &ab);
  MpArgs d = a;
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
  d.in = reinterpret_cast<const __nv_bfloat16*>(w + L.h);
  d.ldi = L.ld_h;
  d.K = dn.k;
  d.KG = (int)dn.kg;
  d.out = w + L.d;
  d.ldo = L.ld_d;
  d.n_out = dn.n;
  d.QN = (int)dn.nt;
  st = launch_mp_fmt<false>(m->fmt, d, dev, s);
  if (st != QG_OK) return st;

  const int64_t H = dn.n;
  const int64_t n4 = T * (H / 4);
  moe_finish4_kernel<<<(unsigned)((n4 + 255) / 256), 256, 0, s>>>(
      reinterpret_cast<const float*>(w + L.d), L.ld_d, topk_w, rv.pair_pos, (int)T, topk, m->has_shared, H,
      static_cast<__nv_bfloat16*>(out), ldo);
  return cudaGetLastError() == cudaSuccess ? QG_OK : QG_ERR_CUDA;
}

}  // namespace qg
