// Tensor-core GEMMs with on-chip dequantisation (TurboEXL3 article §4.1, "Prefill: decode
// once, multiply many times"): every packed 128 x 64 weight tile is decoded once per
// token tile into the tensor cores' operand and multiplied by up to 192 tokens; the decoded
// weights never reach device memory.  One kernel body serves the two GEMMs of the MoE layer:
//
//   MoE gate/up     one grouped GEMM over the router's tile table (tiles of <= 192 pairs of one
//                   expert): a work item is (tile, 128 features f..f+127), whose two row tiles
//                   are the expert's gate rows f.. and up rows F+f..; the token rows are
//                   gathered straight from x by index; the epilogue is the mid step
//                   h = bf16(silu(gate) * up) in fp32 (§4.1 "Mid"), so the gate/up outputs
//                   never reach device memory
//   MoE down        the same on h (rows already in grouped order), two row tiles per item,
//                   outputs per (token, expert) pair for the finish, rounded to bf16 (the
//                   type a GEMM hands on; the finish sums them in fp32)
// The MoE shared expert runs as extra token tiles of the gate/up and down GEMMs.  Tile widths are ragged: the MMA's N is the tile's token count
// rounded up to 16.
//
// Persistent and warp-specialised (one CTA per SM walks the work items):
//   warp 0       raw-weight producer: bulk copies of both packed tiles of a stage into a
//                deep shared-memory ring
//   warp 1       allocates all 512 TMEM columns; one lane issues the tcgen05.mma
//   warps 2-9    decode each stage's two tiles into the bf16 A operand in tensor memory
//                (tcgen05.st; warps 2-5 the even stages, 6-9 the odd ones), so decoded
//                weights cost no shared-memory bandwidth
//   warps 10-21  epilogue: TMEM -> registers -> outputs
//   warps 22-29  token rows: one TMA load per stage when the rows are contiguous, else a
//                cp.async gather by row index into the 128-byte swizzled ring; each
//                thread's copies arrive on the stage's mbarrier when they land, and the MMA
//                thread fences these generic-proxy writes before the tensor cores read them
// Two accumulators (one per row tile, 192 columns each): an item's two row tiles share each
// stage's token rows, so the B operand is loaded once for both.  Every wait is bounded
// (QG_ERR_TIMEOUT in the workspace status word) and TMEM is freed on every path.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <mutex>

#include "qg_common.cuh"
#include "qg_decode_tile.cuh"
#include "qg_internal.h"
#include "qg_route.h"
#include "qg_sync.cuh"
#include "qg_tc.cuh"

namespace qg {

constexpr int kTcDecWarps = 8;  // two groups of four (one per TMEM lane quarter), alternate stages
constexpr int kTcEpiWarps = 12;  // three per TMEM lane quarter, every third 16-column chunk
constexpr int kTcGatWarps = 8;  // the gathered token rows keep 256 threads busy
constexpr int kTcGatThreads = kTcGatWarps * 32;
constexpr int kTcWarps = 2 + kTcDecWarps + kTcEpiWarps + kTcGatWarps;  // 30
constexpr int kTcThreads = kTcWarps * 32;                               // 960
constexpr int kTcEpiWarp0 = 2 + kTcDecWarps;                            // 10
constexpr int kTcGatWarp0 = kTcEpiWarp0 + kTcEpiWarps;                  // 22
constexpr int kTcTile = kRouteTile;  // tokens per tile = largest MMA N (192)
constexpr int kTcSmemCap = 232448;   // opt-in shared memory per block on sm_100-family GPUs

enum TcEpilogue { kEpiSwiglu = 0, kEpiPairBf16 = 1 };

// Tensor memory (512 columns x 128 lanes of 32 bits): accumulators of the two row tiles in
// columns [0, 192) and [192, 384); A ring of 2 stages x 64 columns (first tile's 64 inputs in
// 32 columns, then the second's) in [384, 512).  Shared memory: the gathered token rows
// (6 stages) and the raw packed tiles.
template <int FMT>
struct TcCfg {
  using F = Fmt<FMT>;
  static constexpr int RAW1 = F::TB + 128 * F::SB + (FMT == FMT_Q6K ? 256 : 0);  // one packed tile
  static constexpr int RAWB = 2 * RAW1;
  static constexpr int B = kTcTile * 128;
  static constexpr int BS = 6;
  static constexpr int AS = 2;
  static constexpr uint32_t A_COLS = 64;
  static constexpr uint32_t A0 = 2 * kTcTile;
  static_assert(A0 + AS * A_COLS <= 512, "tensor memory");
  static constexpr int FIT = (kTcSmemCap - 1024 - 512 - BS * B) / RAWB;
  static constexpr int RS = FIT > 16 ? 16 : FIT;
  static constexpr int OFF_RAW = BS * B;
  static constexpr int OFF_BAR = OFF_RAW + RS * RAWB;
  static constexpr int NBAR = 2 * RS + 2 * AS + 2 * BS + 2 + 1;
  static constexpr int SMEM = 1024 + OFF_BAR + NBAR * 8 + 16;
  static_assert(RS >= 4, "raw ring too shallow");
  static_assert(SMEM <= kTcSmemCap, "shared memory");
};

struct TcArgs {
  // routed experts (MoE), concatenated; unused when meta is null
  const uint8_t* codes;
  const uint8_t* scales;
  const uint8_t* aux;
  int64_t cstride, sstride, astride;
  float ts;
  // the MoE shared expert: every token in kTcTile-token tiles
  const uint8_t* sh_codes;
  const uint8_t* sh_scales;
  const uint8_t* sh_aux;
  float sh_ts;
  int n_sh_tiles;
  int sh_in_off, sh_out_off;  // input / output row of token 0 of the shared-expert tiles
  const __nv_bfloat16* in;    // token rows [*][ldi], K inputs each
  int64_t ldi;
  int64_t K;
  int KG;
  int NT;     // 128-row tiles of the weight
  int QN;     // items per token tile
  int T;      // tokens
  int topk;   // routed gate/up: input row = pair / topk
  void* out;  // kEpiSwiglu: bf16 h [*][ldo]; kEpiPairBf16: bf16 [*][ldo]
  int64_t ldo;
  int64_t n_out;
  int64_t F;  // kEpiSwiglu: rows of the gate half (up rows start at F)
  const int* meta;  // router: [1] = routed tiles
  const int* tiles;
  const int* pair_list;
  int* status;
};

struct TcItem {
  const uint8_t* codes;
  const uint8_t* scales;
  const uint8_t* aux;
  const int* in_list;  // routed gate/up: grouped position -> pair; row = pair / topk
  float ts;
  int rt0, rt1;        // the two row tiles
  bool second;         // rt1 exists (else rt1 == rt0 and its outputs are dropped)
  int count, in_base, out_base, feat0;
};

template <int EPI>
__device__ __forceinline__ TcItem tc_item(const TcArgs& a, int n_rt, int i) {
  TcItem it;
  const int ti = i / a.QN;
  const int q = i - ti * a.QN;
  if (EPI == kEpiSwiglu) {
    it.rt0 = q;
    it.rt1 = q + a.QN;
    it.second = true;
    it.feat0 = q * 128;
  } else {
    it.rt0 = 2 * q;
    it.second = 2 * q + 1 < a.NT;
    it.rt1 = it.second ? 2 * q + 1 : 2 * q;
    it.feat0 = 2 * q * 128;
  }
  if (ti < n_rt) {
    const int e = a.tiles[3 * ti], first = a.tiles[3 * ti + 1];
    it.count = a.tiles[3 * ti + 2];
    it.codes = a.codes + (int64_t)e * a.cstride;
    it.scales = a.scales + (int64_t)e * a.sstride;
    it.aux = a.aux ? a.aux + (int64_t)e * a.astride : nullptr;
    it.ts = a.ts;
    it.out_base = first;
    it.in_list = EPI == kEpiSwiglu ? a.pair_list + first : nullptr;
    it.in_base = first;
  } else {
    const int t0 = (ti - n_rt) * kTcTile;
    it.count = min(kTcTile, a.T - t0);
    it.codes = a.sh_codes;
    it.scales = a.sh_scales;
    it.aux = a.sh_aux;
    it.ts = a.sh_ts;
    it.out_base = a.sh_out_off + t0;
    it.in_list = nullptr;
    it.in_base = a.sh_in_off + t0;
  }
  return it;
}

template <int FMT>
__device__ __forceinline__ void tc_load_tile(uint8_t* dst, const TcItem& it, int row_tile, int KG, int kt,
                                             uint64_t* bar) {
  using F = Fmt<FMT>;
  const int64_t tile = (int64_t)row_tile * KG + kt;
  bulk_g2s(dst, it.codes + tile * F::TB, F::TB, bar);
  bulk_g2s(dst + F::TB, it.scales + tile * (128 * F::SB), 128 * F::SB, bar);
  if (FMT == FMT_Q6K)
    bulk_g2s(dst + F::TB + 128 * F::SB, it.aux + ((int64_t)row_tile * (KG / 4) + kt / 4) * 256, 256, bar);
}

template <int FMT, int EPI>
__global__ void __launch_bounds__(kTcThreads, 1) tc_gemm_kernel(const __grid_constant__ CUtensorMap tmb, const TcArgs a) {
  using C = TcCfg<FMT>;
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
  uint64_t* t_empty = t_full + 1;
  uint64_t* fin = t_empty + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(fin + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n_rt = a.meta ? a.meta[1] : 0;
  const int n_items = (n_rt + a.n_sh_tiles) * a.QN;
  const int G = gridDim.x, b = blockIdx.x;
  const int KG = a.KG;

  if (tid == 0) {
    for (int s = 0; s < C::RS; ++s) {
      mbar_init(&r_full[s], 1);
      mbar_init(&r_empty[s], 4);  // the four decode warps of the stage's group
    }
    for (int s = 0; s < C::AS; ++s) {
      mbar_init(&a_full[s], 4);
      mbar_init(&a_empty[s], 1);
    }
    for (int s = 0; s < C::BS; ++s) {
      mbar_init(&b_full[s], kTcGatThreads);  // one cp.async completion arrival per gather thread
      mbar_init(&b_empty[s], 1);
    }
    mbar_init(t_full, 1);
    mbar_init(t_empty, kTcEpiWarps);
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
        const TcItem it = tc_item<EPI>(a, n_rt, i);
        for (int kt = 0; kt < KG; ++kt, ++gs) {
          const uint32_t s = gs % C::RS;
          if (gs >= (uint32_t)C::RS && !mbar_wait_bounded(&r_empty[s], ((gs / C::RS) & 1u) ^ 1u, a.status)) {
            ok = false;
            break;
          }
          uint8_t* dst = sR + s * C::RAWB;
          mbar_arrive_expect_tx(&r_full[s], C::RAWB);
          tc_load_tile<FMT>(dst, it, it.rt0, KG, kt, &r_full[s]);
          tc_load_tile<FMT>(dst + C::RAW1, it, it.rt1, KG, kt, &r_full[s]);
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
        const TcItem it = tc_item<EPI>(a, n_rt, i);
        const int N = (it.count + 15) & ~15;
        const uint32_t idesc = idesc_bf16_f32(128, N);
        if (itc >= 1u && !mbar_wait_bounded(t_empty, (itc & 1u) ^ 1u, a.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
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
            mma_bf16_ts(tmem, ta + kk * 8, bd, idesc, accum);
            mma_bf16_ts(tmem + kTcTile, ta + 32 + kk * 8, bd, idesc, accum);
          }
          mma_commit(&a_empty[sa]);
          mma_commit(&b_empty[sb]);
        }
        if (!ok) break;
        mma_commit(t_full);
      }
      mma_commit(fin);  // every MMA issued so far is complete when this arrives
      mbar_wait_bounded(fin, 0, a.status);
    }
    __syncwarp();
  } else if (warp < kTcEpiWarp0) {
    // ------------------------------------------------------------ decode
    // Warp w may only touch TMEM lanes 32*(w%4)..: it decodes rows 32*(w%4)+lane, all 64
    // inputs of both row tiles of every other stage (warps 2-5 the even stages, 6-9 the odd
    // ones), each tile stored with one 32-column tensor-memory write (wide writes contend
    // less with the MMAs reading tensor memory than 16-column ones: 911 -> 866 us for the
    // 8192-token FFN).
    const int r = (warp & 3) * 32 + lane, grp = (warp - 2) >> 2;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    uint32_t gs = 0;
    bool ok = true;
    for (int i = b; ok && i < n_items; i += G) {
      for (int kt = 0; kt < KG; ++kt, ++gs) {
        if ((int)(gs & 1u) != grp) continue;
        const uint32_t sr = gs % C::RS, sa = gs % C::AS;
        if (!mbar_wait_bounded(&r_full[sr], (gs / C::RS) & 1u, a.status) ||
            (gs >= (uint32_t)C::AS && !mbar_wait_bounded(&a_empty[sa], ((gs / C::AS) & 1u) ^ 1u, a.status))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint8_t* raw = sR + sr * C::RAWB;
        const uint32_t ta = tmem + lane_base + C::A0 + sa * C::A_COLS;
        for (int tl = 0; tl < 2; ++tl) {
          uint32_t o[32];
          decode_regs<FMT>(raw + tl * C::RAW1, r, 0, *reinterpret_cast<uint32_t(*)[16]>(o));
          decode_regs<FMT>(raw + tl * C::RAW1, r, 1, *reinterpret_cast<uint32_t(*)[16]>(o + 16));
          tmem_st32(ta + 32 * tl, o);
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
  } else if (warp < kTcGatWarp0) {
    // ------------------------------------------------------------ epilogue
    const int quarter = warp & 3, third = (warp - kTcEpiWarp0) >> 2;
    const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
    uint32_t itc = 0;
    for (int i = b; i < n_items; i += G, ++itc) {
      const TcItem it = tc_item<EPI>(a, n_rt, i);
      const int N = (it.count + 15) & ~15;
      if (!mbar_wait_bounded(t_full, itc & 1u, a.status)) break;
      tc_fence_after();
      const int r = quarter * 32 + lane;
      for (int c = 16 * third; c < N; c += 48) {
        uint32_t v[16], u[16];
        tmem_ld16(tmem + lane_base + (uint32_t)c, v);
        tmem_ld16(tmem + lane_base + kTcTile + (uint32_t)c, u);
        tmem_ld_wait();
        if (EPI == kEpiSwiglu) {
          // h of features f, f+1 (f even) sits in lanes 2i, 2i+1: as in the down epilogue, the
          // two lanes swap one value per pair of tokens and each stores one 4-byte h pair
          const int odd = lane & 1;
          const int64_t n = it.feat0 + (r & ~1);  // < F: F is a multiple of 128
          uint32_t* hout = reinterpret_cast<uint32_t*>(static_cast<__nv_bfloat16*>(a.out) + n);
#pragma unroll
          for (int j = 0; j < 16; j += 2) {
            float h[2];
#pragma unroll
            for (int i = 0; i < 2; ++i) {
              const float g = it.ts * __uint_as_float(v[j + i]);
              const float up = it.ts * __uint_as_float(u[j + i]);
              // silu(g) = g / (1 + e^-g); e^-g capped at e^80 keeps the quotient finite
              h[i] = __fdividef(g, 1.0f + __expf(-fmaxf(g, -80.0f))) * up;
            }
            const float hr = __shfl_xor_sync(0xffffffffu, odd ? h[0] : h[1], 1);
            const int tok = c + j + odd;
            if (tok < it.count) {
              const __nv_bfloat162 ph = __floats2bfloat162_rn(odd ? hr : h[0], odd ? h[1] : hr);
              hout[((int64_t)(it.out_base + tok) * a.ldo) >> 1] = *reinterpret_cast<const uint32_t*>(&ph);
            }
          }
        } else {
          // lanes 2i and 2i+1 hold features f, f+1 (f even) of the same 16 tokens: each
          // pair of tokens, they swap one value so that the even lane stores both features
          // of token j and the odd lane both of token j+1, as one 4-byte bf16 pair
          const int odd = lane & 1;
          const int64_t n0 = (int64_t)it.rt0 * 128 + (r & ~1), n1 = (int64_t)it.rt1 * 128 + (r & ~1);
          const bool w0 = n0 < a.n_out, w1 = it.second && n1 < a.n_out;  // n_out is even
#pragma unroll
          for (int j = 0; j < 16; j += 2) {
            const float v0 = __uint_as_float(v[j]), v1 = __uint_as_float(v[j + 1]);
            const float u0 = __uint_as_float(u[j]), u1 = __uint_as_float(u[j + 1]);
            const float vr = __shfl_xor_sync(0xffffffffu, odd ? v0 : v1, 1);
            const float ur = __shfl_xor_sync(0xffffffffu, odd ? u0 : u1, 1);
            const int tok = c + j + odd;
            if (tok < it.count) {
              uint32_t* o = reinterpret_cast<uint32_t*>(static_cast<__nv_bfloat16*>(a.out) +
                                                        (int64_t)(it.out_base + tok) * a.ldo);
              const __nv_bfloat162 pv = __floats2bfloat162_rn(it.ts * (odd ? vr : v0), it.ts * (odd ? v1 : vr));
              const __nv_bfloat162 pu = __floats2bfloat162_rn(it.ts * (odd ? ur : u0), it.ts * (odd ? u1 : ur));
              if (w0) o[n0 >> 1] = *reinterpret_cast<const uint32_t*>(&pv);
              if (w1) o[n1 >> 1] = *reinterpret_cast<const uint32_t*>(&pu);
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(t_empty);
    }
  } else {
    // ------------------------------------------------------------ token rows
    // Contiguous rows (dense GEMM, MoE down, shared-expert tiles): one 2-D TMA load of
    // 64 inputs x 192 rows per stage (128-byte swizzle; rows past the tensor read as zero),
    // issued by the first gather thread with the stage's byte count, the other threads
    // arriving plainly.  Routed gate/up tiles: each thread copies 16-byte chunks of the rows
    // by index and arrives on the stage's barrier when its copies land
    // (cp.async.mbarrier.arrive.noinc), so the gather runs up to BS stages ahead without
    // waiting on its own loads.
    const int gt = tid - kTcGatWarp0 * 32;
    constexpr int kRowsPass = kTcGatThreads / 8;  // rows one pass of the gather threads covers
    const int c8 = gt & 7, rs = gt >> 3;          // 16-byte chunk of a 128-byte row; row within a pass
    uint32_t gs = 0;
    bool ok = true;
    for (int i = b; ok && i < n_items; i += G) {
      const TcItem it = tc_item<EPI>(a, n_rt, i);
      const int N = (it.count + 15) & ~15;
      const bool gather = it.in_list != nullptr;
      int row[kTcTile / kRowsPass];
#pragma unroll
      for (int ii = 0; ii < kTcTile / kRowsPass; ++ii) {
        const int j = rs + kRowsPass * ii;
        row[ii] = (gather && j < it.count) ? it.in_list[j] / a.topk : -1;
      }
      for (int kt = 0; kt < KG; ++kt, ++gs) {
        const uint32_t s = gs % C::BS;
        if (gs >= (uint32_t)C::BS && !mbar_wait_bounded(&b_empty[s], ((gs / C::BS) & 1u) ^ 1u, a.status)) {
          ok = false;
          break;
        }
        uint8_t* dst = sB + s * C::B;
        if (!gather) {
          if (gt == 0) {
            mbar_arrive_expect_tx(&b_full[s], C::B);
            tma_load_2d(dst, &tmb, kt * 64, it.in_base, &b_full[s]);
          } else {
            mbar_arrive(&b_full[s]);
          }
          continue;
        }
        const int64_t k0 = (int64_t)kt * 64 + c8 * 8;
        const uint32_t kb = k0 + 8 <= a.K ? 16u : (k0 < a.K ? (uint32_t)(a.K - k0) * 2u : 0u);
#pragma unroll
        for (int ii = 0; ii < kTcTile / kRowsPass; ++ii) {
          const int j = rs + kRowsPass * ii;
          if (j < N) {
            const bool live = row[ii] >= 0 && kb > 0;
            const __nv_bfloat16* src = live ? a.in + (int64_t)row[ii] * a.ldi + k0 : a.in;
            cp_async16(dst + (j >> 3) * 1024 + (j & 7) * 128 + ((c8 ^ (j & 7)) << 4), src, live ? kb : 0u);
          }
        }
        cp_async_arrive_noinc(&b_full[s]);
      }
    }
    // leave no copy in flight into this CTA's shared memory: cp.async here, TMA below
    if (gt == 0)
      for (uint32_t g2 = gs > (uint32_t)C::BS ? gs - C::BS : 0; g2 < gs; ++g2)
        mbar_wait_bounded(&b_full[g2 % C::BS], (g2 / C::BS) & 1u, a.status);
    cp_async_wait_all();  // no copy in flight into shared memory past this point
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// out[t][n] = bf16( sum_j w[t][j] * d[pos(t, j)][n] + g_t * d[T*topk + t][n] ) with d the
// bf16 per-pair down outputs, summed in fp32 in a fixed order, eight features per thread
// (TurboEXL3 article §4.1 "Finish"; g_t: the shared expert's sigmoid gate, §4.2, or 1).
__device__ __forceinline__ void fma_bf16x8(float (&acc)[8], float p, uint4 v) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    acc[2 * i] = fmaf(p, __uint_as_float(w[i] << 16), acc[2 * i]);
    acc[2 * i + 1] = fmaf(p, __uint_as_float(w[i] & 0xffff0000u), acc[2 * i + 1]);
  }
}

__global__ void __launch_bounds__(256) moe_finish8_kernel(const __nv_bfloat16* d, int64_t ldd, const float* w,
                                                          const int* pair_pos, int T, int topk, int has_shared,
                                                          const float* shared_gate, int64_t H, __nv_bfloat16* out,
                                                          int64_t ldo) {
  const int64_t H8 = H / 8;
  const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= (int64_t)T * H8) return;
  const int t = (int)(idx / H8);
  const int64_t n = (idx % H8) * 8;
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  for (int j = 0; j < topk; ++j) {
    const float p = w[(int64_t)t * topk + j];
    fma_bf16x8(acc, p, __ldcs(reinterpret_cast<const uint4*>(d + (int64_t)pair_pos[(int64_t)t * topk + j] * ldd + n)));
  }
  if (has_shared)
    fma_bf16x8(acc, shared_gate_weight(shared_gate, t),
               __ldcs(reinterpret_cast<const uint4*>(d + (int64_t)(T * topk + t) * ldd + n)));
  uint32_t pk[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __nv_bfloat162 b2 = __floats2bfloat162_rn(acc[2 * i], acc[2 * i + 1]);
    pk[i] = *reinterpret_cast<const uint32_t*>(&b2);
  }
  *reinterpret_cast<uint4*>(out + (int64_t)t * ldo + n) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
}

// ---------------------------------------------------------------- host side
namespace {

using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                              const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                              CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
std::once_flag g_encode_once;
EncodeFn g_encode = nullptr;

// The token-row operand as a 2-D TMA tensor: rows x K bf16, row stride ldi elements, box of
// 64 inputs x 192 rows, 128-byte swizzle (the MMA's K-major operand layout), zero fill.
bool encode_rows(CUtensorMap* map, const void* base, int64_t rows, int64_t K, int64_t ldi) {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<EncodeFn>(fn);
  });
  if (!g_encode) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)ldi * 2};
  const cuuint32_t box[2] = {64, (cuuint32_t)kTcTile};
  const cuuint32_t estr[2] = {1, 1};
  return g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int FMT, int EPI>
int launch_tc(const CUtensorMap& map, const TcArgs& a, int grid, const DeviceInfo& dev, cudaStream_t s) {
  using C = TcCfg<FMT>;
  static std::atomic<unsigned long long> configured{0};
  if (C::SMEM > dev.max_smem_optin) return QG_ERR_UNSUPPORTED;
  int devid = 0;
  if (cudaGetDevice(&devid) != cudaSuccess) return QG_ERR_CUDA;
  const unsigned long long bit = 1ull << (devid & 63);
  if (!(configured.load() & bit)) {
    if (cudaFuncSetAttribute((const void*)tc_gemm_kernel<FMT, EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             C::SMEM) != cudaSuccess)
      return QG_ERR_CUDA;
    configured.fetch_or(bit);
  }
  tc_gemm_kernel<FMT, EPI><<<grid, kTcThreads, C::SMEM, s>>>(map, a);
  return cudaGetLastError() == cudaSuccess ? QG_OK : QG_ERR_CUDA;
}

template <int EPI>
int launch_tc_fmt(int fmt, int64_t in_rows, const TcArgs& a, int grid, const DeviceInfo& dev, cudaStream_t s) {
  CUtensorMap map;
  if (!encode_rows(&map, a.in, in_rows, a.K, a.ldi)) return QG_ERR_CUDA;
  switch (fmt) {
    case FMT_MLX: return launch_tc<FMT_MLX, EPI>(map, a, grid, dev, s);
    case FMT_MXFP4: return launch_tc<FMT_MXFP4, EPI>(map, a, grid, dev, s);
    case FMT_NVFP4: return launch_tc<FMT_NVFP4, EPI>(map, a, grid, dev, s);
    default: return launch_tc<FMT_Q6K, EPI>(map, a, grid, dev, s);
  }
}

int tiles_of(int64_t t) { return (int)((t + kTcTile - 1) / kTcTile); }

}  // namespace

int launch_moe_prefill(const qg_moe_layer* m, const Geometry& gu, const Geometry& dn, const void* x, int64_t T,
                       int64_t ldx, int topk, const float* topk_w, const float* shared_gate, const void* route_ws,
                       void* out, int64_t ldo, void* ws, const DeviceInfo& dev, void* stream, int stage) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const RouteView rv = route_view(const_cast<void*>(route_ws), T, m->n_experts, topk);
  const MoeLayout L = moe_layout(gu, dn, T, m->n_experts, topk, dev.sms);
  uint8_t* w = static_cast<uint8_t*>(ws);
  const int F = (int)dn.k;
  size_t cb = 0, sb = 0, ab = 0;
  qg_packed_sizes(m->fmt, gu.n, gu.k, &cb, &sb, &ab);

  TcArgs a{};
  a.codes = static_cast<const uint8_t*>(m->gu_codes);
  a.scales = static_cast<const uint8_t*>(m->gu_scales);
  a.aux = static_cast<const uint8_t*>(m->gu_aux);
  a.cstride = (int64_t)cb;
  a.sstride = (int64_t)sb;
  a.astride = (int64_t)ab;
  a.ts = (m->fmt == FMT_NVFP4) ? m->tensor_scale : 1.0f;
  a.n_sh_tiles = m->has_shared ? tiles_of(T) : 0;
  a.sh_codes = m->has_shared ? static_cast<const uint8_t*>(m->shared_gate_up.codes) : nullptr;
  a.sh_scales = m->has_shared ? static_cast<const uint8_t*>(m->shared_gate_up.scales) : nullptr;
  a.sh_aux = m->has_shared ? static_cast<const uint8_t*>(m->shared_gate_up.aux) : nullptr;
  a.sh_ts = (m->has_shared && m->fmt == FMT_NVFP4) ? m->shared_gate_up.tensor_scale : 1.0f;
  a.sh_in_off = 0;                  // the shared expert reads x rows
  a.sh_out_off = (int)(T * topk);   // and writes h rows after the routed pairs
  a.in = static_cast<const __nv_bfloat16*>(x);
  a.ldi = ldx;
  a.K = gu.k;
  a.KG = (int)gu.kg;
  a.NT = (int)gu.nt;
  a.QN = F / 128;
  a.T = (int)T;
  a.topk = topk;
  a.out = stage == kMoeGateUp ? out : w + L.h;  // h: the caller's (staged call) or ours
  a.ldo = stage == kMoeGateUp ? ldo : L.ld_h;
  a.n_out = F;
  a.F = F;
  a.meta = rv.meta;
  a.tiles = rv.tiles;
  a.pair_list = rv.pair_list;
  a.status = reinterpret_cast<int*>(w);
  int st = QG_OK;
  if (stage != kMoeDown) {
    st = launch_tc_fmt<kEpiSwiglu>(m->fmt, T, a, dev.sms, dev, s);
    if (st != QG_OK) return st;
  }
  if (stage == kMoeGateUp) return QG_OK;

  qg_packed_sizes(m->fmt, dn.n, dn.k, &cb, &sb, &ab);
  TcArgs d = a;
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
  d.sh_in_off = (int)(T * topk);  // the shared expert's h rows
  d.sh_out_off = (int)(T * topk);
  d.in = stage == kMoeDown ? static_cast<const __nv_bfloat16*>(x) : reinterpret_cast<const __nv_bfloat16*>(w + L.h);
  d.ldi = stage == kMoeDown ? ldx : L.ld_h;
  d.K = dn.k;
  d.KG = (int)dn.kg;
  d.NT = (int)dn.nt;
  d.QN = (int)((dn.nt + 1) / 2);
  d.pair_list = nullptr;
  d.out = w + L.d;
  d.ldo = L.ld_d;
  d.n_out = dn.n;
  st = launch_tc_fmt<kEpiPairBf16>(m->fmt, T * topk + (m->has_shared ? T : 0), d, dev.sms, dev, s);
  if (st != QG_OK) return st;

  const int64_t H = dn.n;
  const int64_t n8 = T * (H / 8);
  moe_finish8_kernel<<<(unsigned)((n8 + 255) / 256), 256, 0, s>>>(
      reinterpret_cast<const __nv_bfloat16*>(w + L.d), L.ld_d, topk_w, rv.pair_pos, (int)T, topk, m->has_shared, shared_gate, H,
      static_cast<__nv_bfloat16*>(out), ldo);
  return cudaGetLastError() == cudaSuccess ? QG_OK : QG_ERR_CUDA;
}

}  // namespace qg
