// Host-side internals shared by the C ABI entry points and the kernel launchers.
#pragma once

#include <cuda.h>
#include <stddef.h>
#include <stdint.h>

#include "qgemv.h"

namespace qg {

// Geometry of the packed "T128x64" layout.
struct Geometry {
  int fmt;
  int64_t n, k;      // logical
  int64_t np, kp;    // padded
  int64_t nt, kg;    // row tiles of 128, input groups of 64
  int tile_bytes;    // codes per tile
  int sb;            // scale bytes per row per tile
};
bool geometry(int fmt, int64_t n, int64_t k, Geometry* g);
int format_block(int fmt);  // k must be a multiple of this (64, 32, 16, 256); 0 if unknown
bool is_q5(int fmt);        // one of the 5-bit formats
int aux_group_bytes(int fmt);  // aux bytes per row tile and 256 inputs (Q6_K, Q5_K), else 0

// Per-device attributes, cached once per device.
struct DeviceInfo {
  int sms;
  int max_smem_optin;
};
bool device_info(int device, DeviceInfo* out);
bool current_device_info(DeviceInfo* out);

// GEMV launch plan (persistent stream-K over 128 x 64 tiles).
struct GemvPlan {
  int grid;          // CTAs
  int nslots;        // staged 64-wide activation groups per CTA
  int stages;        // weight pipeline depth
  size_t smem;       // dynamic shared memory bytes
  size_t ws_bytes;   // workspace bytes
  size_t off_cnt, off_part;  // workspace offsets
  int64_t units;
  int csplit;        // > 1: each row tile split across a cluster of csplit CTAs
};
bool plan_gemv(const Geometry& g, int m, const DeviceInfo& dev, GemvPlan* p);
// Host-side checks of a GEMV call's weight, rows, activations, residual and output (every
// rule of qgemv but the workspace's); fills g.  Returns a qg_status.
int check_gemv_call(const qg_weight* w, const void* x, int m, int64_t ldx, const void* residual, int64_t ldr,
                    const void* y, int64_t ldy, Geometry* g);

// Launchers (return a qg_status).
int launch_gemv(const Geometry& g, const qg_weight* w, const void* x, int m, int64_t ldx,
                const void* res, int64_t ldr, void* y, int64_t ldy, void* ws, const GemvPlan& p,
                void* stream);
int launch_dequant(const Geometry& g, const qg_weight* w, int out_dtype, void* out, int64_t ldo, void* stream);
// The token rows as a 2-D TMA tensor (rows x k bf16, row stride ldx elements): box of 64
// inputs x box_rows rows, 128-byte swizzle, zero fill.
bool encode_token_rows(CUtensorMap* map, const void* x, int64_t rows, int64_t k, int64_t ldx, int box_rows);
// Tensor-core GEMM for 5..kSmallGemmMaxRows token rows, one token tile (split K over a
// cluster when the row tiles are few); more rows take the 256-token-tile prefill GEMM.
constexpr int64_t kSmallGemmMaxRows = 128;
int launch_gemm_small(const Geometry& g, const qg_weight* w, const void* x, int64_t t, int64_t ldx, const void* res,
                      int64_t ldr, void* y, int64_t ldy, void* ws, const DeviceInfo& dev, void* stream);
// NVFP4 activation quantisation (W4A4): codes / scales / exact bf16 expansion, each
// output optional (NULL: not written).  Arguments validated by the caller.
int launch_quant_act_nvfp4(const void* x, int64_t m, int64_t k, int64_t ldx, float act_scale, uint8_t* codes,
                           int64_t ldc, uint8_t* scales, int64_t lds, void* xe, int64_t lde, void* stream);
int launch_prefill(const Geometry& g, const qg_weight* w, const void* x, int64_t t, int64_t ldx, const void* res,
                   int64_t ldr, void* y, int64_t ldy, void* ws, void* stream);
// W4A4 GEMM on the block-scaled FP4 tensor cores: NVFP4 weight w, activations already
// quantised to NVFP4 (codes [t][ldc] bytes, two per byte; E4M3 scales [t][lds]; ldc and lds
// multiples of 16, both arrays 16-byte aligned), y = bf16(ts_w * act_scale * sum (+ res)).
int launch_gemm_fp4(const Geometry& g, const qg_weight* w, float act_scale, const uint8_t* xcodes, int64_t ldc,
                    const uint8_t* xscales, int64_t lds, int64_t t, const void* res, int64_t ldr, void* y, int64_t ldy,
                    void* ws, void* stream);

constexpr size_t kWsHeader = 256;  // status word + reserved

// Mixture-of-experts decode workspace (after the status header).
struct MoeLayout {
  size_t gu, h, d, total;
  int64_t ld_gu, ld_h, ld_d;
  int p_gu, p_dn;            // decode: input parts of the gate/up and down GEMVs (outputs per part)
  int64_t pst_gu, pst_dn;    // floats between two parts' outputs
};
MoeLayout moe_layout(const Geometry& gu, const Geometry& dn, int64_t T, int E, int topk, int grid);
// MoE chains: the whole FFN (kMoeAll: x -> out), or one stage of it -- kMoeGateUp: x -> h
// (bf16 [rows][ldo], grouped rows then the shared expert's), kMoeDown: h (x, ldx) -> out.
// shared_gate: fp32 gate logits [T] of the shared expert (its output is weighed by their
// sigmoid in the finish) or null (weight 1).
enum MoeStage { kMoeAll = 0, kMoeGateUp = 1, kMoeDown = 2 };
// logits non-null (decode, kMoeAll): the gate/up launch routes the tokens itself and stores
// the router's outputs (topk_ids_out, topk_w_out, route_ws) on the way.
int launch_moe_decode(const qg_moe_layer* m, const Geometry& gu, const Geometry& dn, const void* x, int64_t T,
                      int64_t ldx, int topk, const float* topk_w, const float* shared_gate, const void* route_ws,
                      void* out, int64_t ldo, void* ws, const DeviceInfo& dev, void* stream, int stage,
                      const float* logits = nullptr, int32_t* topk_ids_out = nullptr, float* topk_w_out = nullptr);
int launch_moe_prefill(const qg_moe_layer* m, const Geometry& gu, const Geometry& dn, const void* x, int64_t T,
                       int64_t ldx, int topk, const float* topk_w, const float* shared_gate, const void* route_ws,
                       void* out, int64_t ldo, void* ws, const DeviceInfo& dev, void* stream, int stage);

}  // namespace qg
