/*
 * qgemv.h -- C ABI of the GB300 (sm_103a) weight-only quantized GEMV / GEMM library.
 *
 * The operation (TurboEXL3 article §2.2, "NVFP4 with 4-bit and with 16-bit
 * activations", W4A16 case): every weight is expanded from its block-scaled
 * code inside the multiply, activations stay 16-bit (bf16), products are
 * accumulated in fp32 and each output is rounded to bf16 once:
 *
 *     y[m, n] = bf16( sum_k w[n, k] * x[m, k]  (+ residual[m, n]) )
 *
 * Weight formats (TurboEXL3 article §2.1, "Block-scaled 4-bit formats";
 * Q6_K operand PR #19, "What changed"):
 *   QG_FMT_MLX_AFFINE4_G64  w = s * code + b; code 0..15; fp16 s, b per 64 weights (4.5 bpw)
 *   QG_FMT_MXFP4            w = e2m1(code) * 2^(E-127); E8M0 byte E per 32 weights (4.25 bpw)
 *   QG_FMT_NVFP4            w = ts * e4m3(S) * e2m1(code); E4M3 byte S per 16 weights,
 *                           one fp32 tensor scale ts (4.5 bpw)
 *   QG_FMT_Q6K              w = d * sc * (code - 32); code 0..63; int8 sc per 16 weights,
 *                           fp16 d per 256 weights (6.5625 bpw)
 * and the 5-bit formats the Q6_K operand PR's 5-bit nibble operand serves (Q5_K, Q5_1,
 * Q5_0), defined as the public GGML blocks (the pages name them without defining them);
 * code 0..31, 32-weight blocks:
 *   QG_FMT_Q5_0             w = d * (code - 16); fp16 d per 32 weights (5.5 bpw)
 *   QG_FMT_Q5_1             w = d * code + m; fp16 d and m per 32 weights (6 bpw)
 *   QG_FMT_Q5_K             w = (d * sc) * code - dmin * mn; 6-bit sc and mn per 32 weights,
 *                           fp16 d and dmin per 256 weights (5.5 bpw)
 * The 5-bit formats run on the dense paths (qgemv, qgemm, qg_dequant); the MoE entry
 * points take the four formats above and return QG_ERR_UNSUPPORTED for them.
 *
 * Conventions shared by every entry point:
 *   - Matrices are N x K (outputs x inputs).  Activations x are bf16 [m][ldx],
 *     outputs y and residuals are bf16 [m][ldy] / [m][ldr] (row m = token).
 *   - Every device pointer must be 16-byte aligned and every leading dimension a
 *     multiple of 8 elements, else QG_ERR_MISALIGNED.
 *   - Memory is owned by the caller; the library allocates nothing and keeps no
 *     mutable global state except a per-device attribute cache filled once.
 *   - Calls are asynchronous on the given stream (a cudaStream_t passed as
 *     void*; NULL = legacy default stream).  Argument errors are found on the
 *     host and returned before anything is launched.  A failed launch returns
 *     QG_ERR_CUDA.  Outputs are undefined after an error.  No C++ exception
 *     crosses this boundary.
 *   - Results are deterministic: every sum runs in a fixed order and no output
 *     is accumulated with floating-point atomics (TurboEXL3 article §4.4).
 *
 * Packed weight layout "T128x64" (written by qg_pack_host, read by every kernel):
 *   Rows are padded to NP = 128*ceil(N/128) and the inputs to KP = KB*ceil(K/KB),
 *   KB = 256 (Q6_K, Q5_K) or 64 (the others).  Tile (q, g) -- rows 128q..128q+127,
 *   inputs 64g..64g+63 -- has index t = q*KG + g, KG = KP/64.  Padding holds
 *   zero codes and zero scales.
 *   codes : TB bytes per tile at t*TB, TB = 4096 (4-bit), 6144 (Q6_K) or 5120 (5-bit).  Row r of
 *           the tile (rt = r/32, lane = r%32):
 *           4-bit (and the 5-bit low nibbles): 16-byte chunks c = 0,1 at byte
 *           ((rt*2 + c)*32 + lane)*16; byte b holds code (64g + 32c + 2b) in its low
 *           nibble and code (64g + 32c + 2b + 1) in its high nibble.
 *           Q6_K: the 16 inputs 64g + 16kq .. +15 (kq = 0..3) are three little-endian
 *           32-bit words, word c (0..2) at byte ((rt*4 + kq)*3 + c)*128 + 4*lane; byte j
 *           of word c holds in bits 2..7 the code of input 64g + 16kq + 4c + j and in bits
 *           0..1 bits 2c..2c+1 of the code of input 64g + 16kq + 12 + j.
 *           5-bit: bytes 0..4095 hold the low nibbles (code & 15) as the 4-bit chunks
 *           (CH = 2); bytes 4096..5119 hold the fifth bits: two little-endian 32-bit
 *           words per row, word j (0, 1) of row r at byte 4096 + 512j + 4r, holding
 *           (code >> 4) of input 64g + 32j + 8u + i (u = 0..3, i = 0..7) at bit
 *           (4i + 4 + u) mod 32.
 *   scales: 128*SB bytes per tile at t*128*SB, SB bytes for row r at r*SB:
 *           NVFP4 (SB=4) byte i = E4M3 scale of inputs 64g+16i..+15;
 *           MXFP4 (SB=2) byte i = E8M0 scale of inputs 64g+32i..+31;
 *           MLX   (SB=4) fp16 s then fp16 b (little-endian) of the 64-input group;
 *           Q6_K  (SB=4) byte i = int8 scale of inputs 64g+16i..+15;
 *           Q5_0  (SB=4) fp16 d of inputs 64g+32i..+31 at bytes 2i..2i+1;
 *           Q5_1  (SB=8) fp16 d then fp16 m of inputs 64g+32i..+31 at bytes 4i..4i+3;
 *           Q5_K  (SB=3) one little-endian 24-bit value: sc of inputs 64g..64g+31 in bits
 *                 0..5, its mn in 6..11, sc and mn of 64g+32..64g+63 in 12..17, 18..23.
 *   aux   : Q6_K: fp16 d of inputs 256u..256u+255 for row r of row tile q at
 *           byte (q*(KG/4) + u)*256 + 2r.  Q5_K: fp16 d then fp16 dmin of those inputs
 *           at byte (q*(KG/4) + u)*512 + 4r.  NULL for the other formats.
 */
#ifndef QGEMV_H
#define QGEMV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  QG_FMT_MLX_AFFINE4_G64 = 1,
  QG_FMT_MXFP4 = 2,
  QG_FMT_NVFP4 = 3,
  QG_FMT_Q6K = 4,
  QG_FMT_Q5_0 = 5,
  QG_FMT_Q5_1 = 6,
  QG_FMT_Q5_K = 7
} qg_format;

typedef enum {
  QG_OK = 0,
  QG_ERR_INVALID_ARG = 1,        /* null pointer, bad size or enum, n/k not a multiple of the block */
  QG_ERR_UNSUPPORTED = 2,        /* valid request this build does not handle (e.g. m out of range) */
  QG_ERR_MISALIGNED = 3,         /* pointer not 16-byte aligned or leading dimension not a multiple of 8 */
  QG_ERR_WORKSPACE_TOO_SMALL = 4,
  QG_ERR_CUDA = 5,               /* a CUDA runtime call or a launch failed */
  QG_ERR_TIMEOUT = 6             /* a bounded device-side wait gave up (reported via qg_workspace_status) */
} qg_status;

typedef enum { QG_OUT_F32 = 0, QG_OUT_BF16 = 1 } qg_out_dtype;

/* A packed weight matrix in device memory (layout "T128x64" above).
 * n, k are the logical sizes; k must be a multiple of the format's block (64 MLX,
 * 32 MXFP4, 16 NVFP4, 256 Q6_K, 32 Q5_0 / Q5_1, 256 Q5_K).  tensor_scale is used by NVFP4 only and must be
 * 1.0f for the other formats. */
typedef struct {
  int32_t fmt;            /* qg_format */
  int32_t reserved;       /* must be 0 */
  int64_t n;
  int64_t k;
  const void* codes;      /* device, 16-byte aligned */
  const void* scales;     /* device, 16-byte aligned */
  const void* aux;        /* device, 16-byte aligned; Q6_K d, Q5_K (d, dmin), NULL otherwise */
  float tensor_scale;
  float reserved2;        /* must be 0 */
} qg_weight;

/* Human-readable name of a status code (static string, never NULL). */
const char* qg_status_str(int status);

/* Byte sizes of the packed codes / scales / aux buffers of an n x k matrix
 * (TurboEXL3 article §2.1 bits per weight; Q6_K operand PR #19: 1.04 GB for the
 * 248320 x 5120 output layer).  Host only; no GPU needed. */
qg_status qg_packed_sizes(int fmt, int64_t n, int64_t k,
                          size_t* codes_bytes, size_t* scales_bytes, size_t* aux_bytes);

/* Host-side packer: logical row-major arrays -> packed layout (host memory).
 *   logical_codes  : uint8 [n][k], one code per byte (0..15; 0..63 Q6_K; 0..31 5-bit)
 *   logical_scales : MLX fp16 s [n][k/64]; MXFP4 uint8 E8M0 [n][k/32];
 *                    NVFP4 uint8 E4M3 [n][k/16]; Q6_K int8 sc [n][k/16];
 *                    Q5_0 / Q5_1 fp16 d [n][k/32]; Q5_K uint8 (sc, mn) [n][k/32][2]
 *   logical_aux    : MLX fp16 b [n][k/64]; Q6_K fp16 d [n][k/256]; Q5_1 fp16 m [n][k/32];
 *                    Q5_K fp16 (d, dmin) [n][k/256][2]; NULL otherwise
 *   codes/scales/aux: outputs sized by qg_packed_sizes (aux NULL unless Q6_K or Q5_K).
 * Codes (or Q5_K sc / mn above 63) out of range return QG_ERR_INVALID_ARG.  No GPU
 * needed. */
qg_status qg_pack_host(int fmt, int64_t n, int64_t k,
                       const uint8_t* logical_codes, const void* logical_scales, const void* logical_aux,
                       void* codes, void* scales, void* aux);

/* Debug / test: dequantise the whole matrix into out [n][ldo] (device).
 *   QG_OUT_F32 : the exact weight rounded once to fp32 (NVFP4 includes the tensor scale).
 *   QG_OUT_BF16: the operand the prefill GEMM feeds the tensor cores: for MXFP4 /
 *                NVFP4 the block-scaled E2M1 value without the tensor scale (exact in
 *                bf16); for MLX / Q6_K / the 5-bit formats the fp32 weight rounded to
 *                bf16. */
qg_status qg_dequant(const qg_weight* w, int out_dtype, void* out, int64_t ldo, void* stream);

/* Workspace bytes qgemv needs for this shape on the current device (split-K
 * partial sums and per-row-tile tickets).  The workspace must be zero-filled
 * before its first use (qg_workspace_init); every successful call leaves it
 * ready for the next.  One workspace per stream: calls that overlap on the
 * GPU must not share it. */
size_t qg_gemv_workspace_size(int fmt, int64_t n, int64_t k, int m);

/* Zero a workspace of `bytes` bytes on `stream` (cudaMemsetAsync). */
qg_status qg_workspace_init(void* workspace, size_t bytes, void* stream);

/* Read (and clear) the device status word at the start of a workspace: QG_OK, or
 * QG_ERR_TIMEOUT if a bounded wait inside a kernel gave up.  Synchronises `stream`. */
qg_status qg_workspace_status(void* workspace, int* status, void* stream);

/* Quantized GEMV for 1..4 activation rows (speculative-verify widths):
 *   y[m][n] = bf16( sum_k w[n,k] * x[m][k] (+ residual[m][n]) ),  m = 0..m_rows-1.
 * Each weight is read from memory once for all rows (TurboEXL3 article §4.2: tokens
 * share one decode; §4.3: 1-4 rows in one launch, the last-arriving block of
 * an output tile finishes it).  residual may be NULL (ldr ignored).  x, residual
 * and y must not overlap.  m_rows outside 1..4 returns QG_ERR_UNSUPPORTED. */
qg_status qgemv(const qg_weight* w, const void* x, int m_rows, int64_t ldx,
                const void* residual, int64_t ldr, void* y, int64_t ldy,
                void* workspace, size_t workspace_bytes, void* stream);

/* Workspace bytes qgemm needs: the qgemv size for 1..4 rows, else 256 (status word). */
size_t qg_gemm_workspace_size(int fmt, int64_t n, int64_t k, int m);

/* Quantized GEMM for any number of activation rows (tokens), dispatching by rows
 * (TurboEXL3 article §4.3, a path per row count): 1..4 rows run qgemv; 5..128 rows the
 * small-token tensor-core GEMM (one token tile of 16 / 32 / 64 / 128); more rows the
 * prefill GEMM with 256-token tiles.  Both tensor-core GEMMs decode each 128 x 64 weight
 * slice once, on chip, into bf16 operands in tensor memory and multiply it against the
 * tile's tokens (tcgen05, fp32 accumulation in tensor memory), splitting K over a cluster
 * when the tiles fill less than half the GPU -- TurboEXL3 article §4.1: each weight
 * decoded once and used for many tokens; no dequantised copy of the weights is written
 * to device memory.
 *   y[t][n] = bf16( sum_k w[n,k] * x[t][k] (+ residual[t][n]) ),  t = 0..m_rows-1.
 * Same argument rules as qgemv; the workspace holds the device status word
 * (qg_workspace_status) and must be zero-filled before first use. */
qg_status qgemm(const qg_weight* w, const void* x, int64_t m_rows, int64_t ldx,
                const void* residual, int64_t ldr, void* y, int64_t ldy,
                void* workspace, size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------ W4A4: NVFP4 activations
 * TurboEXL3 article §2.2: besides W4A16, an NVFP4 checkpoint can run W4A4, quantising the
 * activations to NVFP4 as well during the forward pass, with one scale per 16 values.
 * The pages leave the activations' tensor scale open: here it is the caller's fp32
 * act_scale (finite, > 0; a calibrated constant).  Per block of 16 consecutive values
 * of a row along K, each step one fp32 operation rounded to nearest even:
 *   S    = E4M3( amax / (6 * act_scale) )            nearest even, saturating at 448
 *   den  = E4M3(S) * act_scale
 *   code = E2M1( x / den )   (x * 0 when den == 0)    nearest even, saturating at 6,
 *                                                     sign bit from x (-0 gives 8)
 * Activations must be finite. */

/* Quantise bf16 activations x [m][ldx] (k a multiple of 16; x 16-byte aligned, ldx a
 * multiple of 8) to NVFP4.  Outputs, device memory, each optional (NULL: not written):
 *   codes  : uint8 [m][ldc], two E2M1 codes per byte, value k in byte k/2, the even k in
 *            the low nibble (ldc >= k/2, a multiple of 8; 16-byte aligned);
 *   scales : uint8 [m][lds], the E4M3 byte of block k/16 (lds >= k/16);
 *   xe     : bf16 [m][lde], E4M3(S) * E2M1(code) -- exact in bf16, act_scale left out --
 *            the operand a bf16 GEMM multiplies (lde >= k, a multiple of 8; 16-byte aligned).
 * m_rows * k/16 must stay below 2^31 (QG_ERR_UNSUPPORTED otherwise).  Argument errors
 * return before anything is launched. */
qg_status qg_quant_act_nvfp4(const void* x, int64_t m_rows, int64_t k, int64_t ldx, float act_scale,
                             uint8_t* codes, int64_t ldc, uint8_t* scales, int64_t lds,
                             void* xe, int64_t lde, void* stream);

/* Workspace bytes qgemm_w4a4 needs: the qgemm workspace of the same shape (first, so the
 * status word stays at offset 0) plus m_rows x k bf16 quantised activations.  0 for a
 * format other than NVFP4. */
size_t qgemm_w4a4_workspace_size(int fmt, int64_t n, int64_t k, int64_t m_rows);

/* W4A4 GEMM for an NVFP4 weight (other formats: QG_ERR_UNSUPPORTED):
 *   y[t][n] = bf16( sum_k w[n,k] * xq[t][k] (+ residual[t][n]) ),
 *   xq[t][k] = act_scale * E4M3(S) * E2M1(code)  (qg_quant_act_nvfp4 above).
 * qg_quant_act_nvfp4 writes the expansion into the workspace, then qgemm multiplies it
 * (the GEMV for 1..4 rows, the tensor-core GEMMs above that) with act_scale folded into
 * the weight's tensor scale for the epilogue.  Both operands are exact in bf16, so each
 * product is exactly that of the two FP4 values and their scales; the tensor cores run
 * the bf16 kind, not a block-scaled FP4 one.  Same argument rules and workspace contract
 * as qgemm (zero-filled before first use); act_scale * tensor_scale must be a finite
 * positive fp32. */
qg_status qgemm_w4a4(const qg_weight* w, const void* x, int64_t m_rows, int64_t ldx, float act_scale,
                     const void* residual, int64_t ldr, void* y, int64_t ldy,
                     void* workspace, size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------ mixture of experts
 * A layer of n_experts routed experts plus an optional shared expert, each an FFN with
 * gate/up (2F x H: rows 0..F-1 gate, F..2F-1 up) and down (H x F) quantized matrices.
 * The routed experts' packed matrices lie back to back: expert e's gate/up codes start
 * at gu_codes + e * (codes bytes of one 2F x H matrix), and likewise for every array
 * (sizes from qg_packed_sizes).  Limits: n_experts <= 512, topk <= 16. */
typedef struct {
  int32_t fmt;              /* qg_format of every matrix */
  int32_t n_experts;
  int64_t hidden;           /* H */
  int64_t ffn;              /* F */
  const void* gu_codes;     /* device, n_experts packed 2F x H matrices */
  const void* gu_scales;
  const void* gu_aux;       /* Q6_K d, else NULL */
  const void* dn_codes;     /* device, n_experts packed H x F matrices */
  const void* dn_scales;
  const void* dn_aux;
  float tensor_scale;       /* NVFP4 tensor scale of the routed experts, else 1.0f */
  int32_t has_shared;       /* 1: the shared expert below joins every token (weight 1, or its
                               sigmoid gate when the call passes gate logits) */
  qg_weight shared_gate_up; /* 2F x H */
  qg_weight shared_down;    /* H x F */
} qg_moe_layer;

/* Router workspace bytes for t tokens. */
size_t qmoe_route_workspace_size(int64_t t, int n_experts, int topk);

/* Router (TurboEXL3 article §4.1 "Route", §4.2 top-k and softmax): for each token the
 * topk experts by fp32 logit (ties to the lower index) and the softmax of the kept logits,
 *   topk_ids [t][topk] int32, topk_w [t][topk] fp32 (device),
 * and, in route_ws, the (token, slot) pairs grouped by expert -- experts ascending, tokens
 * ascending within an expert -- with counts, offsets, the active experts and a tile
 * table; deterministic, one launch for up to 32 tokens.  logits: fp32 [t][n_experts]. */
qg_status qmoe_route(const float* logits, int64_t t, int n_experts, int topk,
                     int32_t* topk_ids, float* topk_w, void* route_ws, size_t route_ws_bytes, void* stream);

/* Workspace bytes qmoe_ffn needs for t tokens on the current device. */
size_t qmoe_workspace_size(const qg_moe_layer* layer, int64_t t, int topk);

/* One MoE FFN layer after qmoe_route on the same logits:
 *   out[t] = bf16( sum_j topk_w[t][j] * down_e(h) + g_t * shared(h) ),
 *   g_t = sigmoid(shared_gate[t]) = 1 / (1 + exp(-shared_gate[t])) in fp32 when the
 *   shared expert's gate logits are given (TurboEXL3 article §4.2: the shared expert's
 *   sigmoid gate), else 1.  shared_gate: fp32 [t] on the device, or NULL; non-NULL
 *   without a shared expert is QG_ERR_INVALID_ARG.  Like the router's logits, the gate
 *   logit (the 1-output projection of x) is the caller's input.  The finish forms the
 *   weighted sum in fp32 and rounds it to bf16 once; its terms, the per-(token, expert) down
 *   outputs, are fp32 at 1..4 tokens and rounded to bf16 (the GEMM's output type) in the
 *   prefill chain.
 *   h = bf16(silu(gate) * up) per (token, expert), gate = rows 0..F-1 and up = rows
 *   F..2F-1 of the expert's 2F x H gate/up weight.
 * 1..4 tokens (decode / speculative verify; TurboEXL3 article §4.2): three launches --
 *   gate/up as one grouped GEMV over the active experts that reads each expert's weights
 *   once for all its tokens, with the shared expert as one more group of all the tokens;
 *   down, whose blocks compute the mid (h = bf16(silu(gate) * up)) while staging their
 *   inputs; finish.
 * More tokens (prefill; §4.1): three launches -- one grouped tensor-core GEMM over the
 *   router's tile table for gate/up whose epilogue runs the mid, the same GEMM for down
 *   (bf16 outputs per pair), and the finish; the shared expert runs as extra tiles of both
 *   GEMMs.  Needs
 *   ffn % 128 == 0 and hidden % 8 == 0, else QG_ERR_UNSUPPORTED.
 * x: bf16 [t][ldx] (H inputs); out: bf16 [t][ldo].  The workspace (qmoe_workspace_size
 * bytes for this t) must be zero-filled before first use and not be shared by
 * overlapping calls.  Deterministic: no atomics in any sum. */
qg_status qmoe_ffn(const qg_moe_layer* layer, const void* x, int64_t t, int64_t ldx, int topk,
                   const float* topk_w, const float* shared_gate, const void* route_ws, void* out, int64_t ldo,
                   void* workspace, size_t workspace_bytes, void* stream);

/* Router and FFN in one call: qmoe_route on `logits` (fp32 [t][n_experts], device) followed
 * by qmoe_ffn, with the same outputs -- topk_ids, topk_w and route_ws as qmoe_route stores
 * them, out as qmoe_ffn computes it, bit for bit.  At 1..4 tokens the gate/up launch routes
 * the tokens itself (every CTA computes the same small table; the first also stores the
 * router's outputs), so the layer takes three launches instead of four (TurboEXL3 article
 * §4.2: the router's top-k and softmax run inside the FFN chain); needs t * topk <= 64.
 * More tokens: the router's launches, then the prefill chain.  Same arguments, limits and
 * errors as qmoe_route and qmoe_ffn together. */
qg_status qmoe_forward(const qg_moe_layer* layer, const void* x, int64_t t, int64_t ldx, const float* logits,
                       int topk, const float* shared_gate, int32_t* topk_ids, float* topk_w, void* route_ws,
                       size_t route_ws_bytes, void* out, int64_t ldo, void* workspace, size_t workspace_bytes,
                       void* stream);

/* The MoE FFN one stage at a time (the grouped GEMM of the two stages, for callers that
 * keep h or run something between the stages); the same results as qmoe_ffn, bit for bit.
 * rows = t * topk + (has_shared ? t : 0).
 *   QG_MOE_GATE_UP_SWIGLU: in = x bf16 [t][ldi] (H inputs); out = h bf16 [rows][ldo] (F
 *       columns): row p < t*topk is the p-th (token, slot) pair in the router's grouped order
 *       (experts ascending, tokens ascending within an expert), h = bf16(silu(gate) * up)
 *       with the gate/up rows of that pair's expert; row t*topk + i is token i's shared-expert
 *       h.  topk_w may be NULL.
 *   QG_MOE_DOWN_COMBINE: in = h [rows][ldi] as above; out = bf16 [t][ldo] (H columns),
 *       out[i] = bf16( sum_j topk_w[i][j] * down_e(h of pair (i, j)) + g_i * shared down(h) ),
 *       g_i from shared_gate as in qmoe_ffn (NULL: 1).  The gate/up stage ignores
 *       shared_gate.
 * route_ws from qmoe_route on the same t, n_experts and topk.  The workspace holds
 * qgemm_grouped_workspace_size bytes (the qmoe_ffn size), zero-filled before first use.
 * Same limits and errors as qmoe_ffn; stage values other than the two return
 * QG_ERR_INVALID_ARG. */
typedef enum { QG_MOE_GATE_UP_SWIGLU = 1, QG_MOE_DOWN_COMBINE = 2 } qg_moe_stage;
size_t qgemm_grouped_workspace_size(const qg_moe_layer* layer, int64_t t, int topk, int stage);
qg_status qgemm_grouped(const qg_moe_layer* layer, int stage, const void* in, int64_t t, int64_t ldi, int topk,
                        const float* topk_w, const float* shared_gate, const void* route_ws, void* out, int64_t ldo,
                        void* workspace, size_t workspace_bytes, void* stream);

/* Workspace-free variant of qgemv, for callers that cannot allocate device memory:
 * plugins hosted by a runtime that owns all of the GPU's memory and gives them no
 * allocator, and code on paths where cudaMalloc's implicit device synchronisation is not
 * acceptable.  The source pages have no counterpart; it exists for such callers only.
 * Same arguments and results as qgemv, minus the workspace.  The split-K scratch lives in
 * a fixed device array of QG_STATIC_WORKSPACE_BYTES inside the library, present on every
 * GPU that loads the library until the process exits.  The first call on a device looks
 * up that array's address (make it before any stream capture; a failed lookup returns
 * QG_ERR_CUDA and is tried again on the next call).  Every call clears the array's
 * row-tile tickets; its status word is sticky, as a workspace's is, and a bounded wait
 * that gave up (QG_ERR_TIMEOUT) is read with qgemv_static_ws_status.  All calls share the
 * array, so calls that overlap on the GPU race -- serialise them (one stream).  Shapes
 * needing more scratch than the array holds return QG_ERR_WORKSPACE_TOO_SMALL; nothing is
 * allocated. */
#define QG_STATIC_WORKSPACE_BYTES (4u << 20)
qg_status qgemv_static_ws(const qg_weight* w, const void* x, int m_rows, int64_t ldx,
                          const void* residual, int64_t ldr, void* y, int64_t ldy, void* stream);
/* Status word of the array qgemv_static_ws uses on the current device, as
 * qg_workspace_status reads a workspace's: synchronises `stream`, stores the word in
 * *status (QG_OK, or QG_ERR_TIMEOUT after a wait gave up) and clears it. */
qg_status qgemv_static_ws_status(int* status, void* stream);

/* Self-test of the shared failure path: launches one CTA whose mbarrier wait nothing will
 * complete; after the library's wait limit (2 s) the kernel records QG_ERR_TIMEOUT in the
 * workspace's status word and returns -- no fault, no hang, the context stays usable.
 * Read the result with qg_workspace_status.  The pages have no counterpart; it exists to
 * test failure detection.  workspace: device, 16-byte aligned, >= 4 bytes. */
qg_status qg_selftest_wait_timeout(void* workspace, size_t workspace_bytes, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* QGEMV_H */
