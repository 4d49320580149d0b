// C ABI entry points: argument validation on the host, device attribute cache,
// dispatch to the kernel launchers.  No entry point allocates memory.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <mutex>

#include "qg_internal.h"
#include "qg_route.h"

namespace qg {

namespace {
constexpr int kMaxDevices = 64;
std::once_flag g_once[kMaxDevices];
DeviceInfo g_info[kMaxDevices];
bool g_ok[kMaxDevices];

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
}  // namespace

bool device_info(int device, DeviceInfo* out) {
  if (device < 0 || device >= kMaxDevices) return false;
  std::call_once(g_once[device], [device] {
    int sms = 0, smem = 0;
    g_ok[device] = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) == cudaSuccess &&
                   cudaDeviceGetAttribute(&smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, device) == cudaSuccess;
    g_info[device].sms = sms;
    g_info[device].max_smem_optin = smem;
  });
  if (!g_ok[device]) return false;
  *out = g_info[device];
  return true;
}

bool current_device_info(DeviceInfo* out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  return device_info(dev, out);
}

static int check_weight(const qg_weight* w, Geometry* g) {
  if (!w) return QG_ERR_INVALID_ARG;
  if (w->reserved != 0 || w->reserved2 != 0.0f) return QG_ERR_INVALID_ARG;
  if (!geometry(w->fmt, w->n, w->k, g)) return QG_ERR_INVALID_ARG;
  if (!w->codes || !w->scales) return QG_ERR_INVALID_ARG;
  if ((w->fmt == QG_FMT_Q6K || w->fmt == QG_FMT_Q5_K) && !w->aux) return QG_ERR_INVALID_ARG;
  if (w->fmt != QG_FMT_NVFP4 && w->tensor_scale != 1.0f) return QG_ERR_INVALID_ARG;
  if (!aligned16(w->codes) || !aligned16(w->scales) || (w->aux && !aligned16(w->aux))) return QG_ERR_MISALIGNED;
  return QG_OK;
}

int check_gemv_call(const qg_weight* w, const void* x, int m, int64_t ldx, const void* residual, int64_t ldr,
                    const void* y, int64_t ldy, Geometry* g) {
  int st = check_weight(w, g);
  if (st != QG_OK) return st;
  if (m < 1 || m > 4) return QG_ERR_UNSUPPORTED;
  if (!x || !y) return QG_ERR_INVALID_ARG;
  if (ldx < w->k || ldy < w->n || (residual && ldr < w->n)) return QG_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(y) || (residual && !aligned16(residual))) return QG_ERR_MISALIGNED;
  if (ldx % 8 || ldy % 8 || (residual && ldr % 8)) return QG_ERR_MISALIGNED;
  return QG_OK;
}

}  // namespace qg

using namespace qg;

extern "C" const char* qg_status_str(int status) {
  switch (status) {
    case QG_OK: return "QG_OK";
    case QG_ERR_INVALID_ARG: return "QG_ERR_INVALID_ARG";
    case QG_ERR_UNSUPPORTED: return "QG_ERR_UNSUPPORTED";
    case QG_ERR_MISALIGNED: return "QG_ERR_MISALIGNED";
    case QG_ERR_WORKSPACE_TOO_SMALL: return "QG_ERR_WORKSPACE_TOO_SMALL";
    case QG_ERR_CUDA: return "QG_ERR_CUDA";
    case QG_ERR_TIMEOUT: return "QG_ERR_TIMEOUT";
    default: return "QG_ERR_UNKNOWN";
  }
}

extern "C" qg_status qg_dequant(const qg_weight* w, int out_dtype, void* out, int64_t ldo, void* stream) {
  Geometry g;
  int st = check_weight(w, &g);
  if (st != QG_OK) return (qg_status)st;
  if (!out || (out_dtype != QG_OUT_F32 && out_dtype != QG_OUT_BF16) || ldo < w->k) return QG_ERR_INVALID_ARG;
  if (!aligned16(out) || ldo % 8 != 0) return QG_ERR_MISALIGNED;
  return (qg_status)launch_dequant(g, w, out_dtype, out, ldo, stream);
}

extern "C" size_t qg_gemv_workspace_size(int fmt, int64_t n, int64_t k, int m) {
  Geometry g;
  if (!geometry(fmt, n, k, &g) || m < 1 || m > 4) return 0;
  DeviceInfo dev;
  if (!current_device_info(&dev)) return 0;
  GemvPlan p;
  if (!plan_gemv(g, m, dev, &p)) return 0;
  return p.ws_bytes;
}

extern "C" qg_status qg_workspace_init(void* workspace, size_t bytes, void* stream) {
  if (!workspace && bytes) return QG_ERR_INVALID_ARG;
  if (!bytes) return QG_OK;
  return cudaMemsetAsync(workspace, 0, bytes, static_cast<cudaStream_t>(stream)) == cudaSuccess ? QG_OK
                                                                                                 : QG_ERR_CUDA;
}

extern "C" qg_status qgemv(const qg_weight* w, const void* x, int m, int64_t ldx, const void* residual, int64_t ldr,
                           void* y, int64_t ldy, void* workspace, size_t workspace_bytes, void* stream) {
  Geometry g;
  int st = check_gemv_call(w, x, m, ldx, residual, ldr, y, ldy, &g);
  if (st != QG_OK) return (qg_status)st;
  if (!workspace) return QG_ERR_INVALID_ARG;
  if (!aligned16(workspace)) return QG_ERR_MISALIGNED;
  DeviceInfo dev;
  if (!current_device_info(&dev)) return QG_ERR_CUDA;
  GemvPlan p;
  if (!plan_gemv(g, m, dev, &p)) return QG_ERR_UNSUPPORTED;
  if (workspace_bytes < p.ws_bytes) return QG_ERR_WORKSPACE_TOO_SMALL;
  return (qg_status)launch_gemv(g, w, x, m, ldx, residual, ldr, y, ldy, workspace, p, stream);
}

extern "C" qg_status qg_workspace_status(void* workspace, int* status, void* stream) {
  if (!workspace || !status) return QG_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int v = 0;
  if (cudaMemcpyAsync(&v, workspace, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess) return QG_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return QG_ERR_CUDA;
  if (v != 0 && cudaMemsetAsync(workspace, 0, sizeof(int), s) != cudaSuccess) return QG_ERR_CUDA;
  *status = v;
  return QG_OK;
}

extern "C" size_t qg_gemm_workspace_size(int fmt, int64_t n, int64_t k, int m) {
  if (m >= 1 && m <= 4) return qg_gemv_workspace_size(fmt, n, k, m);
  Geometry g;
  if (!geometry(fmt, n, k, &g) || m < 1) return 0;
  return kWsHeader;
}

extern "C" qg_status qgemm(const qg_weight* w, const void* x, int64_t m, int64_t ldx, const void* residual,
                           int64_t ldr, void* y, int64_t ldy, void* workspace, size_t workspace_bytes, void* stream) {
  if (m >= 1 && m <= 4)  // 1..4 rows: the GEMV reads each weight once for all rows
    return qgemv(w, x, (int)m, ldx, residual, ldr, y, ldy, workspace, workspace_bytes, stream);
  Geometry g;
  int st = check_weight(w, &g);
  if (st != QG_OK) return (qg_status)st;
  if (m < 1) return QG_ERR_UNSUPPORTED;
  if (!x || !y || !workspace) return QG_ERR_INVALID_ARG;
  if (ldx < w->k || ldy < w->n || (residual && ldr < w->n)) return QG_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(y) || (residual && !aligned16(residual)) || !aligned16(workspace))
    return QG_ERR_MISALIGNED;
  if (ldx % 8 || ldy % 8 || (residual && ldr % 8)) return QG_ERR_MISALIGNED;
  if (workspace_bytes < kWsHeader) return QG_ERR_WORKSPACE_TOO_SMALL;
  if ((m + 255) / 256 > 65535 || g.nt > 0x7FFFFFFF) return QG_ERR_UNSUPPORTED;
  if (m <= kSmallGemmMaxRows) {
    DeviceInfo dev;
    if (!current_device_info(&dev)) return QG_ERR_CUDA;
    return (qg_status)launch_gemm_small(g, w, x, m, ldx, residual, ldr, y, ldy, workspace, dev, stream);
  }
  return (qg_status)launch_prefill(g, w, x, m, ldx, residual, ldr, y, ldy, workspace, stream);
}

extern "C" qg_status qg_quant_act_nvfp4(const void* x, int64_t m, int64_t k, int64_t ldx, float act_scale,
                                        uint8_t* codes, int64_t ldc, uint8_t* scales, int64_t lds, void* xe,
                                        int64_t lde, void* stream) {
  if (!x || m < 1 || k < 16 || k % 16 || !(act_scale > 0.0f) || !std::isfinite(act_scale)) return QG_ERR_INVALID_ARG;
  if (ldx < k || (codes && ldc < k / 2) || (scales && lds < k / 16) || (xe && lde < k)) return QG_ERR_INVALID_ARG;
  if (!aligned16(x) || ldx % 8 || (codes && (!aligned16(codes) || ldc % 8)) || (xe && (!aligned16(xe) || lde % 8)))
    return QG_ERR_MISALIGNED;
  if (m > 0x7FFFFFFF / (k / 16)) return QG_ERR_UNSUPPORTED;  // 2^31 blocks of 16 at most
  return (qg_status)launch_quant_act_nvfp4(x, m, k, ldx, act_scale, codes, ldc, scales, lds, xe, lde, stream);
}

// W4A4 workspace: the qgemm workspace first (its status word at offset 0), then the
// quantised activations' bf16 expansion, m rows of k rounded up to 8.
static size_t w4a4_gemm_part(int fmt, int64_t n, int64_t k, int64_t m) {
  const size_t g = qg_gemm_workspace_size(fmt, n, k, (int)std::min<int64_t>(m, 1 << 30));
  return g ? (g + 255) / 256 * 256 : 0;
}

// 5 or more rows: the block-scaled FP4 GEMM, its workspace the status header, then the
// quantised activations' codes [m][w4a4_ldc] and E4M3 scales [m][w4a4_lds].
static int64_t w4a4_ldc(int64_t k) { return (k / 2 + 15) / 16 * 16; }
static int64_t w4a4_lds(int64_t k) { return (k / 16 + 15) / 16 * 16; }
static size_t w4a4_fp4_codes_off() { return kWsHeader; }
static size_t w4a4_fp4_scales_off(int64_t k, int64_t m) {
  return (w4a4_fp4_codes_off() + (size_t)m * (size_t)w4a4_ldc(k) + 255) / 256 * 256;
}

extern "C" size_t qgemm_w4a4_workspace_size(int fmt, int64_t n, int64_t k, int64_t m) {
  if (fmt != QG_FMT_NVFP4 || m < 1) return 0;
  Geometry g;
  if (!geometry(fmt, n, k, &g)) return 0;
  if (m >= 5) return w4a4_fp4_scales_off(k, m) + (size_t)m * (size_t)w4a4_lds(k);
  const size_t gp = w4a4_gemm_part(fmt, n, k, m);
  return gp ? gp + (size_t)m * (size_t)((k + 7) / 8 * 8) * 2 : 0;
}

extern "C" qg_status qgemm_w4a4(const qg_weight* w, const void* x, int64_t m, int64_t ldx, float act_scale,
                                const void* residual, int64_t ldr, void* y, int64_t ldy, void* workspace,
                                size_t workspace_bytes, void* stream) {
  // every check qgemm makes, before anything is launched
  Geometry g;
  int st = check_weight(w, &g);
  if (st != QG_OK) return (qg_status)st;
  if (w->fmt != QG_FMT_NVFP4 || m < 1) return QG_ERR_UNSUPPORTED;
  if (!x || !y || !workspace || !(act_scale > 0.0f) || !std::isfinite(act_scale)) return QG_ERR_INVALID_ARG;
  qg_weight w_scaled = *w;  // the activation tensor scale joins the weight's in the GEMM's epilogue
  w_scaled.tensor_scale = w->tensor_scale * act_scale;
  if (!(w_scaled.tensor_scale > 0.0f) || !std::isfinite(w_scaled.tensor_scale)) return QG_ERR_INVALID_ARG;
  if (ldx < w->k || ldy < w->n || (residual && ldr < w->n)) return QG_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(y) || (residual && !aligned16(residual)) || !aligned16(workspace))
    return QG_ERR_MISALIGNED;
  if (ldx % 8 || ldy % 8 || (residual && ldr % 8)) return QG_ERR_MISALIGNED;
  if ((m + 255) / 256 > 65535 || g.nt > 0x7FFFFFFF || m > 0x7FFFFFFF / (w->k / 16)) return QG_ERR_UNSUPPORTED;
  const size_t need = qgemm_w4a4_workspace_size(w->fmt, w->n, w->k, m);
  if (!need) {  // 1..4 rows: the GEMV's plan needs the device; none, or no plan for this shape
    DeviceInfo dev;
    return current_device_info(&dev) ? QG_ERR_UNSUPPORTED : QG_ERR_CUDA;
  }
  if (workspace_bytes < need) return QG_ERR_WORKSPACE_TOO_SMALL;
  if (m >= 5) {  // quantise to codes and scales, then the block-scaled FP4 GEMM multiplies them
    uint8_t* codes = static_cast<uint8_t*>(workspace) + w4a4_fp4_codes_off();
    uint8_t* scales = static_cast<uint8_t*>(workspace) + w4a4_fp4_scales_off(w->k, m);
    st = launch_quant_act_nvfp4(x, m, w->k, ldx, act_scale, codes, w4a4_ldc(w->k), scales, w4a4_lds(w->k), nullptr, 0,
                                stream);
    if (st != QG_OK) return (qg_status)st;
    return (qg_status)launch_gemm_fp4(g, w, act_scale, codes, w4a4_ldc(w->k), scales, w4a4_lds(w->k), m, residual,
                                      ldr, y, ldy, workspace, stream);
  }
  const size_t off = w4a4_gemm_part(w->fmt, w->n, w->k, m);
  void* xe = static_cast<char*>(workspace) + off;
  const int64_t lde = (w->k + 7) / 8 * 8;
  st = launch_quant_act_nvfp4(x, m, w->k, ldx, act_scale, nullptr, 0, nullptr, 0, xe, lde, stream);
  if (st != QG_OK) return (qg_status)st;
  return qgemm(&w_scaled, xe, m, lde, residual, ldr, y, ldy, workspace, off, stream);
}

extern "C" size_t qmoe_route_workspace_size(int64_t t, int n_experts, int topk) {
  if (t < 1 || n_experts < 1 || n_experts > kMaxExperts || topk < 1 || topk > kMaxTopk || topk > n_experts) return 0;
  return route_layout(t, n_experts, topk).total;
}

extern "C" qg_status qmoe_route(const float* logits, int64_t t, int n_experts, int topk, int32_t* topk_ids,
                                float* topk_w, void* route_ws, size_t route_ws_bytes, void* stream) {
  if (t < 1 || n_experts < 1 || topk < 1 || topk > n_experts) return QG_ERR_INVALID_ARG;
  if (n_experts > kMaxExperts || topk > kMaxTopk || t * topk > 0x7FFFFFFF) return QG_ERR_UNSUPPORTED;
  if (!logits || !topk_ids || !topk_w || !route_ws) return QG_ERR_INVALID_ARG;
  if (!aligned16(logits) || !aligned16(topk_ids) || !aligned16(topk_w) || !aligned16(route_ws))
    return QG_ERR_MISALIGNED;
  if (route_ws_bytes < route_layout(t, n_experts, topk).total) return QG_ERR_WORKSPACE_TOO_SMALL;
  return (qg_status)launch_route(logits, t, n_experts, topk, topk_ids, topk_w, route_ws, stream);
}

static int check_moe(const qg_moe_layer* m, int64_t t, int topk, Geometry* gu, Geometry* dn) {
  if (!m || t < 1 || topk < 1) return QG_ERR_INVALID_ARG;
  if (m->n_experts < 1 || topk > m->n_experts) return QG_ERR_INVALID_ARG;
  if (m->n_experts > kMaxExperts || topk > kMaxTopk) return QG_ERR_UNSUPPORTED;
  if (is_q5(m->fmt)) return QG_ERR_UNSUPPORTED;  // the 5-bit formats run on the dense paths only
  if (!geometry(m->fmt, 2 * m->ffn, m->hidden, gu) || !geometry(m->fmt, m->hidden, m->ffn, dn))
    return QG_ERR_INVALID_ARG;
  if (!m->gu_codes || !m->gu_scales || !m->dn_codes || !m->dn_scales) return QG_ERR_INVALID_ARG;
  if (m->fmt == QG_FMT_Q6K && (!m->gu_aux || !m->dn_aux)) return QG_ERR_INVALID_ARG;
  if (m->fmt != QG_FMT_NVFP4 && m->tensor_scale != 1.0f) return QG_ERR_INVALID_ARG;
  if (!aligned16(m->gu_codes) || !aligned16(m->gu_scales) || !aligned16(m->dn_codes) || !aligned16(m->dn_scales) ||
      (m->gu_aux && !aligned16(m->gu_aux)) || (m->dn_aux && !aligned16(m->dn_aux)))
    return QG_ERR_MISALIGNED;
  if (m->has_shared) {
    Geometry g1, g2;
    int st = check_weight(&m->shared_gate_up, &g1);
    if (st != QG_OK) return st;
    st = check_weight(&m->shared_down, &g2);
    if (st != QG_OK) return st;
    if (m->shared_gate_up.fmt != m->fmt || m->shared_down.fmt != m->fmt || g1.n != gu->n || g1.k != gu->k ||
        g2.n != dn->n || g2.k != dn->k)
      return QG_ERR_INVALID_ARG;
  }
  return QG_OK;
}

extern "C" size_t qmoe_workspace_size(const qg_moe_layer* layer, int64_t t, int topk) {
  Geometry gu, dn;
  if (check_moe(layer, t, topk, &gu, &dn) != QG_OK) return 0;
  DeviceInfo dev;
  if (!current_device_info(&dev)) return 0;
  return moe_layout(gu, dn, t, layer->n_experts, topk, dev.sms).total;
}

extern "C" qg_status qmoe_ffn(const qg_moe_layer* layer, const void* x, int64_t t, int64_t ldx, int topk,
                              const float* topk_w, const float* shared_gate, const void* route_ws, void* out,
                              int64_t ldo, void* workspace, size_t workspace_bytes, void* stream) {
  Geometry gu, dn;
  int st = check_moe(layer, t, topk, &gu, &dn);
  if (st != QG_OK) return (qg_status)st;
  if (!x || !topk_w || !route_ws || !out || !workspace) return QG_ERR_INVALID_ARG;
  if (shared_gate && !layer->has_shared) return QG_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(shared_gate) % 4) return QG_ERR_MISALIGNED;
  // the prefill chain pairs gate rows f.. with up rows F+f.. inside one 128-row tile and
  // finishes eight features at a time
  if (t > 4 && (layer->ffn % 128 != 0 || layer->hidden % 8 != 0)) return QG_ERR_UNSUPPORTED;
  if (t * (int64_t)(topk + 1) >= ((int64_t)1 << 31)) return QG_ERR_UNSUPPORTED;
  if (ldx < layer->hidden || ldo < layer->hidden) return QG_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(out) || !aligned16(workspace) || !aligned16(route_ws) || !aligned16(topk_w))
    return QG_ERR_MISALIGNED;
  if (ldx % 8 || ldo % 8) return QG_ERR_MISALIGNED;
  DeviceInfo dev;
  if (!current_device_info(&dev)) return QG_ERR_CUDA;
  if (workspace_bytes < moe_layout(gu, dn, t, layer->n_experts, topk, dev.sms).total)
    return QG_ERR_WORKSPACE_TOO_SMALL;
  if (t > 4)
    return (qg_status)launch_moe_prefill(layer, gu, dn, x, t, ldx, topk, topk_w, shared_gate, route_ws, out, ldo,
                                         workspace, dev, stream, kMoeAll);
  return (qg_status)launch_moe_decode(layer, gu, dn, x, t, ldx, topk, topk_w, shared_gate, route_ws, out, ldo,
                                      workspace, dev, stream, kMoeAll);
}

extern "C" size_t qgemm_grouped_workspace_size(const qg_moe_layer* layer, int64_t t, int topk, int stage) {
  if (stage != QG_MOE_GATE_UP_SWIGLU && stage != QG_MOE_DOWN_COMBINE) return 0;
  return qmoe_workspace_size(layer, t, topk);
}

extern "C" qg_status qgemm_grouped(const qg_moe_layer* layer, int stage, const void* in, int64_t t, int64_t ldi,
                                   int topk, const float* topk_w, const float* shared_gate, const void* route_ws,
                                   void* out, int64_t ldo, void* workspace, size_t workspace_bytes, void* stream) {
  Geometry gu, dn;
  int st = check_moe(layer, t, topk, &gu, &dn);
  if (st != QG_OK) return (qg_status)st;
  if (stage != QG_MOE_GATE_UP_SWIGLU && stage != QG_MOE_DOWN_COMBINE) return QG_ERR_INVALID_ARG;
  if (!in || !route_ws || !out || !workspace || (stage == QG_MOE_DOWN_COMBINE && !topk_w)) return QG_ERR_INVALID_ARG;
  if (shared_gate && !layer->has_shared) return QG_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(shared_gate) % 4) return QG_ERR_MISALIGNED;
  if (stage == QG_MOE_GATE_UP_SWIGLU) shared_gate = nullptr;
  if (t > 4 && (layer->ffn % 128 != 0 || layer->hidden % 8 != 0)) return QG_ERR_UNSUPPORTED;
  if (t * (int64_t)(topk + 1) >= ((int64_t)1 << 31)) return QG_ERR_UNSUPPORTED;
  // gate/up: in = x [t][H], out = h [rows][F]; down: in = h [rows][F], out = [t][H]
  const int64_t in_cols = stage == QG_MOE_GATE_UP_SWIGLU ? layer->hidden : layer->ffn;
  const int64_t out_cols = stage == QG_MOE_GATE_UP_SWIGLU ? layer->ffn : layer->hidden;
  if (ldi < in_cols || ldo < out_cols) return QG_ERR_INVALID_ARG;
  if (!aligned16(in) || !aligned16(out) || !aligned16(workspace) || !aligned16(route_ws) ||
      (topk_w && !aligned16(topk_w)))
    return QG_ERR_MISALIGNED;
  if (ldi % 8 || ldo % 8) return QG_ERR_MISALIGNED;
  DeviceInfo dev;
  if (!current_device_info(&dev)) return QG_ERR_CUDA;
  if (workspace_bytes < moe_layout(gu, dn, t, layer->n_experts, topk, dev.sms).total)
    return QG_ERR_WORKSPACE_TOO_SMALL;
  const int ms = stage == QG_MOE_GATE_UP_SWIGLU ? kMoeGateUp : kMoeDown;
  if (t > 4)
    return (qg_status)launch_moe_prefill(layer, gu, dn, in, t, ldi, topk, topk_w, shared_gate, route_ws, out, ldo,
                                         workspace, dev, stream, ms);
  return (qg_status)launch_moe_decode(layer, gu, dn, in, t, ldi, topk, topk_w, shared_gate, route_ws, out, ldo,
                                      workspace, dev, stream, ms);
}

extern "C" qg_status qmoe_forward(const qg_moe_layer* layer, const void* x, int64_t t, int64_t ldx, const float* logits,
                                  int topk, const float* shared_gate, int32_t* topk_ids, float* topk_w, void* route_ws,
                                  size_t route_ws_bytes, void* out, int64_t ldo, void* workspace,
                                  size_t workspace_bytes, void* stream) {
  Geometry gu, dn;
  int st = check_moe(layer, t, topk, &gu, &dn);
  if (st != QG_OK) return (qg_status)st;
  if (!x || !logits || !topk_ids || !topk_w || !route_ws || !out || !workspace) return QG_ERR_INVALID_ARG;
  if (shared_gate && !layer->has_shared) return QG_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(shared_gate) % 4) return QG_ERR_MISALIGNED;
  if (t > 4 && (layer->ffn % 128 != 0 || layer->hidden % 8 != 0)) return QG_ERR_UNSUPPORTED;
  if (t * (int64_t)(topk + 1) >= ((int64_t)1 << 31)) return QG_ERR_UNSUPPORTED;
  if (ldx < layer->hidden || ldo < layer->hidden) return QG_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(out) || !aligned16(workspace) || !aligned16(route_ws) || !aligned16(topk_w) ||
      !aligned16(topk_ids) || !aligned16(logits))
    return QG_ERR_MISALIGNED;
  if (ldx % 8 || ldo % 8) return QG_ERR_MISALIGNED;
  if (route_ws_bytes < route_layout(t, layer->n_experts, topk).total) return QG_ERR_WORKSPACE_TOO_SMALL;
  DeviceInfo dev;
  if (!current_device_info(&dev)) return QG_ERR_CUDA;
  if (workspace_bytes < moe_layout(gu, dn, t, layer->n_experts, topk, dev.sms).total)
    return QG_ERR_WORKSPACE_TOO_SMALL;
  if (t > 4) {  // the router's own launches, then the prefill chain
    st = launch_route(logits, t, layer->n_experts, topk, topk_ids, topk_w, route_ws, stream);
    if (st != QG_OK) return (qg_status)st;
    return (qg_status)launch_moe_prefill(layer, gu, dn, x, t, ldx, topk, topk_w, shared_gate, route_ws, out, ldo,
                                         workspace, dev, stream, kMoeAll);
  }
  if (t * topk > kBlockRoutePairs) return QG_ERR_UNSUPPORTED;
  return (qg_status)launch_moe_decode(layer, gu, dn, x, t, ldx, topk, topk_w, shared_gate, route_ws, out, ldo,
                                      workspace, dev, stream, kMoeAll, logits, topk_ids, topk_w);
}
