// C ABI entry points: argument validation on the host, device attribute cache,
// dispatch to the kernel launchers.  No entry point allocates memory.
#include <cuda_runtime.h>

#include <mutex>

#include "qg_internal.h"

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
  if (w->fmt == QG_FMT_Q6K && !w->aux) return QG_ERR_INVALID_ARG;
  if (w->fmt != QG_FMT_NVFP4 && w->tensor_scale != 1.0f) return QG_ERR_INVALID_ARG;
  if (!aligned16(w->codes) || !aligned16(w->scales) || (w->aux && !aligned16(w->aux))) return QG_ERR_MISALIGNED;
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
  int st = check_weight(w, &g);
  if (st != QG_OK) return (qg_status)st;
  if (m < 1 || m > 4) return QG_ERR_UNSUPPORTED;
  if (!x || !y || !workspace) return QG_ERR_INVALID_ARG;
  if (ldx < w->k || ldy < w->n || (residual && ldr < w->n)) return QG_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(y) || (residual && !aligned16(residual)) || !aligned16(workspace))
    return QG_ERR_MISALIGNED;
  if (ldx % 8 || ldy % 8 || (residual && ldr % 8)) return QG_ERR_MISALIGNED;
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
  return (qg_status)launch_prefill(g, w, x, m, ldx, residual, ldr, y, ldy, workspace, stream);
}
