// qgemv_static_ws: the quantized GEMV without a caller-provided workspace.
//
// Some callers cannot allocate device memory: a plugin hosted by a runtime that owns
// all of the GPU's memory (a serving engine that reserved it up front for its KV cache
// and model weights and gives plugins no allocator), or code on a latency-critical path
// where cudaMalloc's implicit device-wide synchronisation is not acceptable.  For them
// this entry point keeps the GEMV's split-K scratch (status word, row-tile tickets and
// partial sums) in a file-scope device array of fixed size instead of a workspace
// argument.  It calls no cudaMalloc, cudaFree or other allocating routine.
//
// Properties a caller must know:
//  * The array (QG_STATIC_WORKSPACE_BYTES) exists once per GPU that loads the library
//    and stays allocated until the process exits.
//  * Its device address is looked up (cudaGetSymbolAddress) on the first call on each
//    device, with that device current; make that first call before any stream capture.
//  * All calls share the array: calls that overlap on the GPU (on different streams, or
//    from different threads) race and produce wrong results.  Calls on one stream are
//    ordered and safe.  Every call clears the status word and the tickets first.
//  * Shapes whose scratch would exceed QG_STATIC_WORKSPACE_BYTES are rejected with
//    QG_ERR_WORKSPACE_TOO_SMALL before anything is launched.
#include <cuda_runtime.h>

#include <mutex>

#include "qg_internal.h"

namespace {

static __device__ __align__(256) unsigned char g_static_ws[QG_STATIC_WORKSPACE_BYTES];

constexpr int kMaxDevices = 64;
std::once_flag g_once[kMaxDevices];
void* g_ptr[kMaxDevices];
cudaError_t g_err[kMaxDevices];

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" qg_status qgemv_static_ws(const qg_weight* w, const void* x, int m, int64_t ldx, const void* residual,
                                     int64_t ldr, void* y, int64_t ldy, void* stream) {
  // argument checks (the same rules as qgemv)
  qg::Geometry g;
  if (!w) return QG_ERR_INVALID_ARG;
  if (w->reserved != 0 || w->reserved2 != 0.0f) return QG_ERR_INVALID_ARG;
  if (!qg::geometry(w->fmt, w->n, w->k, &g)) return QG_ERR_INVALID_ARG;
  if (!w->codes || !w->scales) return QG_ERR_INVALID_ARG;
  if ((w->fmt == QG_FMT_Q6K || w->fmt == QG_FMT_Q5_K) && !w->aux) return QG_ERR_INVALID_ARG;
  if (w->fmt != QG_FMT_NVFP4 && w->tensor_scale != 1.0f) return QG_ERR_INVALID_ARG;
  if (!aligned16(w->codes) || !aligned16(w->scales) || (w->aux && !aligned16(w->aux))) return QG_ERR_MISALIGNED;
  if (m < 1 || m > 4) return QG_ERR_UNSUPPORTED;
  if (!x || !y) return QG_ERR_INVALID_ARG;
  if (ldx < w->k || ldy < w->n || (residual && ldr < w->n)) return QG_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(y) || (residual && !aligned16(residual))) return QG_ERR_MISALIGNED;
  if (ldx % 8 || ldy % 8 || (residual && ldr % 8)) return QG_ERR_MISALIGNED;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return QG_ERR_CUDA;
  std::call_once(g_once[dev], [dev] { g_err[dev] = cudaGetSymbolAddress(&g_ptr[dev], g_static_ws); });
  if (g_err[dev] != cudaSuccess || !g_ptr[dev]) return QG_ERR_CUDA;

  qg::DeviceInfo info;
  if (!qg::device_info(dev, &info)) return QG_ERR_CUDA;
  qg::GemvPlan p;
  if (!qg::plan_gemv(g, m, info, &p)) return QG_ERR_UNSUPPORTED;
  if (p.ws_bytes > QG_STATIC_WORKSPACE_BYTES) return QG_ERR_WORKSPACE_TOO_SMALL;

  // status word and tickets must start at zero (partial sums are always written first)
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(g_ptr[dev], 0, p.off_part, s) != cudaSuccess) return QG_ERR_CUDA;
  return (qg_status)qg::launch_gemv(g, w, x, m, ldx, residual, ldr, y, ldy, g_ptr[dev], p, stream);
}
