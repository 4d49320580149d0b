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
//    A failed lookup is not remembered: the next call tries again.
//  * All calls share the array: calls that overlap on the GPU (on different streams, or
//    from different threads) race and produce wrong results.  Calls on one stream are
//    ordered and safe.  Every call clears the row-tile tickets first; the status word is
//    sticky, like a workspace's, until qgemv_static_ws_status reads and clears it.
//  * Shapes whose scratch would exceed QG_STATIC_WORKSPACE_BYTES are rejected with
//    QG_ERR_WORKSPACE_TOO_SMALL before anything is launched.
#include <cuda_runtime.h>

#include <mutex>

#include "qg_internal.h"

namespace {

static __device__ __align__(256) unsigned char g_static_ws[QG_STATIC_WORKSPACE_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_ptr[kMaxDevices];

// The array's device address on the current device, looked up once it succeeds.
int static_ws_ptr(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return QG_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_ws) != cudaSuccess || !p) {
      cudaGetLastError();  // the failure is reported here, not left for the next launch
      return QG_ERR_CUDA;
    }
    g_ptr[dev] = p;
  }
  *out = g_ptr[dev];
  return QG_OK;
}

}  // namespace

extern "C" qg_status qgemv_static_ws(const qg_weight* w, const void* x, int m, int64_t ldx, const void* residual,
                                     int64_t ldr, void* y, int64_t ldy, void* stream) {
  qg::Geometry g;
  int st = qg::check_gemv_call(w, x, m, ldx, residual, ldr, y, ldy, &g);  // qgemv's rules
  if (st != QG_OK) return (qg_status)st;
  void* ws = nullptr;
  if ((st = static_ws_ptr(&ws)) != QG_OK) return (qg_status)st;
  qg::DeviceInfo info;
  if (!qg::current_device_info(&info)) return QG_ERR_CUDA;
  qg::GemvPlan p;
  if (!qg::plan_gemv(g, m, info, &p)) return QG_ERR_UNSUPPORTED;
  if (p.ws_bytes > QG_STATIC_WORKSPACE_BYTES) return QG_ERR_WORKSPACE_TOO_SMALL;

  // the tickets must start at zero (a call that timed out may have left some behind);
  // partial sums are always written before they are read
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(static_cast<unsigned char*>(ws) + p.off_cnt, 0, p.off_part - p.off_cnt, s) != cudaSuccess)
    return QG_ERR_CUDA;
  return (qg_status)qg::launch_gemv(g, w, x, m, ldx, residual, ldr, y, ldy, ws, p, stream);
}

extern "C" qg_status qgemv_static_ws_status(int* status, void* stream) {
  if (!status) return QG_ERR_INVALID_ARG;
  void* ws = nullptr;
  int st = static_ws_ptr(&ws);
  if (st != QG_OK) return (qg_status)st;
  return qg_workspace_status(ws, status, stream);
}
