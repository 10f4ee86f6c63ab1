// qk_noalloc.cu -- RMSNorm backward for callers that cannot allocate device memory.
//
// qk_rmsnorm_bwd needs a device workspace for its per-CTA partial sums of dw,
// which the caller allocates.  Some callers cannot: code that runs under a
// fixed device-memory budget reserved up front, hooks that a host framework
// hands only tensors and a stream (the framework owns every allocation), or
// code that must not trigger the implicit device synchronisation that
// cudaMalloc / cudaFree may cause.  qk_rmsnorm_bwd_noalloc gives them the same
// operator with the workspace taken from a fixed array in this library's
// device memory instead.
//
// The array is a file-scope __device__ object of kNoAllocScratchBytes: every
// GPU on which the library's device code is loaded holds it until the process
// exits.  In host code the array's name is only a host-side stand-in, so its
// device address is looked up with cudaGetSymbolAddress, once per device, with
// that device current, on the first call made on the device.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/qk.h"

// Largest workspace the no-allocation variant can serve: 16 MiB per device.
// The workspace holds one row of N fp32 dw partials per CTA (or per cluster)
// of the launch, so the need grows with N and with the CTA count of the plan;
// a call that would need more is refused with QK_ERR_UNSUPPORTED.
static constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch[kMaxDevices] = {};

// Device address of the scratch array on the current device; looked up on the
// first call made on each device.
qk_status scratch_on_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return QK_ERR_NO_DEVICE;
  }
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_scratch[dev] == nullptr) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr) {
      cudaGetLastError();
      return QK_ERR_LAUNCH;
    }
    g_scratch[dev] = ptr;
  }
  *out = g_scratch[dev];
  return QK_OK;
}

}  // namespace

extern "C" qk_status qk_rmsnorm_bwd_noalloc(const void* x, const void* w, const float* rstd,
                                            const void* dy, void* dx, float* dw, int64_t M,
                                            int64_t N, qk_dtype dtype, void* stream) {
  size_t need = 0;
  qk_status st = qk_rmsnorm_bwd_workspace_size(M, N, dtype, &need);  // checks M, N, dtype
  if (st != QK_OK) return st;
  if (M == 0) return QK_OK;
  if (need > kNoAllocScratchBytes) return QK_ERR_UNSUPPORTED;  // more than the fixed array holds
  void* scratch = nullptr;
  st = scratch_on_current_device(&scratch);
  if (st != QK_OK) return st;
  // Nothing in the scratch needs to start at zero: every partial row the
  // kernel later sums is written by the same call first.
  return qk_rmsnorm_bwd(x, w, rstd, dy, dx, dw, scratch, kNoAllocScratchBytes, M, N, dtype, stream);
}
