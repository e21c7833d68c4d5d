// Allocation-free entry point of the fused operator.
//
// Some callers cannot hand the library a workspace: a host framework whose
// custom-operator interface passes only input and output buffers, or a
// runtime that fixes its device memory at start-up and forbids allocations
// afterwards (cudaMalloc can synchronize the device, fail under memory
// pressure, or fragment a carefully planned heap in the middle of a run). For
// them, wq_matmul_add_rmsnorm_noalloc runs the same kernels as
// wq_matmul_add_rmsnorm, but their scratch memory (split-K partial sums, the
// device status word) lives in the fixed array below instead of a
// caller-provided workspace.
//
// The array is a file-scope __device__ variable: every GPU that loads this
// library holds WQ_NOALLOC_SCRATCH_BYTES for it until the process exits. In
// host code its name is only a host-side stand-in, not a device address, so the
// device address is looked up with cudaGetSymbolAddress once per device, with
// that device current, on the first call made on it; that first call should
// therefore come before any stream capture. No cudaMalloc, cudaFree or other
// allocating routine is called.
#include <cstdio>
#include <mutex>

#include "wq_internal.h"

namespace {

constexpr uint64_t kScratchBytes = WQ_NOALLOC_SCRATCH_BYTES;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

struct DeviceScratch {
  int device;
  void *ptr;
};

std::mutex g_scratch_mu;
DeviceScratch g_scratch_tab[256];
int g_scratch_n = 0;

// Device address of g_noalloc_scratch on the current device (set-up on first use).
int32_t scratch_address(void **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    char msg[160];
    snprintf(msg, sizeof(msg), "cudaGetDevice: %s", cudaGetErrorString(e));
    wq::set_last_error(WQ_ERR_CUDA, msg);
    return WQ_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  for (int i = 0; i < g_scratch_n; ++i) {
    if (g_scratch_tab[i].device == dev) {
      *out = g_scratch_tab[i].ptr;
      return WQ_OK;
    }
  }
  void *ptr = nullptr;
  e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
  if (e != cudaSuccess || ptr == nullptr) {
    char msg[160];
    snprintf(msg, sizeof(msg), "cudaGetSymbolAddress of the static scratch on device %d: %s", dev,
             cudaGetErrorString(e));
    wq::set_last_error(WQ_ERR_CUDA, msg);
    return WQ_ERR_CUDA;
  }
  if (g_scratch_n < 256) g_scratch_tab[g_scratch_n++] = {dev, ptr};
  *out = ptr;
  return WQ_OK;
}

}  // namespace

extern "C" int32_t wq_matmul_add_rmsnorm_noalloc(
    const wq_tensor *x1, const wq_tensor *x2, const wq_tensor *scale, const wq_tensor *offset,
    const wq_tensor *bias, const wq_tensor *residual, const wq_tensor *gamma, double eps,
    int64_t group, const wq_tensor *y, const wq_tensor *normOut, void *stream) {
  uint64_t need = 0;
  int32_t st = wq_matmul_add_rmsnorm_get_workspace(x1, x2, scale, offset, bias, residual, gamma,
                                                   eps, group, y, normOut, &need);
  if (st != WQ_OK) return st;
  if (need > kScratchBytes) {
    char msg[200];
    snprintf(msg, sizeof(msg),
             "this problem needs %llu bytes of scratch; the static scratch of the no-alloc entry "
             "point holds %llu (use wq_matmul_add_rmsnorm with a workspace)",
             (unsigned long long)need, (unsigned long long)kScratchBytes);
    wq::set_last_error(WQ_ERR_WORKSPACE, msg);
    return WQ_ERR_WORKSPACE;
  }
  void *ws = nullptr;
  st = scratch_address(&ws);
  if (st != WQ_OK) return st;
  // The shared array keeps whatever the previous call left; the status word
  // must start at zero for this call.
  cudaError_t e = cudaMemsetAsync(ws, 0, wq::kWsHeader, (cudaStream_t)stream);
  if (e != cudaSuccess) {
    char msg[160];
    snprintf(msg, sizeof(msg), "clearing the static scratch header: %s", cudaGetErrorString(e));
    wq::set_last_error(WQ_ERR_CUDA, msg);
    return WQ_ERR_CUDA;
  }
  return wq_matmul_add_rmsnorm(x1, x2, scale, offset, bias, residual, gamma, eps, group, y,
                               normOut, ws, kScratchBytes, stream);
}
