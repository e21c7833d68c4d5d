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
// device address is looked up with cudaGetSymbolAddress once per CUDA context
// (in practice once per device), with that device current, on the first call
// made in it; that first call should therefore come before any stream capture.
// No cudaMalloc, cudaFree or other allocating routine is called.
//
// Device-side errors of these calls (a bounded wait that gave up) land in the
// array's status word; wq_noalloc_read_device_status reads it. The next
// no-alloc call on the device clears it again.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstdio>
#include <mutex>

#include "wq_internal.h"

namespace {

constexpr uint64_t kScratchBytes = WQ_NOALLOC_SCRATCH_BYTES;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

// The array's device address belongs to the module loaded in one CUDA
// context: a device reset (or another context on the same device) loads the
// module again, possibly elsewhere. The cache is therefore keyed by the
// current context's unique id (cuCtxGetId), not by the device number.
struct ContextScratch {
  unsigned long long ctx_id;
  void *ptr;
};

std::mutex g_scratch_mu;
constexpr int kCacheSlots = 64;
ContextScratch g_scratch_tab[kCacheSlots];
int g_scratch_n = 0, g_scratch_next = 0;

using CtxGetCurrentFn = CUresult (*)(CUcontext *);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long *);

template <typename Fn>
Fn driver_fn(const char *name) {
  void *p = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion(name, &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
      q == cudaDriverEntryPointSuccess)
    return reinterpret_cast<Fn>(p);
  cudaGetLastError();
  return nullptr;
}

// Unique id of the calling thread's current context, or 0 if there is none yet.
unsigned long long current_context_id() {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    get_current = driver_fn<CtxGetCurrentFn>("cuCtxGetCurrent");
    get_id = driver_fn<CtxGetIdFn>("cuCtxGetId");
  });
  if (!get_current || !get_id) return 0;
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
  if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

int32_t cuda_error(cudaError_t e, const char *what) {
  char msg[200];
  snprintf(msg, sizeof(msg), "%s: %s", what, cudaGetErrorString(e));
  wq::set_last_error(WQ_ERR_CUDA, msg);
  return WQ_ERR_CUDA;
}

// Device address of g_noalloc_scratch in the current context. The first call
// in a context looks it up (cudaGetSymbolAddress, which also loads the module
// and, if needed, initialises the device's primary context).
int32_t scratch_address(void **out) {
  unsigned long long id = current_context_id();
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (id != 0) {
    for (int i = 0; i < g_scratch_n; ++i)
      if (g_scratch_tab[i].ctx_id == id) {
        *out = g_scratch_tab[i].ptr;
        return WQ_OK;
      }
  }
  void *ptr = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
  if (e != cudaSuccess || ptr == nullptr)
    return cuda_error(e, "cudaGetSymbolAddress of the static scratch");
  if (id == 0) id = current_context_id();  // the lookup made a context current
  if (id != 0) {
    g_scratch_tab[g_scratch_next] = {id, ptr};
    g_scratch_next = (g_scratch_next + 1) % kCacheSlots;
    if (g_scratch_n < kCacheSlots) ++g_scratch_n;
  }
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
  if (e != cudaSuccess) return cuda_error(e, "clearing the static scratch header");
  return wq_matmul_add_rmsnorm(x1, x2, scale, offset, bias, residual, gamma, eps, group, y,
                               normOut, ws, kScratchBytes, stream);
}

extern "C" int32_t wq_noalloc_read_device_status(void *stream, int32_t *device_status) {
  if (!device_status) {
    wq::set_last_error(WQ_ERR_NULL, "device_status is required");
    return WQ_ERR_NULL;
  }
  void *ws = nullptr;
  int32_t st = scratch_address(&ws);
  if (st != WQ_OK) return st;
  cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_error(e, "stream synchronize");
  uint32_t word = 0;
  e = cudaMemcpy(&word, ws, sizeof(word), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_error(e, "status word copy");
  *device_status = (int32_t)word;
  wq::set_last_error(WQ_OK, "");
  return WQ_OK;
}
