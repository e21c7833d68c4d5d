// Host side of the C ABI: argument validation (the "first phase" of each
// operator), workspace sizing, kernel selection and launch.
//
// Validation follows aclnnWeightQuantMatmulAllReduceAddRmsNorm, "Constraints":
// x1 2-D (s, k) or 3-D (b, s, k) with b*s and s in [1, 2^31-1] (0 allowed as an
// empty tensor), k and n in [1, 65535] (k = 0 rejected, n = 0 empty), x2 2-D
// (k, n) INT8/INT4, bias (n), residual (b, s, n) with b*s = s of a 2-D x1,
// gamma (n), y/normOut shaped like residual, one floating dtype for x1, scale,
// offset, bias, residual and gamma, scale (1) / (n) / (1, n) /
// (ceil(k/group), n), offset shaped like scale, group in [32, k-1] and a
// multiple of 32. The INT4 storage rule (last dimension even) is the one of
// aclnnDynamicQuant, "Constraints".
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "wq_internal.h"
#include "wq_sync.cuh"

namespace wq {
namespace {

thread_local std::string g_last_error;

// Wait limits of the operator kernels' cross-CTA waits (wq_test_set_wait_limits).
std::atomic<long long> g_wait_budget{kWaitBudget};
std::atomic<uint32_t> g_wait_extra{0};

int32_t fail(int32_t code, const char *fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return code;
}

int32_t ok() {
  g_last_error.clear();
  return WQ_OK;
}

int64_t numel(const wq_tensor *t) {
  int64_t n = 1;
  for (int i = 0; i < t->ndim; ++i) n *= t->shape[i];
  return n;
}

int64_t elem_bits(int dt) {
  switch (dt) {
    case WQ_F16: case WQ_BF16: return 16;
    case WQ_INT8: case WQ_INT8_T: case WQ_E8M0: return 8;
    case WQ_INT4: case WQ_INT4_TILED: case WQ_INT4_T: case WQ_FP4_E2M1: case WQ_FP4_E2M1_T:
      return 4;
    case WQ_INT32: case WQ_F32: return 32;
    default: return 0;
  }
}

uint64_t nbytes(const wq_tensor *t) {
  if (t->dtype == WQ_INT4_TILED && t->ndim == 2)  // K padded to a multiple of 64
    return tiled_int4_bytes(t->shape[0], t->shape[1]);
  return (uint64_t)((numel(t) * elem_bits(t->dtype) + 7) / 8);
}

bool valid_rank(const wq_tensor *t) {
  if (t->ndim < 1 || t->ndim > 3) return false;
  for (int i = 0; i < t->ndim; ++i)
    if (t->shape[i] < 0) return false;
  return true;
}

bool overlap(const wq_tensor *a, const wq_tensor *b) {
  if (!a || !b || !a->data || !b->data) return false;
  uint64_t a0 = (uint64_t)(uintptr_t)a->data, a1 = a0 + nbytes(a);
  uint64_t b0 = (uint64_t)(uintptr_t)b->data, b1 = b0 + nbytes(b);
  if (a1 == a0 || b1 == b0) return false;
  return a0 < b1 && b0 < a1;
}

bool same_shape(const wq_tensor *a, const wq_tensor *b) {
  if (a->ndim != b->ndim) return false;
  for (int i = 0; i < a->ndim; ++i)
    if (a->shape[i] != b->shape[i]) return false;
  return true;
}

const char *dtname(int dt) {
  switch (dt) {
    case WQ_F16: return "F16"; case WQ_BF16: return "BF16"; case WQ_INT8: return "INT8";
    case WQ_INT4: return "INT4"; case WQ_INT32: return "INT32";
    case WQ_INT4_TILED: return "INT4_TILED"; case WQ_F32: return "F32";
    case WQ_INT8_T: return "INT8_T"; case WQ_INT4_T: return "INT4_T";
    case WQ_FP4_E2M1: return "FP4_E2M1"; case WQ_E8M0: return "E8M0";
    case WQ_FP4_E2M1_T: return "FP4_E2M1_T"; default: return "?";
  }
}

constexpr int64_t kMaxRows = 2147483647LL;  // b*s upper bound
constexpr int64_t kMaxKN = 65535;           // k, n upper bound

// Full validation of the fused operator; fills `p` on success.
int32_t validate(const wq_tensor *x1, const wq_tensor *x2, const wq_tensor *scale,
                 const wq_tensor *offset, const wq_tensor *bias, const wq_tensor *residual,
                 const wq_tensor *gamma, double eps, int64_t group, const wq_tensor *y,
                 const wq_tensor *normOut, Problem &p) {
  if (!x1 || !x2 || !scale || !residual || !gamma || !y || !normOut)
    return fail(WQ_ERR_NULL, "x1, x2, scale, residual, gamma, y and normOut are required");
  const wq_tensor *all[] = {x1, x2, scale, offset, bias, residual, gamma, y, normOut};
  const char *names[] = {"x1", "x2", "scale", "offset", "bias", "residual", "gamma", "y", "normOut"};
  for (int i = 0; i < 9; ++i)
    if (all[i] && !valid_rank(all[i]))
      return fail(WQ_ERR_SHAPE, "%s: rank must be 1..3 with non-negative dims", names[i]);

  // dtypes
  const int dt = x1->dtype;
  if (dt != WQ_F16 && dt != WQ_BF16)
    return fail(WQ_ERR_DTYPE, "x1 must be F16 or BF16, got %s", dtname(dt));
  if (x2->dtype != WQ_INT8 && x2->dtype != WQ_INT4 && x2->dtype != WQ_INT4_TILED &&
      x2->dtype != WQ_INT8_T && x2->dtype != WQ_INT4_T)
    return fail(WQ_ERR_DTYPE, "x2 must be INT8, INT4, INT4_TILED, INT8_T or INT4_T, got %s",
                dtname(x2->dtype));
  const bool x2t = x2->dtype == WQ_INT8_T || x2->dtype == WQ_INT4_T;  // stored (n, k)
  const wq_tensor *same[] = {scale, offset, bias, residual, gamma, y, normOut};
  const char *snames[] = {"scale", "offset", "bias", "residual", "gamma", "y", "normOut"};
  for (int i = 0; i < 7; ++i)
    if (same[i] && same[i]->dtype != dt)
      return fail(WQ_ERR_DTYPE, "%s must have x1's dtype %s, got %s", snames[i], dtname(dt),
                  dtname(same[i]->dtype));

  // x1: (s, k) or (b, s, k)
  if (x1->ndim != 2 && x1->ndim != 3) return fail(WQ_ERR_SHAPE, "x1 must be 2-D or 3-D");
  const int64_t K = x1->shape[x1->ndim - 1];
  int64_t M = 1;
  for (int i = 0; i < x1->ndim - 1; ++i) {
    if (x1->shape[i] > kMaxRows) return fail(WQ_ERR_SHAPE, "x1 dim %d exceeds 2^31-1", i);
    M *= x1->shape[i];
  }
  if (M > kMaxRows) return fail(WQ_ERR_SHAPE, "b*s = %lld exceeds 2^31-1", (long long)M);
  if (K < 1) return fail(WQ_ERR_SHAPE, "k must be >= 1 (empty k is not supported)");
  if (K > kMaxKN) return fail(WQ_ERR_SHAPE, "k = %lld exceeds 65535", (long long)K);

  // x2: (k, n), or (n, k) when transposed
  if (x2->ndim != 2) return fail(WQ_ERR_SHAPE, "x2 must be 2-D (k, n), or (n, k) when transposed");
  if (x2->shape[x2t ? 1 : 0] != K)
    return fail(WQ_ERR_SHAPE, "x2 has k = %lld, x1 has k = %lld", (long long)x2->shape[x2t ? 1 : 0],
                (long long)K);
  const int64_t N = x2->shape[x2t ? 0 : 1];
  if (x2->dtype == WQ_INT4_T && (K % 2) != 0)
    return fail(WQ_ERR_SHAPE, "INT4_T x2 packs along k, which must be even, got k = %lld",
                (long long)K);
  if (N > kMaxKN) return fail(WQ_ERR_SHAPE, "n = %lld exceeds 65535", (long long)N);
  if (x2->dtype == WQ_INT4 && (N % 2) != 0)
    return fail(WQ_ERR_SHAPE, "INT4 x2 needs an even last dimension, got n = %lld", (long long)N);
  if (x2->dtype == WQ_INT4_TILED && (N % 16) != 0)
    return fail(WQ_ERR_SHAPE, "INT4_TILED x2 needs n %% 16 == 0, got n = %lld", (long long)N);
  if (x2->dtype == WQ_INT4_TILED && ((uintptr_t)x2->data % 16) != 0)
    return fail(WQ_ERR_UNSUPPORTED, "INT4_TILED x2 must be 16-byte aligned");

  // scale / group
  int smode;
  int64_t G = 1, Ns = 1;
  if (group != 0) {
    if (group < 32 || group > K - 1 || group % 32 != 0)
      return fail(WQ_ERR_GROUP, "group = %lld must be a multiple of 32 in [32, k-1 = %lld]",
                  (long long)group, (long long)(K - 1));
    const int64_t want = (K + group - 1) / group;
    if (scale->ndim != 2 || scale->shape[0] != want || scale->shape[1] != N)
      return fail(WQ_ERR_GROUP, "per-group scale must be (ceil(k/group) = %lld, n = %lld)",
                  (long long)want, (long long)N);
    smode = kPerGroup;
    G = want;
    Ns = N;
  } else {
    if (scale->ndim == 1 && scale->shape[0] == 1) {
      smode = kPerTensor;
    } else if (scale->ndim == 1 && scale->shape[0] == N) {
      smode = kPerChannel;
      Ns = N;
    } else if (scale->ndim == 2 && scale->shape[0] == 1 && scale->shape[1] == N) {
      smode = kPerChannel;
      Ns = N;
    } else if (scale->ndim == 2 && scale->shape[1] == N && scale->shape[0] > 1) {
      return fail(WQ_ERR_GROUP, "a (%lld, n) scale is per-group and needs group != 0",
                  (long long)scale->shape[0]);
    } else {
      return fail(WQ_ERR_SHAPE, "scale must be (1), (n), (1, n) or (ceil(k/group), n)");
    }
    if (smode == kPerTensor && N == 1) { smode = kPerChannel; Ns = 1; }
  }
  if (offset && !same_shape(offset, scale))
    return fail(WQ_ERR_SHAPE, "offset must have the scale's shape");

  // bias (n), gamma (n)
  if (bias && (bias->ndim != 1 || bias->shape[0] != N))
    return fail(WQ_ERR_SHAPE, "bias must be 1-D (n = %lld)", (long long)N);
  if (gamma->ndim != 1 || gamma->shape[0] != N)
    return fail(WQ_ERR_SHAPE, "gamma must be 1-D (n = %lld)", (long long)N);

  // residual: (b, s, n) with b*s = M, or (M, n)
  if (residual->ndim != 2 && residual->ndim != 3)
    return fail(WQ_ERR_SHAPE, "residual must be 3-D (b, s, n) or 2-D (b*s, n)");
  {
    int64_t rm = 1;
    for (int i = 0; i < residual->ndim - 1; ++i) rm *= residual->shape[i];
    if (rm != M || residual->shape[residual->ndim - 1] != N)
      return fail(WQ_ERR_SHAPE, "residual must hold b*s = %lld rows of n = %lld", (long long)M,
                  (long long)N);
  }
  if (!same_shape(y, residual)) return fail(WQ_ERR_SHAPE, "y must have residual's shape");
  if (!same_shape(normOut, residual)) return fail(WQ_ERR_SHAPE, "normOut must have residual's shape");

  if (!(eps >= 0.0) || !std::isfinite(eps))
    return fail(WQ_ERR_SHAPE, "eps must be finite and >= 0");

  // data pointers of non-empty tensors
  for (int i = 0; i < 9; ++i)
    if (all[i] && numel(all[i]) > 0 && !all[i]->data)
      return fail(WQ_ERR_NULL, "%s has elements but a NULL data pointer", names[i]);

  // aliasing: y may be exactly residual (in-place variant), nothing else overlaps
  const wq_tensor *ins[] = {x1, x2, scale, offset, bias, residual, gamma};
  const char *inames[] = {"x1", "x2", "scale", "offset", "bias", "residual", "gamma"};
  for (int i = 0; i < 7; ++i) {
    if (overlap(normOut, ins[i]))
      return fail(WQ_ERR_ALIAS, "normOut overlaps %s", inames[i]);
    if (i == 5) {
      if (overlap(y, residual) && y->data != residual->data)
        return fail(WQ_ERR_ALIAS, "y partially overlaps residual (only y == residual is allowed)");
      continue;
    }
    if (overlap(y, ins[i])) return fail(WQ_ERR_ALIAS, "y overlaps %s", inames[i]);
  }
  if (overlap(normOut, y)) return fail(WQ_ERR_ALIAS, "normOut overlaps y");

  p = Problem();
  p.M = M; p.K = K; p.N = N;
  p.dtype = dt;
  p.wbits = (x2->dtype == WQ_INT8 || x2->dtype == WQ_INT8_T) ? 8 : 4;
  p.tiled = x2->dtype == WQ_INT4_TILED;
  p.transposed = x2t;
  p.smode = smode; p.group = smode == kPerGroup ? group : 0; p.G = G; p.Ns = Ns;
  p.eps = (float)eps;
  p.x1 = x1->data; p.x2 = x2->data; p.scale = scale->data;
  p.offset = offset ? offset->data : nullptr;
  p.bias = bias ? bias->data : nullptr;
  p.residual = residual->data; p.gamma = gamma->data;
  p.y = y->data; p.normOut = normOut->data;
  return WQ_OK;
}

// Picks the kernel and sizes the workspace. Returns WQ_ERR_UNSUPPORTED for a
// forced kernel that cannot run the problem.
int32_t make_plan(const Problem &p, int32_t kernel, Plan &plan) {
  plan = Plan();
  if (kernel < WQ_KERNEL_AUTO || kernel > WQ_KERNEL_PREFILL)
    return fail(WQ_ERR_UNSUPPORTED, "unknown kernel selector %d", kernel);
  if (p.M == 0 || p.N == 0) {  // empty output: nothing to launch
    plan.kernel = kernel == WQ_KERNEL_AUTO ? WQ_KERNEL_GENERIC : kernel;
    plan.ws_bytes = 0;
    return WQ_OK;
  }
  int chosen = kernel;
  if (p.transposed) {
    // a transposed weight: the transposed-operand large-M kernel (INT4, bf16
    // per-group scales, no offset), else the generic kernel reads it in place
    if (chosen == WQ_KERNEL_DECODE)
      return fail(WQ_ERR_UNSUPPORTED, "the decode kernels do not read a transposed x2 "
                                      "(convert an INT4_T weight with wq_convert_int4_layout)");
    if (chosen == WQ_KERNEL_PREFILL || (chosen == WQ_KERNEL_AUTO && p.M > 16)) {
      if (plan_prefill_t(p, plan)) return WQ_OK;
      if (chosen == WQ_KERNEL_PREFILL)
        return fail(WQ_ERR_UNSUPPORTED,
                    "the prefill kernel reads a transposed x2 only as INT4 with bf16 per-group "
                    "scales (group %% 32 == 0) and no offset, k %% 64 == 0, n %% 32 == 0 and "
                    "16-byte aligned tensors");
    }
    chosen = WQ_KERNEL_GENERIC;
  }
  if (p.tiled) {
    // the tiled layout: the tiled decode kernels for small M (the k-major one
    // for 9..32 rows), else the generic kernel
    if (chosen == WQ_KERNEL_AUTO)
      chosen = ((p.M <= 16 && decode_tiled_applicable(p)) || decode_km_applicable(p))
                   ? WQ_KERNEL_DECODE
                   : WQ_KERNEL_GENERIC;
    if (chosen == WQ_KERNEL_DECODE) {
      if (!plan_decode_tiled(p, plan))
        return fail(WQ_ERR_UNSUPPORTED,
                    "the tiled decode kernels need 1 <= m <= 16, k %% 8 == 0, 16-byte aligned x1, "
                    "scale, offset, bias, residual and gamma, 4-byte aligned y and normOut, and at "
                    "most 32 column groups of 16 per CTA; or 9 <= m <= 64, k %% 128 == 0, group "
                    "%% 128 == 0 (or per-channel / per-tensor scales) and at most 14 column "
                    "groups of 16 per CTA");
      return WQ_OK;
    }
    if (chosen == WQ_KERNEL_PREFILL)
      return fail(WQ_ERR_UNSUPPORTED, "the prefill kernel does not read the INT4_TILED layout");
  }
  if (chosen == WQ_KERNEL_AUTO) {
    if (p.M <= 16 && decode_applicable(p))
      chosen = WQ_KERNEL_DECODE;
    else if (prefill_applicable(p))
      chosen = WQ_KERNEL_PREFILL;
    else
      chosen = WQ_KERNEL_GENERIC;
  }
  if (chosen == WQ_KERNEL_DECODE) {
    if (!plan_decode(p, plan))
      return fail(WQ_ERR_UNSUPPORTED,
                  "the decode kernel needs 1 <= m <= 16, INT4 weights, n %% 32 == 0, k %% 8 == 0, "
                  "16-byte aligned x1, x2, scale and offset and 8-byte aligned bias, residual, "
                  "gamma, y and normOut");
    return WQ_OK;
  }
  if (chosen == WQ_KERNEL_PREFILL) {
    if (!plan_prefill(p, plan))
      return fail(WQ_ERR_UNSUPPORTED,
                  "the prefill kernel needs k %% 8 == 0, n %% 32 == 0 (INT4) or n %% 16 == 0 "
                  "(INT8), 16-byte aligned tensors and ceil(n/256) <= SM count");
    return WQ_OK;
  }
  if (!plan_generic(p, plan)) return fail(WQ_ERR_UNSUPPORTED, "generic plan failed");
  plan_epilogue(p, plan);
  plan.kernel = chosen;
  return WQ_OK;
}

int32_t cuda_fail(cudaError_t e, const char *what) {
  return fail(WQ_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

}  // namespace

long long wait_budget() { return g_wait_budget.load(std::memory_order_relaxed); }
uint32_t wait_extra_arrivals() { return g_wait_extra.load(std::memory_order_relaxed); }

void set_last_error(int32_t code, const char *msg) {
  if (code == WQ_OK)
    g_last_error.clear();
  else
    g_last_error = msg;
}

const DeviceInfo &device_info() {
  // One entry per device id; filled on first use with that device current.
  static std::mutex mu;
  static std::vector<DeviceInfo> cache;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) dev = 0;
  std::lock_guard<std::mutex> lock(mu);
  for (auto &d : cache)
    if (d.device == dev) return d;
  DeviceInfo d;
  d.device = dev;
  cudaDeviceProp prop;
  if (cudaGetDeviceProperties(&prop, dev) == cudaSuccess) {
    d.sms = prop.multiProcessorCount;
    d.cc_major = prop.major;
    d.cc_minor = prop.minor;
    d.smem_optin = prop.sharedMemPerBlockOptin;
  } else {
    cudaGetLastError();
  }
  cache.push_back(d);
  return cache.back();
}

}  // namespace wq

using namespace wq;

extern "C" {

int32_t wq_version(void) { return 100; }

const char *wq_status_string(int32_t s) {
  switch (s) {
    case WQ_OK: return "WQ_OK";
    case WQ_ERR_NULL: return "WQ_ERR_NULL";
    case WQ_ERR_DTYPE: return "WQ_ERR_DTYPE";
    case WQ_ERR_SHAPE: return "WQ_ERR_SHAPE";
    case WQ_ERR_GROUP: return "WQ_ERR_GROUP";
    case WQ_ERR_WORKSPACE: return "WQ_ERR_WORKSPACE";
    case WQ_ERR_UNSUPPORTED: return "WQ_ERR_UNSUPPORTED";
    case WQ_ERR_CUDA: return "WQ_ERR_CUDA";
    case WQ_ERR_DEVICE_TIMEOUT: return "WQ_ERR_DEVICE_TIMEOUT";
    case WQ_ERR_ALIAS: return "WQ_ERR_ALIAS";
    default: return "WQ_ERR_UNKNOWN";
  }
}

const char *wq_last_error(void) { return g_last_error.c_str(); }

// ------------------------------------------------------------------ pack

static int32_t validate_pack(const wq_tensor *w, const wq_tensor *o) {
  if (!w || !o) return fail(WQ_ERR_NULL, "weight and weight_int4 are required");
  if (w->dtype == WQ_F32 || o->dtype == WQ_FP4_E2M1) {  // FLOAT -> FLOAT4_E2M1
    if (w->dtype != WQ_F32 || o->dtype != WQ_FP4_E2M1)
      return fail(WQ_ERR_DTYPE, "an FP4_E2M1 pack takes an F32 weight, got %s -> %s",
                  dtname(w->dtype), dtname(o->dtype));
    if (!valid_rank(w) || !valid_rank(o) || w->ndim != 2 || !same_shape(w, o))
      return fail(WQ_ERR_SHAPE, "weight and the output must be 2-D of one logical shape");
    if (w->shape[1] % 2 != 0) return fail(WQ_ERR_SHAPE, "the last dimension must be even for FP4");
    if (numel(w) > 0 && (!w->data || !o->data))
      return fail(WQ_ERR_NULL, "non-empty tensors need data pointers");
    if (overlap(w, o)) return fail(WQ_ERR_ALIAS, "the output overlaps the weight");
    return WQ_OK;
  }
  if (w->dtype != WQ_INT32) return fail(WQ_ERR_DTYPE, "weight must be INT32, got %s", dtname(w->dtype));
  if (o->dtype != WQ_INT4 && o->dtype != WQ_INT4_TILED && o->dtype != WQ_INT4_T)
    return fail(WQ_ERR_DTYPE, "weight_int4 must be INT4, INT4_TILED or INT4_T, got %s",
                dtname(o->dtype));
  if (!valid_rank(w) || !valid_rank(o) || w->ndim != 2 || o->ndim != 2)
    return fail(WQ_ERR_SHAPE, "weight and weight_int4 must be 2-D");
  if (!same_shape(w, o)) return fail(WQ_ERR_SHAPE, "weight_int4 must have weight's logical shape");
  if (w->shape[1] % 2 != 0) return fail(WQ_ERR_SHAPE, "the last dimension must be even for INT4");
  if (o->dtype == WQ_INT4_TILED && w->shape[1] % 16 != 0)
    return fail(WQ_ERR_SHAPE, "the INT4_TILED layout needs the last dimension divisible by 16");
  if (o->dtype == WQ_INT4_TILED && ((uintptr_t)o->data % 16) != 0)
    return fail(WQ_ERR_UNSUPPORTED, "an INT4_TILED tensor must be 16-byte aligned");
  if (numel(w) > 0 && (!w->data || !o->data))
    return fail(WQ_ERR_NULL, "non-empty tensors need data pointers");
  if (overlap(w, o)) return fail(WQ_ERR_ALIAS, "weight_int4 overlaps weight");
  return WQ_OK;
}

int32_t wq_pack_int4_get_workspace(const wq_tensor *w, const wq_tensor *o, uint64_t *ws_bytes) {
  if (!ws_bytes) return fail(WQ_ERR_NULL, "ws_bytes is required");
  int32_t st = validate_pack(w, o);
  if (st) return st;
  *ws_bytes = 0;
  return ok();
}

int32_t wq_pack_int4(const wq_tensor *w, const wq_tensor *o, void *ws, uint64_t ws_bytes,
                     void *stream) {
  (void)ws; (void)ws_bytes;
  int32_t st = validate_pack(w, o);
  if (st) return st;
  if (numel(w) == 0) return ok();
  if (o->dtype == WQ_FP4_E2M1) {
    cudaError_t e = launch_pack_fp4((const float *)w->data, (uint8_t *)o->data, w->shape[0],
                                    w->shape[1], (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "FP4 pack kernel launch");
    return ok();
  }
  cudaError_t e = o->dtype == WQ_INT4_TILED
                      ? launch_pack_int4_tiled((const int32_t *)w->data, (uint8_t *)o->data,
                                               w->shape[0], w->shape[1], (cudaStream_t)stream)
                      : launch_pack_int4((const int32_t *)w->data, (uint8_t *)o->data, w->shape[0],
                                         w->shape[1], (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "pack kernel launch");
  return ok();
}

int32_t wq_convert_int4_layout(const wq_tensor *src, const wq_tensor *dst, void *stream) {
  if (!src || !dst) return fail(WQ_ERR_NULL, "src and dst are required");
  auto is4 = [](int d) { return d == WQ_INT4 || d == WQ_INT4_TILED || d == WQ_INT4_T; };
  if (!is4(src->dtype) || !is4(dst->dtype) || src->dtype == dst->dtype)
    return fail(WQ_ERR_DTYPE, "converts between two of INT4, INT4_TILED and INT4_T, got %s -> %s",
                dtname(src->dtype), dtname(dst->dtype));
  if (!valid_rank(src) || !valid_rank(dst) || src->ndim != 2 || dst->ndim != 2)
    return fail(WQ_ERR_SHAPE, "src and dst must be 2-D");
  // logical (K, N) of each side (INT4_T is given as its stored (N, K))
  auto kn = [](const wq_tensor *t, int64_t &K, int64_t &N) {
    K = t->shape[t->dtype == WQ_INT4_T ? 1 : 0];
    N = t->shape[t->dtype == WQ_INT4_T ? 0 : 1];
  };
  int64_t K, N, K2, N2;
  kn(src, K, N);
  kn(dst, K2, N2);
  if (K != K2 || N != N2) return fail(WQ_ERR_SHAPE, "src and dst must hold one (k, n) weight");
  const bool tiled = src->dtype == WQ_INT4_TILED || dst->dtype == WQ_INT4_TILED;
  if (tiled && N % 16 != 0)
    return fail(WQ_ERR_SHAPE, "the INT4_TILED layout needs n divisible by 16");
  if (src->dtype == WQ_INT4_T || dst->dtype == WQ_INT4_T ? K % 2 != 0 : false)
    return fail(WQ_ERR_SHAPE, "the INT4_T layout packs along k, which must be even");
  if (src->dtype == WQ_INT4 || dst->dtype == WQ_INT4 ? N % 2 != 0 : false)
    return fail(WQ_ERR_SHAPE, "the INT4 layout packs along n, which must be even");
  if (K * N > 0 && (!src->data || !dst->data))
    return fail(WQ_ERR_NULL, "non-empty tensors need data pointers");
  if (K * N > 0 && tiled) {
    const wq_tensor *tl = src->dtype == WQ_INT4_TILED ? src : dst;
    if (((uintptr_t)tl->data % 16) != 0)
      return fail(WQ_ERR_UNSUPPORTED, "an INT4_TILED tensor must be 16-byte aligned");
  }
  if (overlap(src, dst)) return fail(WQ_ERR_ALIAS, "dst overlaps src");
  if (K * N == 0) return ok();
  cudaStream_t s = (cudaStream_t)stream;
  const uint8_t *in = (const uint8_t *)src->data;
  uint8_t *out = (uint8_t *)dst->data;
  cudaError_t e;
  if (src->dtype == WQ_INT4 && dst->dtype == WQ_INT4_TILED)
    e = launch_int4_nd_to_tiled(in, out, K, N, s);
  else if (src->dtype == WQ_INT4_TILED && dst->dtype == WQ_INT4)
    e = launch_int4_tiled_to_nd(in, out, K, N, s);
  else
    e = launch_int4_remap(in, src->dtype, out, dst->dtype, K, N, s);
  if (e != cudaSuccess) return cuda_fail(e, "layout conversion launch");
  return ok();
}

// ------------------------------------------------------------------ mx block-scaled matmul

static int32_t validate_mx(const wq_tensor *x1, const wq_tensor *s1, const wq_tensor *x2,
                           const wq_tensor *s2, const wq_tensor *y, int64_t &M, int64_t &K,
                           int64_t &N) {
  if (!x1 || !s1 || !x2 || !s2 || !y) return fail(WQ_ERR_NULL, "x1, scale1, x2, scale2 and y are required");
  const wq_tensor *all[] = {x1, s1, x2, s2, y};
  for (const wq_tensor *t : all)
    if (!valid_rank(t) || t->ndim != 2) return fail(WQ_ERR_SHAPE, "every operand is 2-D");
  if ((x1->dtype != WQ_FP4_E2M1 && x1->dtype != WQ_FP4_E2M1_T) || x2->dtype != WQ_FP4_E2M1)
    return fail(WQ_ERR_DTYPE, "x1 must be FP4_E2M1 or FP4_E2M1_T and x2 FP4_E2M1");
  if (s1->dtype != WQ_E8M0 || s2->dtype != WQ_E8M0)
    return fail(WQ_ERR_DTYPE, "scale1 and scale2 must be E8M0");
  if (y->dtype != WQ_F32) return fail(WQ_ERR_DTYPE, "y must be F32");
  const bool x1t = x1->dtype == WQ_FP4_E2M1_T;
  M = x1t ? x1->shape[1] : x1->shape[0];
  K = x1t ? x1->shape[0] : x1->shape[1];
  N = x2->shape[1];
  if (K < 1 || K > kMaxKN || N > kMaxKN || M > kMaxRows)
    return fail(WQ_ERR_SHAPE, "k must lie in [1, 65535], n in [0, 65535]");
  if (K % 2 || N % 2) return fail(WQ_ERR_SHAPE, "k and n must be even (two FP4 codes per byte)");
  if (x1t && M % 2) return fail(WQ_ERR_SHAPE, "a transposed x1 packs along m: m must be even");
  if (x2->shape[0] != K) return fail(WQ_ERR_SHAPE, "x2 must be (k, n) with x1's k");
  const int64_t J = (K + 31) / 32;
  if (!x1t && (s1->shape[0] != M || s1->shape[1] != J))
    return fail(WQ_ERR_SHAPE, "scale1 must be (m, ceil(k/32) = %lld)", (long long)J);
  if (x1t && (s1->shape[0] != J || s1->shape[1] != M))
    return fail(WQ_ERR_SHAPE, "with a transposed x1, scale1 must be (ceil(k/32) = %lld, m)",
                (long long)J);
  if (s2->shape[0] != J || s2->shape[1] != N)
    return fail(WQ_ERR_SHAPE, "scale2 must be (ceil(k/32) = %lld, n)", (long long)J);
  if (y->shape[0] != M || y->shape[1] != N) return fail(WQ_ERR_SHAPE, "y must be (m, n)");
  for (const wq_tensor *t : all)
    if (numel(t) > 0 && !t->data) return fail(WQ_ERR_NULL, "a non-empty tensor has no data");
  const wq_tensor *ins[] = {x1, s1, x2, s2};
  for (const wq_tensor *t : ins)
    if (overlap(y, t)) return fail(WQ_ERR_ALIAS, "y overlaps an input");
  return WQ_OK;
}

int32_t wq_mx_matmul_add_get_workspace(const wq_tensor *x1, const wq_tensor *s1,
                                       const wq_tensor *x2, const wq_tensor *s2,
                                       const wq_tensor *y, uint64_t *ws_bytes) {
  if (!ws_bytes) return fail(WQ_ERR_NULL, "ws_bytes is required");
  int64_t M, K, N;
  int32_t st = validate_mx(x1, s1, x2, s2, y, M, K, N);
  if (st) return st;
  *ws_bytes = 0;
  return ok();
}

int32_t wq_mx_matmul_add_ex(const wq_tensor *x1, const wq_tensor *s1, const wq_tensor *x2,
                            const wq_tensor *s2, const wq_tensor *y, int32_t kernel, void *ws,
                            uint64_t ws_bytes, void *stream) {
  (void)ws; (void)ws_bytes;
  if (kernel != WQ_MX_KERNEL_TENSOR && kernel != WQ_MX_KERNEL_EXACT)
    return fail(WQ_ERR_UNSUPPORTED, "unknown mx kernel %d", (int)kernel);
  int64_t M, K, N;
  int32_t st = validate_mx(x1, s1, x2, s2, y, M, K, N);
  if (st) return st;
  if (M == 0 || N == 0) return ok();
  const bool x1t = x1->dtype == WQ_FP4_E2M1_T;
  const uint8_t *a = (const uint8_t *)x1->data, *sa = (const uint8_t *)s1->data;
  const uint8_t *b = (const uint8_t *)x2->data, *sb = (const uint8_t *)s2->data;
  cudaError_t e = kernel == WQ_MX_KERNEL_EXACT
                      ? launch_mx_matmul_add(a, sa, x1t, b, sb, (float *)y->data, M, K, N,
                                             (cudaStream_t)stream)
                      : launch_mx_matmul_add_tc(a, sa, x1t, b, sb, (float *)y->data, M, K, N,
                                                (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "mx matmul launch");
  return ok();
}

int32_t wq_mx_matmul_add(const wq_tensor *x1, const wq_tensor *s1, const wq_tensor *x2,
                         const wq_tensor *s2, const wq_tensor *y, void *ws, uint64_t ws_bytes,
                         void *stream) {
  return wq_mx_matmul_add_ex(x1, s1, x2, s2, y, WQ_MX_KERNEL_TENSOR, ws, ws_bytes, stream);
}

// ------------------------------------------------------------------ dynamic quantization

static int32_t validate_dq(const wq_tensor *x, const wq_tensor *sm, const wq_tensor *y,
                           const wq_tensor *sc, int64_t &M, int64_t &K, int &bits) {
  if (!x || !y || !sc) return fail(WQ_ERR_NULL, "x, y and scale are required");
  const wq_tensor *all[] = {x, sm, y, sc};
  for (const wq_tensor *t : all)
    if (t && !valid_rank(t)) return fail(WQ_ERR_SHAPE, "ranks must be 1..3 with non-negative dims");
  if (x->dtype != WQ_F16 && x->dtype != WQ_BF16)
    return fail(WQ_ERR_DTYPE, "x must be F16 or BF16, got %s", dtname(x->dtype));
  if (sm && sm->dtype != x->dtype) return fail(WQ_ERR_DTYPE, "smooth_scales must have x's dtype");
  if (y->dtype != WQ_INT8 && y->dtype != WQ_INT4)
    return fail(WQ_ERR_DTYPE, "y must be INT8 or INT4, got %s", dtname(y->dtype));
  if (sc->dtype != WQ_F32) return fail(WQ_ERR_DTYPE, "scale must be F32, got %s", dtname(sc->dtype));
  K = x->shape[x->ndim - 1];
  M = 1;
  for (int i = 0; i < x->ndim - 1; ++i) M *= x->shape[i];
  if (K < 1 || K > kMaxKN) return fail(WQ_ERR_SHAPE, "the last dimension must lie in [1, 65535]");
  if (M > kMaxRows) return fail(WQ_ERR_SHAPE, "more than 2^31-1 rows");
  if (sm && (sm->ndim != 1 || sm->shape[0] != K))
    return fail(WQ_ERR_SHAPE, "smooth_scales must be 1-D (k = %lld)", (long long)K);
  if (!same_shape(x, y)) return fail(WQ_ERR_SHAPE, "y must have x's (logical) shape");
  bits = y->dtype == WQ_INT8 ? 8 : 4;
  if (bits == 4 && K % 2 != 0) return fail(WQ_ERR_SHAPE, "INT4 output needs an even last dimension");
  if (numel(sc) != M || (x->ndim > 1 && (sc->ndim != x->ndim - 1 ||
                                         [&] { for (int i = 0; i < sc->ndim; ++i)
                                                 if (sc->shape[i] != x->shape[i]) return true;
                                               return false; }())))
    return fail(WQ_ERR_SHAPE, "scale must have x's leading shape");
  for (const wq_tensor *t : all)
    if (t && numel(t) > 0 && !t->data) return fail(WQ_ERR_NULL, "a non-empty tensor has no data");
  if (overlap(y, x) || overlap(y, sm) || overlap(y, sc) || overlap(sc, x) || overlap(sc, sm))
    return fail(WQ_ERR_ALIAS, "the outputs must not overlap the inputs or each other");
  return WQ_OK;
}

int32_t wq_dynamic_quant_get_workspace(const wq_tensor *x, const wq_tensor *sm, const wq_tensor *y,
                                       const wq_tensor *sc, uint64_t *ws_bytes) {
  if (!ws_bytes) return fail(WQ_ERR_NULL, "ws_bytes is required");
  int64_t M, K;
  int bits;
  int32_t st = validate_dq(x, sm, y, sc, M, K, bits);
  if (st) return st;
  *ws_bytes = 0;
  return ok();
}

int32_t wq_dynamic_quant(const wq_tensor *x, const wq_tensor *sm, const wq_tensor *y,
                         const wq_tensor *sc, void *ws, uint64_t ws_bytes, void *stream) {
  (void)ws; (void)ws_bytes;
  int64_t M, K;
  int bits;
  int32_t st = validate_dq(x, sm, y, sc, M, K, bits);
  if (st) return st;
  if (M == 0) return ok();
  cudaError_t e = launch_dynamic_quant(x->data, sm ? sm->data : nullptr, x->dtype, M, K, bits,
                                       y->data, static_cast<float *>(sc->data), (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "dynamic quantization launch");
  return ok();
}

// ------------------------------------------------------------------ matmul

int32_t wq_matmul_add_rmsnorm_get_workspace_ex(
    const wq_tensor *x1, const wq_tensor *x2, const wq_tensor *scale, const wq_tensor *offset,
    const wq_tensor *bias, const wq_tensor *residual, const wq_tensor *gamma, double eps,
    int64_t group, const wq_tensor *y, const wq_tensor *normOut, int32_t kernel,
    uint64_t *ws_bytes) {
  if (!ws_bytes) return fail(WQ_ERR_NULL, "ws_bytes is required");
  Problem p;
  int32_t st = validate(x1, x2, scale, offset, bias, residual, gamma, eps, group, y, normOut, p);
  if (st) return st;
  Plan plan;
  st = make_plan(p, kernel, plan);
  if (st) return st;
  *ws_bytes = plan.ws_bytes;
  return ok();
}

int32_t wq_matmul_add_rmsnorm_get_workspace(
    const wq_tensor *x1, const wq_tensor *x2, const wq_tensor *scale, const wq_tensor *offset,
    const wq_tensor *bias, const wq_tensor *residual, const wq_tensor *gamma, double eps,
    int64_t group, const wq_tensor *y, const wq_tensor *normOut, uint64_t *ws_bytes) {
  return wq_matmul_add_rmsnorm_get_workspace_ex(x1, x2, scale, offset, bias, residual, gamma, eps,
                                                group, y, normOut, WQ_KERNEL_AUTO, ws_bytes);
}

int32_t wq_matmul_add_rmsnorm_select_kernel(
    const wq_tensor *x1, const wq_tensor *x2, const wq_tensor *scale, const wq_tensor *offset,
    const wq_tensor *bias, const wq_tensor *residual, const wq_tensor *gamma, double eps,
    int64_t group, const wq_tensor *y, const wq_tensor *normOut) {
  Problem p;
  int32_t st = validate(x1, x2, scale, offset, bias, residual, gamma, eps, group, y, normOut, p);
  if (st) return -st;
  Plan plan;
  st = make_plan(p, WQ_KERNEL_AUTO, plan);
  if (st) return -st;
  ok();
  return plan.kernel;
}

int32_t wq_matmul_add_rmsnorm_ex(
    const wq_tensor *x1, const wq_tensor *x2, const wq_tensor *scale, const wq_tensor *offset,
    const wq_tensor *bias, const wq_tensor *residual, const wq_tensor *gamma, double eps,
    int64_t group, const wq_tensor *y, const wq_tensor *normOut, int32_t kernel, void *ws,
    uint64_t ws_bytes, void *stream) {
  Problem p;
  int32_t st = validate(x1, x2, scale, offset, bias, residual, gamma, eps, group, y, normOut, p);
  if (st) return st;
  Plan plan;
  st = make_plan(p, kernel, plan);
  if (st) return st;
  if (p.M == 0 || p.N == 0) return ok();
  if (ws_bytes < plan.ws_bytes || (plan.ws_bytes > 0 && !ws))
    return fail(WQ_ERR_WORKSPACE, "workspace of %llu bytes given, %llu needed",
                (unsigned long long)ws_bytes, (unsigned long long)plan.ws_bytes);
  if (((uintptr_t)ws) % 256 != 0)
    return fail(WQ_ERR_WORKSPACE, "workspace must be 256-byte aligned");
  cudaStream_t s = (cudaStream_t)stream;
  cudaError_t e;
  switch (plan.kernel) {
    case WQ_KERNEL_GENERIC:
      e = launch_generic(p, plan, ws, s);
      if (e != cudaSuccess) return cuda_fail(e, "generic kernel launch");
      e = launch_epilogue(p, plan, ws, false, s);
      if (e != cudaSuccess) return cuda_fail(e, "epilogue kernel launch");
      break;
    case WQ_KERNEL_PREFILL:
      e = plan.mode == 2 ? launch_prefill_t(p, plan, ws, s) : launch_prefill(p, plan, ws, s);
      if (e != cudaSuccess) return cuda_fail(e, "prefill kernel launch");
      break;
    case WQ_KERNEL_DECODE:
      e = p.tiled ? launch_decode_tiled(p, plan, ws, s) : launch_decode(p, plan, ws, s);
      if (e != cudaSuccess) return cuda_fail(e, "decode kernel launch");
      break;
    default:
      return fail(WQ_ERR_UNSUPPORTED, "kernel %d is not available", plan.kernel);
  }
  return ok();
}

int32_t wq_matmul_add_rmsnorm(
    const wq_tensor *x1, const wq_tensor *x2, const wq_tensor *scale, const wq_tensor *offset,
    const wq_tensor *bias, const wq_tensor *residual, const wq_tensor *gamma, double eps,
    int64_t group, const wq_tensor *y, const wq_tensor *normOut, void *ws, uint64_t ws_bytes,
    void *stream) {
  return wq_matmul_add_rmsnorm_ex(x1, x2, scale, offset, bias, residual, gamma, eps, group, y,
                                  normOut, WQ_KERNEL_AUTO, ws, ws_bytes, stream);
}

int32_t wq_read_device_status(const void *ws, uint64_t ws_bytes, void *stream,
                              int32_t *device_status) {
  if (!ws || !device_status) return fail(WQ_ERR_NULL, "ws and device_status are required");
  if (ws_bytes < 16) return fail(WQ_ERR_WORKSPACE, "workspace smaller than its status word");
  cudaStream_t s = (cudaStream_t)stream;
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "stream synchronize");
  uint32_t word = 0;
  e = cudaMemcpy(&word, ws, sizeof(word), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "status word copy");
  *device_status = (int32_t)word;
  return ok();
}

int32_t wq_check_device_timeout(void *ws, uint64_t ws_bytes, uint64_t budget_cycles,
                                void *stream) {
  if (!ws) return fail(WQ_ERR_NULL, "ws is required");
  if (ws_bytes < kWsHeader) return fail(WQ_ERR_WORKSPACE, "workspace smaller than its header");
  const uint64_t b = budget_cycles < 1000 ? 1000 : (budget_cycles > 4000000000ull ? 4000000000ull
                                                                                   : budget_cycles);
  cudaError_t e = launch_timeout_check(static_cast<uint32_t *>(ws), (long long)b,
                                       (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "self-check kernel launch");
  return ok();
}

int32_t wq_test_set_wait_limits(uint64_t budget_cycles, uint32_t extra_arrivals) {
  if (budget_cycles == 0 && extra_arrivals == 0) {
    g_wait_budget.store(kWaitBudget);
    g_wait_extra.store(0);
    return ok();
  }
  if (budget_cycles < 1000 || budget_cycles > (uint64_t)kWaitBudget)
    return fail(WQ_ERR_SHAPE, "budget_cycles must lie in [1000, %lld]", (long long)kWaitBudget);
  if (extra_arrivals > (1u << 20))
    return fail(WQ_ERR_SHAPE, "extra_arrivals must be at most 2^20");
  g_wait_budget.store((long long)budget_cycles);
  g_wait_extra.store(extra_arrivals);
  return ok();
}

}  // extern "C"
