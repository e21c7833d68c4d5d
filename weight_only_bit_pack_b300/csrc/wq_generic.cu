// Generic weight-only quantized matmul: a predicated CUDA-core kernel that is
// correct for every shape the ABI accepts (odd n, k not a multiple of anything,
// any alignment). It writes split-K partial sums of x1 @ W (no bias) into the
// workspace; the shared epilogue kernel then adds bias and residual and applies
// RMSNorm (aclnnWeightQuantMatmulAllReduceAddRmsNorm, "Function description").
//
// W[k][n] = q[k][n] * S[r(k)][c(n)] + O[r(k)][c(n)] is formed in fp32 (q*S is
// exact in fp32; adding O rounds once), r(k) = floor(k/group) or 0, c(n) = n or
// 0. One thread owns one column n and eight rows; each block covers 128
// columns, one split of k, and a grid-stride range of 8-row blocks. The weight
// is INT8, dense INT4 or INT4 in the kernel-native tiled layout (LAYOUT 8, 4, 6),
// or transposed -- stored (N, K), K contiguous -- as INT8 (LAYOUT 10) or INT4
// packed along K (LAYOUT 9).
#include "wq_internal.h"
#include "wq_common.cuh"

namespace wq {
namespace {

constexpr int kGenThreads = 128;
constexpr int kGenRows = 8;

template <int DT, int LAYOUT>
__global__ void __launch_bounds__(kGenThreads)
    generic_gemm_kernel(const typename Elem<DT>::T *__restrict__ x1, const uint8_t *__restrict__ x2,
                        const typename Elem<DT>::T *__restrict__ S,
                        const typename Elem<DT>::T *__restrict__ O, int64_t M, int64_t K, int64_t N,
                        int64_t group, int64_t Ns, int64_t ksplit, float *__restrict__ part) {
  using E = Elem<DT>;
  const int64_t n = (int64_t)blockIdx.x * kGenThreads + threadIdx.x;
  const int64_t s = blockIdx.y;
  const int64_t k0 = s * ksplit;
  const int64_t k1 = (k0 + ksplit < K) ? k0 + ksplit : K;
  if (n >= N) return;
  const int64_t c = (Ns == 1) ? 0 : n;
  for (int64_t m0 = (int64_t)blockIdx.z * kGenRows; m0 < M; m0 += (int64_t)gridDim.z * kGenRows) {
    float acc[kGenRows];
#pragma unroll
    for (int i = 0; i < kGenRows; ++i) acc[i] = 0.f;
    for (int64_t k = k0; k < k1; ++k) {
      int q;
      if (LAYOUT == 4) {
        const uint32_t b = x2[k * (N / 2) + (n >> 1)];
        const int nib = (n & 1) ? (int)(b >> 4) : (int)(b & 0xFu);
        q = nib >= 8 ? nib - 16 : nib;
      } else if (LAYOUT == 6) {
        const int nib = (int)tiled_nibble(x2, k, n, N);
        q = nib >= 8 ? nib - 16 : nib;
      } else if (LAYOUT == 9) {
        const uint32_t b = x2[n * (K / 2) + (k >> 1)];
        const int nib = (k & 1) ? (int)(b >> 4) : (int)(b & 0xFu);
        q = nib >= 8 ? nib - 16 : nib;
      } else if (LAYOUT == 10) {
        q = (int)reinterpret_cast<const int8_t *>(x2)[n * K + k];
      } else {
        q = (int)reinterpret_cast<const int8_t *>(x2)[k * N + n];
      }
      const int64_t r = group > 0 ? k / group : 0;
      float w = (float)q * E::to_f(S[r * Ns + c]);
      if (O) w += E::to_f(O[r * Ns + c]);
#pragma unroll
      for (int i = 0; i < kGenRows; ++i)
        if (m0 + i < M) acc[i] = fmaf(E::to_f(x1[(m0 + i) * K + k]), w, acc[i]);
    }
#pragma unroll
    for (int i = 0; i < kGenRows; ++i)
      if (m0 + i < M) part[(s * M + m0 + i) * N + n] = acc[i];
  }
}

}  // namespace

bool plan_generic(const Problem &p, Plan &plan) {
  const int64_t nb = (p.N + kGenThreads - 1) / kGenThreads;
  int64_t mb = (p.M + kGenRows - 1) / kGenRows;
  if (mb > 65535) mb = 65535;
  const int64_t ctas = nb * mb;
  const int64_t want = 2LL * device_info().sms;
  int64_t S = (want + ctas - 1) / ctas;
  int64_t smax = p.K / 32 > 0 ? p.K / 32 : 1;
  if (S > smax) S = smax;
  if (S > 64) S = 64;
  if (S < 1) S = 1;
  int64_t ksplit = (p.K + S - 1) / S;
  S = (p.K + ksplit - 1) / ksplit;
  plan.kernel = WQ_KERNEL_GENERIC;
  plan.parts = (int)S;
  plan.ksplit = ksplit;
  plan.part_off = kWsHeader;
  plan.ws_bytes = kWsHeader + (uint64_t)S * (uint64_t)p.M * (uint64_t)p.N * sizeof(float);
  return true;
}

cudaError_t launch_generic(const Problem &p, const Plan &plan, void *ws, cudaStream_t s) {
  const int64_t nb = (p.N + kGenThreads - 1) / kGenThreads;
  int64_t mb = (p.M + kGenRows - 1) / kGenRows;
  if (mb > 65535) mb = 65535;
  dim3 grid((unsigned)nb, (unsigned)plan.parts, (unsigned)mb);
  float *part = reinterpret_cast<float *>(static_cast<char *>(ws) + plan.part_off);
  const uint8_t *x2 = static_cast<const uint8_t *>(p.x2);
#define WQ_GEN_LAUNCH(DT, LAYOUT)                                                                 \
  generic_gemm_kernel<DT, LAYOUT><<<grid, kGenThreads, 0, s>>>(                                   \
      static_cast<const Elem<DT>::T *>(p.x1), x2, static_cast<const Elem<DT>::T *>(p.scale),      \
      static_cast<const Elem<DT>::T *>(p.offset), p.M, p.K, p.N, p.group, p.Ns, plan.ksplit, part)
  const int layout = p.transposed ? (p.wbits == 8 ? 10 : 9)
                                  : (p.wbits == 8 ? 8 : (p.tiled ? 6 : 4));
#define WQ_GEN_LAYOUTS(DT)                                       \
  switch (layout) {                                              \
    case 4: WQ_GEN_LAUNCH(DT, 4); break;                         \
    case 6: WQ_GEN_LAUNCH(DT, 6); break;                         \
    case 9: WQ_GEN_LAUNCH(DT, 9); break;                         \
    case 10: WQ_GEN_LAUNCH(DT, 10); break;                       \
    default: WQ_GEN_LAUNCH(DT, 8); break;                        \
  }
  if (p.dtype == WQ_BF16) {
    WQ_GEN_LAYOUTS(WQ_BF16)
  } else {
    WQ_GEN_LAYOUTS(WQ_F16)
  }
#undef WQ_GEN_LAYOUTS
#undef WQ_GEN_LAUNCH
  return cudaGetLastError();
}

}  // namespace wq
