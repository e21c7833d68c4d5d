// Per-token symmetric dynamic quantization of activations (aclnnDynamicQuant,
// "Function description": scaleOut = row_max(|x|) / dtypeMax, yOut =
// round(x / scaleOut), with x first multiplied by smoothScales per column when
// they are given) -- the step that feeds a quantized-activation matmul.
//
// One CTA per row: the row is read from HBM once into shared memory (16-byte
// loads when the row is 16-byte aligned), its absolute maximum is reduced in the
// CTA, and the codes are formed from the shared copy and written as INT8 or as
// INT4 packed two per byte along the row (the element of even column 2j in bits
// 3:0 of byte j, as the weight pack). Every floating-point step is one IEEE fp32
// operation -- x * smooth, the maximum, max / dtypeMax, x / scale -- and the
// code is the round-half-to-even integer of the quotient (cvt.rni), clamped to
// [-dtypeMax, dtypeMax], with a NaN quotient giving 0; a row whose maximum is 0
// gets scale 0 and codes 0. The kernel is bound by HBM: 2 bytes read and 1 (or
// 1/2) written per element.
#include <cfloat>

#include "wq_common.cuh"
#include "wq_internal.h"

namespace wq {
namespace {

constexpr int kDqThreads = 256;

template <int DT, int BITS, bool VEC>
__global__ void __launch_bounds__(kDqThreads)
    dynamic_quant_kernel(const typename Elem<DT>::T *__restrict__ x,
                         const typename Elem<DT>::T *__restrict__ smooth, int64_t M, int K,
                         uint8_t *__restrict__ y, float *__restrict__ scale) {
  using E = Elem<DT>;
  using T = typename E::T;
  constexpr int QMAX = BITS == 8 ? 127 : 7;
  extern __shared__ __align__(16) uint8_t dq_smem[];
  T *row = reinterpret_cast<T *>(dq_smem);
  __shared__ float s_max[kDqThreads / 32];
  __shared__ float s_scale;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  for (int64_t m = blockIdx.x; m < M; m += gridDim.x) {
    const T *xr = x + m * K;
    float amax = 0.f;
    if constexpr (VEC) {  // K % 8 == 0 and 16-byte aligned rows
      for (int k = 8 * tid; k < K; k += 8 * kDqThreads) {
        const uint4 v = *reinterpret_cast<const uint4 *>(xr + k);
        *reinterpret_cast<uint4 *>(row + k) = v;
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          float2 f = unpack2<DT>(w[i]);
          if (smooth) {
            f.x = __fmul_rn(f.x, E::to_f(smooth[k + 2 * i]));
            f.y = __fmul_rn(f.y, E::to_f(smooth[k + 2 * i + 1]));
          }
          amax = fmaxf(amax, fmaxf(fabsf(f.x), fabsf(f.y)));
        }
      }
    } else {
      for (int k = tid; k < K; k += kDqThreads) {
        const T v = xr[k];
        row[k] = v;
        float f = E::to_f(v);
        if (smooth) f = __fmul_rn(f, E::to_f(smooth[k]));
        amax = fmaxf(amax, fabsf(f));
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    if (lane == 0) s_max[warp] = amax;
    __syncthreads();
    if (tid == 0) {
      float mx = s_max[0];
      for (int w = 1; w < kDqThreads / 32; ++w) mx = fmaxf(mx, s_max[w]);
      const float s = __fdiv_rn(mx, (float)QMAX);
      s_scale = s;
      scale[m] = s;
    }
    __syncthreads();
    const float s = s_scale;
    // the code of f: rint(fl(f / s)) (IEEE division, ties to even), clamped; NaN -> 0
    auto code_of = [&](float f) -> int {
      if (s == 0.f) return 0;
      const int c = __float2int_rn(__fdiv_rn(f, s));
      return c > QMAX ? QMAX : (c < -QMAX ? -QMAX : c);
    };
    auto code = [&](int k) -> int {
      float f = E::to_f(row[k]);
      if (smooth) f = __fmul_rn(f, E::to_f(smooth[k]));
      return code_of(f);
    };
    uint8_t *yr = y + (BITS == 8 ? m * K : m * (K / 2));
    if constexpr (VEC) {
      // 8 elements per step: one 16-byte shared read, one 8-byte (INT8) or
      // 4-byte (INT4) store
      for (int k = 8 * tid; k < K; k += 8 * kDqThreads) {
        const uint4 v = *reinterpret_cast<const uint4 *>(row + k);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        int c[8];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          float2 f = unpack2<DT>(w[i]);
          if (smooth) {
            f.x = __fmul_rn(f.x, E::to_f(smooth[k + 2 * i]));
            f.y = __fmul_rn(f.y, E::to_f(smooth[k + 2 * i + 1]));
          }
          c[2 * i] = code_of(f.x);
          c[2 * i + 1] = code_of(f.y);
        }
        if constexpr (BITS == 8) {
          uint32_t lo = 0, hi = 0;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            lo |= (uint32_t)(c[i] & 0xFF) << (8 * i);
            hi |= (uint32_t)(c[4 + i] & 0xFF) << (8 * i);
          }
          *reinterpret_cast<uint2 *>(yr + k) = make_uint2(lo, hi);
        } else {
          uint32_t wq4 = 0;
#pragma unroll
          for (int i = 0; i < 8; ++i) wq4 |= (uint32_t)(c[i] & 0xF) << (4 * i);
          *reinterpret_cast<uint32_t *>(yr + k / 2) = wq4;
        }
      }
    } else if constexpr (BITS == 8) {
      for (int k = tid; k < K; k += kDqThreads) yr[k] = (uint8_t)(int8_t)code(k);
    } else {
      for (int j = tid; j < K / 2; j += kDqThreads)
        yr[j] = (uint8_t)((code(2 * j) & 0xF) | ((code(2 * j + 1) & 0xF) << 4));
    }
    __syncthreads();  // the shared row is reused by the next row of this CTA
  }
}

}  // namespace

cudaError_t launch_dynamic_quant(const void *x, const void *smooth, int dtype, int64_t M, int64_t K,
                                 int bits, void *y, float *scale, cudaStream_t s) {
  // the vector path also stores 8 (INT8) or 4 (INT4) bytes at a time
  const bool vec = K % 8 == 0 && reinterpret_cast<uintptr_t>(x) % 16 == 0 &&
                   reinterpret_cast<uintptr_t>(y) % 8 == 0;
  const size_t smem = (size_t)K * 2;
  int64_t grid = M;
  const int64_t cap = (int64_t)device_info().sms * 64;
  if (grid > cap) grid = cap;
  cudaError_t e = cudaSuccess;
#define WQ_DQ(DT, BITS, VEC)                                                                      \
  do {                                                                                            \
    auto kern = dynamic_quant_kernel<DT, BITS, VEC>;                                              \
    if (smem > 48 * 1024) {                                                                       \
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);     \
      if (e != cudaSuccess) return e;                                                             \
    }                                                                                             \
    kern<<<(unsigned)grid, kDqThreads, smem, s>>>(                                                \
        static_cast<const Elem<DT>::T *>(x), static_cast<const Elem<DT>::T *>(smooth), M, (int)K, \
        static_cast<uint8_t *>(y), scale);                                                        \
  } while (0)
  if (dtype == WQ_BF16) {
    if (bits == 8) { if (vec) WQ_DQ(WQ_BF16, 8, true); else WQ_DQ(WQ_BF16, 8, false); }
    else { if (vec) WQ_DQ(WQ_BF16, 4, true); else WQ_DQ(WQ_BF16, 4, false); }
  } else {
    if (bits == 8) { if (vec) WQ_DQ(WQ_F16, 8, true); else WQ_DQ(WQ_F16, 8, false); }
    else { if (vec) WQ_DQ(WQ_F16, 4, true); else WQ_DQ(WQ_F16, 4, false); }
  }
#undef WQ_DQ
  return cudaGetLastError();
}

}  // namespace wq
