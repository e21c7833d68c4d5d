// FP4 E2M1 pack and the mx block-scaled matmul with in-place add.
//
// Pack (aclnnConvertWeightToINT4Pack, "Function description": FLOAT weights
// packed into dense FLOAT4_E2M1): each fp32 becomes the nearest E2M1 value
// (magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6; ties to the even code; saturating at
// 6) by the hardware conversion cvt.rn.satfinite.e2m1x2.f32, two codes per byte
// along the last dimension, the even column in bits 3:0 (as the INT4 pack).
// HBM-bound: 4 bytes read and half a byte written per element.
//
// mx matmul (aclnnQuantBatchMatmulInplaceAdd, "Function description", mx
// quantization; x1 as given or transposed, (K, M) in memory, the form the
// page's constraints list): y[m,n] += sum_j (sum_{k in slice j} x1[m,k] x2[k,n]) *
// scale1[m,j] * scale2[j,n], slices of gsK = 32 along K (the last one may be
// short), FP4 E2M1 operands and E8M0 scales (byte e = 2^(e - 127), 255 = NaN).
// A CUDA-core kernel: one thread per output column n and 8 rows; a slice's sum
// of at most 32 products of E2M1 values is exact in fp32 (multiples of 1/4
// below 2^11), the scaled slices are added in fp64, and the result is rounded
// once to fp32 when it is added to y.
#include "wq_common.cuh"
#include "wq_internal.h"

namespace wq {
namespace {

__device__ __forceinline__ uint32_t e2m1x2(float even, float odd) {
  uint16_t r;
  asm("{\n\t.reg .b8 t;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\t"  // first source -> bits 7:4
      "mov.b16 %0, {t, 0};\n\t}"
      : "=h"(r)
      : "f"(odd), "f"(even));
  return r & 0xFFu;
}

__global__ void __launch_bounds__(256) pack_fp4_kernel(const float *__restrict__ in,
                                                      uint8_t *__restrict__ out, int64_t nvec,
                                                      int64_t tail_begin, int64_t nbytes) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  for (int64_t i = tid; i < nvec; i += stride) {  // 8 floats -> 4 bytes
    const float4 a = __ldcs(reinterpret_cast<const float4 *>(in) + 2 * i);
    const float4 b = __ldcs(reinterpret_cast<const float4 *>(in) + 2 * i + 1);
    const uint32_t w = e2m1x2(a.x, a.y) | (e2m1x2(a.z, a.w) << 8) | (e2m1x2(b.x, b.y) << 16) |
                       (e2m1x2(b.z, b.w) << 24);
    __stcs(reinterpret_cast<uint32_t *>(out) + i, w);
  }
  for (int64_t j = tail_begin + tid; j < nbytes; j += stride) out[j] = (uint8_t)e2m1x2(in[2 * j], in[2 * j + 1]);
}

constexpr int kMxThreads = 128, kMxRows = 8, kGs = 32;

// Value of an E2M1 code: sign (bit 3), exponent e (bits 2:1), mantissa m (bit 0);
// e = 0 is 0 or 0.5, otherwise 2^(e-1) * (1 + m/2).
__device__ __forceinline__ float e2m1_value(uint32_t code) {
  const uint32_t e = (code >> 1) & 3u, m = code & 1u;
  const float v = e ? __int_as_float((int)(((e + 126u) << 23) | (m << 22))) : 0.5f * (float)m;
  return (code & 8u) ? -v : v;
}

// grid (ceil(N / 128), <= 65535 row blocks); thread = column n, 8 rows per block.
// X1T: x1 stored (K, M) packed along M, scale1 stored (J, M).
template <bool X1T>
__global__ void __launch_bounds__(kMxThreads)
    mx_matmul_add_kernel(const uint8_t *__restrict__ x1, const uint8_t *__restrict__ s1,
                         const uint8_t *__restrict__ x2, const uint8_t *__restrict__ s2,
                         float *__restrict__ y, int64_t M, int64_t K, int64_t N) {
  __shared__ float xs[kMxRows][kGs];
  __shared__ uint8_t ss[kMxRows];
  const int64_t n = (int64_t)blockIdx.x * kMxThreads + threadIdx.x;
  const int64_t J = (K + kGs - 1) / kGs;
  for (int64_t m0 = (int64_t)blockIdx.y * kMxRows; m0 < M; m0 += (int64_t)gridDim.y * kMxRows) {
    double acc[kMxRows];
#pragma unroll
    for (int r = 0; r < kMxRows; ++r) acc[r] = 0.0;
    for (int64_t j = 0; j < J; ++j) {
      const int64_t k0 = j * kGs, klen = K - k0 < kGs ? K - k0 : kGs;
      __syncthreads();  // the previous slice's operands have been used
      for (int i = threadIdx.x; i < kMxRows * kGs; i += kMxThreads) {
        const int r = i / kGs, kk = i % kGs;
        float v = 0.f;
        if (m0 + r < M && kk < klen) {
          const int64_t k = k0 + kk, m = m0 + r;
          if constexpr (X1T) {
            const uint32_t b = x1[k * (M / 2) + m / 2];
            v = e2m1_value((m & 1) ? (b >> 4) : (b & 15u));
          } else {
            const uint32_t b = x1[m * (K / 2) + k / 2];
            v = e2m1_value((k & 1) ? (b >> 4) : (b & 15u));
          }
        }
        xs[r][kk] = v;
      }
      if (threadIdx.x < kMxRows) {
        const int64_t m = m0 + threadIdx.x;
        ss[threadIdx.x] = m < M ? (X1T ? s1[j * M + m] : s1[m * J + j]) : 127;
      }
      __syncthreads();
      if (n >= N) continue;
      float slice[kMxRows];
#pragma unroll
      for (int r = 0; r < kMxRows; ++r) slice[r] = 0.f;
      for (int kk = 0; kk < klen; ++kk) {
        const uint32_t b = x2[(k0 + kk) * (N / 2) + n / 2];
        const float w = e2m1_value((n & 1) ? (b >> 4) : (b & 15u));
#pragma unroll
        for (int r = 0; r < kMxRows; ++r) slice[r] = fmaf(xs[r][kk], w, slice[r]);  // exact
      }
      const uint32_t e2 = s2[j * N + n];
#pragma unroll
      for (int r = 0; r < kMxRows; ++r) {
        const uint32_t e1 = ss[r];
        if (e1 == 255u || e2 == 255u)
          acc[r] += __longlong_as_double(0x7FF8000000000000LL);  // an E8M0 NaN scale
        else
          acc[r] += ldexp((double)slice[r], (int)e1 + (int)e2 - 254);
      }
    }
    if (n < N) {
#pragma unroll
      for (int r = 0; r < kMxRows; ++r)
        if (m0 + r < M) y[(m0 + r) * N + n] = (float)((double)y[(m0 + r) * N + n] + acc[r]);
    }
    __syncthreads();  // the next row block refills the shared operands
  }
}

}  // namespace

cudaError_t launch_pack_fp4(const float *in, uint8_t *out, int64_t K, int64_t N, cudaStream_t s) {
  const int64_t nbytes = K * (N / 2);
  const bool aligned = ((uintptr_t)in % 16 == 0) && ((uintptr_t)out % 4 == 0);
  const int64_t nvec = aligned ? nbytes / 4 : 0;
  const int64_t tail = nvec * 4;
  int64_t blocks = ((nvec > 0 ? nvec : nbytes - tail) + 255) / 256;
  const int64_t cap = (int64_t)device_info().sms * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  pack_fp4_kernel<<<(unsigned)blocks, 256, 0, s>>>(in, out, nvec, tail, nbytes);
  return cudaGetLastError();
}

cudaError_t launch_mx_matmul_add(const uint8_t *x1, const uint8_t *s1, bool x1t, const uint8_t *x2,
                                 const uint8_t *s2, float *y, int64_t M, int64_t K, int64_t N,
                                 cudaStream_t s) {
  int64_t rows = (M + kMxRows - 1) / kMxRows;
  if (rows > 65535) rows = 65535;
  const dim3 grid((unsigned)((N + kMxThreads - 1) / kMxThreads), (unsigned)rows, 1);
  if (x1t)
    mx_matmul_add_kernel<true><<<grid, kMxThreads, 0, s>>>(x1, s1, x2, s2, y, M, K, N);
  else
    mx_matmul_add_kernel<false><<<grid, kMxThreads, 0, s>>>(x1, s1, x2, s2, y, M, K, N);
  return cudaGetLastError();
}

}  // namespace wq
