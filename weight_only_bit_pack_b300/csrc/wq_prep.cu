// Per-call preparation passes of the prefill kernel.
//
// row_prep: for each row m of x1, the fp32 row sum (the factor of the offset
//   term when the offset is applied after the k-sum: sum_k x1[m,k]*O[n]) and,
//   for the fp16-operand mode, a power-of-two exponent e_m and an fp16 copy
//   x16[m,k] = x1[m,k] * 2^-e_m. bf16 -> fp16 is exact for every value in the
//   fp16 normal range; e_m is nonzero only for rows whose magnitude would
//   overflow fp16, and it is undone exactly in the epilogue.
// so_prep: for the fp16-operand mode, a per-column exponent e_n and fp16
//   copies S16 = S * 2^-e_n, O16 = O * 2^-e_n, chosen so that
//   qmax*|S16| + |O16| lies in [2^12, 2^13): then q*S16 is an exact fp16 value
//   for every 4-bit q (an 8-bit bf16 significand times a 3-bit integer fits the
//   11-bit fp16 significand), and only the offset add rounds, at 2^-12.
//   Each value is stored twice, as the two halves of a 32-bit word (the form
//   the packed fp16 arithmetic of the dequantization consumes). With `odd16`
//   the scale of every odd column is stored divided by 16 (exact): the kernel
//   reads those columns' nibbles in place at bits 7:4, i.e. as 16 q.
// Both passes are deterministic (fixed reduction order).
#include <cfloat>

#include "wq_common.cuh"
#include "wq_internal.h"

namespace wq {
namespace {

__device__ __forceinline__ float exp2i(int e) {
  // 2^e as an fp32 for e in [-126, 127]
  return __int_as_float((e + 127) << 23);
}

// Exponent e >= 0 such that amax * 2^-e < 2^14 (0 when it already is).
__device__ __forceinline__ int row_exponent(float amax) {
  if (!(amax >= 16384.f)) return 0;  // also 0 for NaN
  if (amax > FLT_MAX) return 0;       // inf: let it propagate
  int e;
  frexpf(amax, &e);                   // amax = f * 2^e, f in [0.5, 1)
  return e - 14;                      // amax * 2^-(e-14) < 2^14
}

template <int DT>
__global__ void __launch_bounds__(256)
    row_prep_kernel(const typename Elem<DT>::T *__restrict__ x1, int64_t M, int K,
                    float *__restrict__ rowsum, int8_t *__restrict__ e_row, __half *__restrict__ x16) {
  const int lane = threadIdx.x & 31;
  const int64_t warp0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  for (int64_t m = warp0; m < M; m += nwarps) {
    const typename Elem<DT>::T *row = x1 + m * K;
    float s = 0.f, amax = 0.f;
    // K % 8 == 0 (prefill precondition): 16-byte vectors of 8 values
#pragma unroll 4
    for (int k = lane * 8; k < K; k += 256) {
      const uint4 v = *reinterpret_cast<const uint4 *>(row + k);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 f = unpack2<DT>(w[i]);
        s += f.x;
        s += f.y;
        amax = fmaxf(amax, fmaxf(fabsf(f.x), fabsf(f.y)));
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      s += __shfl_xor_sync(0xffffffffu, s, o);
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    }
    if (rowsum && lane == 0) rowsum[m] = s;
    if (x16) {
      const int e = row_exponent(amax);
      if (lane == 0) e_row[m] = (int8_t)e;
      const float sc = exp2i(-e);
      __half *out = x16 + m * K;
#pragma unroll 4
      for (int k = lane * 8; k < K; k += 256) {
        const uint4 v = *reinterpret_cast<const uint4 *>(row + k);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        uint32_t o[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float2 f = unpack2<DT>(w[i]);
          o[i] = pack2<WQ_F16>(f.x * sc, f.y * sc);
        }
        *reinterpret_cast<uint4 *>(out + k) = make_uint4(o[0], o[1], o[2], o[3]);
      }
    }
  }
}

// One block covers 32 columns; its 8 warps split the group rows, so every warp
// load reads 32 consecutive columns (coalesced) and the G loads of a column
// are spread over 8 warps.
__device__ __forceinline__ uint32_t half_pair(float v) {
  const __half h = __float2half_rn(v);
  const uint32_t b = (uint32_t)__half_as_ushort(h);
  return b | (b << 16);
}

template <int DT>
__global__ void __launch_bounds__(256)
    so_prep_kernel(const typename Elem<DT>::T *__restrict__ S, const typename Elem<DT>::T *__restrict__ O,
                   int G, int N, int ld, float qmax, int int4, int8_t *__restrict__ e_col,
                   uint32_t *__restrict__ S16, uint32_t *__restrict__ O16) {
  using E = Elem<DT>;
  __shared__ float s_max[8][32];
  __shared__ float s_scale[32];
  const int cx = threadIdx.x & 31, gy = threadIdx.x >> 5;
  const int n = blockIdx.x * 32 + cx;
  float mx = 0.f;
  if (n < N) {
#pragma unroll 4
    for (int g = gy; g < G; g += 8) {
      const float sv = fabsf(E::to_f(S[(int64_t)g * N + n]));
      const float ov = O ? fabsf(E::to_f(O[(int64_t)g * N + n])) : 0.f;
      mx = fmaxf(mx, fmaf(qmax, sv, ov));
    }
  }
  s_max[gy][cx] = mx;
  __syncthreads();
  if (gy == 0) {
    float m = s_max[0][cx];
#pragma unroll
    for (int i = 1; i < 8; ++i) m = fmaxf(m, s_max[i][cx]);
    int e = 0;
    if (m > 0.f && m <= FLT_MAX) {
      int ex;
      frexpf(m, &ex);  // m in [2^(ex-1), 2^ex)
      e = ex - 13;     // m * 2^-e in [2^12, 2^13)
      if (e < -100) e = -100;
      if (e > 100) e = 100;
    }
    if (n < N) e_col[n] = (int8_t)e;
    s_scale[cx] = exp2i(-e);
  }
  __syncthreads();
  // Destination word of column n in a row of ld words. INT4: within each
  // 256-column tile, column 8l + i goes to word 4l + i (i < 4) or 128 + 4l +
  // (i - 4), so that the dequant lane l reads its eight columns as two 16-byte
  // chunks that the warp's lanes take side by side (no bank conflicts); the
  // rows are padded to whole tiles (ld >= N), the padding holds zeros.
  int dst = n;
  if (int4) {
    const int c = n & 255, l = c >> 3, i = c & 7;
    dst = (n - c) + (i < 4 ? 4 * l + i : 128 + 4 * l + (i - 4));
  }
  if (n < ld) {
    const float sc = s_scale[cx];
    const float ssc = (int4 && (n & 1)) ? sc * 0.0625f : sc;  // exact power-of-two factors
#pragma unroll 4
    for (int g = gy; g < G; g += 8) {
      const bool live = n < N;
      S16[(int64_t)g * ld + dst] = live ? half_pair(E::to_f(S[(int64_t)g * N + n]) * ssc) : 0u;
      if (O) O16[(int64_t)g * ld + dst] = live ? half_pair(E::to_f(O[(int64_t)g * N + n]) * sc) : 0u;
    }
  }
}

}  // namespace

cudaError_t launch_row_prep(const Problem &p, float *rowsum, int8_t *e_row, __half *x16,
                            cudaStream_t s) {
  const int64_t warps_needed = p.M;
  int64_t blocks = (warps_needed * 32 + 255) / 256;
  const int64_t cap = (int64_t)device_info().sms * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  if (p.dtype == WQ_BF16)
    row_prep_kernel<WQ_BF16><<<(unsigned)blocks, 256, 0, s>>>(
        static_cast<const __nv_bfloat16 *>(p.x1), p.M, (int)p.K, rowsum, e_row, x16);
  else
    row_prep_kernel<WQ_F16><<<(unsigned)blocks, 256, 0, s>>>(static_cast<const __half *>(p.x1), p.M,
                                                             (int)p.K, rowsum, e_row, x16);
  return cudaGetLastError();
}

cudaError_t launch_so_prep(const Problem &p, int64_t ld, int8_t *e_col, uint32_t *S16,
                           uint32_t *O16, cudaStream_t s) {
  const int N = (int)p.N;
  const int blocks = (int)((ld + 31) / 32);
  const float qmax = p.wbits == 4 ? 8.f : 128.f;
  const int int4 = p.wbits == 4 ? 1 : 0;
  if (p.dtype == WQ_BF16)
    so_prep_kernel<WQ_BF16><<<blocks, 256, 0, s>>>(static_cast<const __nv_bfloat16 *>(p.scale),
                                                   static_cast<const __nv_bfloat16 *>(p.offset),
                                                   (int)p.G, N, (int)ld, qmax, int4, e_col, S16, O16);
  else
    so_prep_kernel<WQ_F16><<<blocks, 256, 0, s>>>(static_cast<const __half *>(p.scale),
                                                  static_cast<const __half *>(p.offset), (int)p.G,
                                                  N, (int)ld, qmax, int4, e_col, S16, O16);
  return cudaGetLastError();
}

}  // namespace wq
