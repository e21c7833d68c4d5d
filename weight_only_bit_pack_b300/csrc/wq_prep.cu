// Per-call preparation passes of the prefill kernel.
//
// row_prep: for each row m of x1, the fp32 row sum (the factor of the offset
//   term when the offset is applied after the k-sum: sum_k x1[m,k]*O[n]) and,
//   for the fp16-operand mode, a power-of-two exponent e_m and an fp16 copy
//   x16[m,k] = x1[m,k] * 2^-e_m. e_m puts the row's largest magnitude into
//   [2^13, 2^14), scaling small rows up as well as large rows down, so every
//   element within a factor 2^27 of the row maximum converts to fp16 exactly
//   (bf16 has 8 significant bits, fp16 11 above 2^-14 and its subnormals reach
//   2^-24). Elements further below the maximum round (or flush to zero): their
//   share of any dot product is below 2^-27 of the largest term's. Rows that are
//   all zero or hold an Inf get e_m = 0 (NaN and Inf then propagate). e_m is
//   undone exactly in the epilogue.
//   With an offset, row_prep also writes the operand of the offset term
//   sum_g O[g][n] * d[m][g], d[m][g] = sum of x16[m][k] over group g (fp32, in
//   ascending k): each d split into two bf16 parts hi + lo (together within
//   2^-18 of d), stored as row m of an (M, ldx) bf16 array [hi | lo | zero
//   padding], ldx = 2G rounded up to 64.
// so_prep: for the fp16-operand mode, a per-column exponent e_n and fp16
//   copies S16 = S * 2^-e_n chosen so that qmax*|S16| lies in [2^12, 2^13):
//   then for 4-bit q, q*S16 is an exact fp16 value (an 8-bit bf16 significand
//   times a 3-bit integer fits the 11-bit fp16 significand) as long as S16
//   stays in the fp16 normal range (scales within 2^25 of the column's
//   largest). For 8-bit q the product needs up to 15 bits and is rounded once
//   to fp16 (relative error at most 2^-11 of q*S). Each value is stored twice,
//   as the two halves of a 32-bit word (the form the packed fp16 arithmetic of
//   the dequantization consumes). With `odd16` the scale of every odd column is
//   stored divided by 16 (exact): the kernel reads those columns' nibbles in
//   place at bits 7:4, i.e. as 16 q. With an offset, the offsets scaled by the
//   same 2^-e_n (exact in bf16, which has fp32's exponent range) go to an
//   (N, ldx) bf16 array whose row n is [O' | O' | zero padding], the K-major
//   operand that multiplies the hi and lo parts of d.
// Both passes are deterministic (fixed reduction order).
#include <cfloat>

#include "wq_common.cuh"
#include "wq_internal.h"

namespace wq {
namespace {

// floor(log2(v)) of a finite v > 0, subnormals included.
__device__ __forceinline__ int ilog2f(float v) {
  if (v < 1.17549435e-38f) return ((__float_as_int(v * 18446744073709551616.f) >> 23) & 0xFF) - 127 - 64;
  return ((__float_as_int(v) >> 23) & 0xFF) - 127;
}

// Exponent e with amax * 2^-e in [2^13, 2^14) for a finite amax > 0; 0 for a
// zero row and for a row whose maximum is Inf or NaN.
__device__ __forceinline__ int row_exponent(float amax) {
  if (!(amax > 0.f) || amax > FLT_MAX) return 0;
  return ilog2f(amax) - 13;
}

template <int DT>
__global__ void __launch_bounds__(256)
    row_prep_kernel(const typename Elem<DT>::T *__restrict__ x1, int64_t M, int K,
                    float *__restrict__ rowsum, int16_t *__restrict__ e_row, __half *__restrict__ x16,
                    __nv_bfloat16 *__restrict__ dext, int group, int G, int ldx) {
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
      if (lane == 0) e_row[m] = (int16_t)e;
      __half *out = x16 + m * K;
#pragma unroll 4
      for (int k = lane * 8; k < K; k += 256) {
        const uint4 v = *reinterpret_cast<const uint4 *>(row + k);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        uint32_t o[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float2 f = unpack2<DT>(w[i]);
          o[i] = pack2<WQ_F16>(scale_pow2(f.x, -e), scale_pow2(f.y, -e));
        }
        *reinterpret_cast<uint4 *>(out + k) = make_uint4(o[0], o[1], o[2], o[3]);
      }
      if (dext) {
        // per-group sums of the fp16 row just written (the warp's own stores:
        // __syncwarp orders them before the loads of the other lanes)
        __syncwarp();
        __nv_bfloat16 *drow = dext + m * ldx;
        for (int gi = lane; gi < G; gi += 32) {
          const int k0 = gi * group, k1 = k0 + group < K ? k0 + group : K;
          float d = 0.f;
          for (int k = k0; k < k1; k += 8) {  // group % 32 == 0 and K % 8 == 0
            const uint4 v = *reinterpret_cast<const uint4 *>(out + k);
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const float2 f = unpack2<WQ_F16>(w[i]);
              d += f.x;
              d += f.y;
            }
          }
          // d = hi + lo to 2^-18, each bf16 (the difference d - hi is exact in fp32)
          const __nv_bfloat16 hi = __float2bfloat16_rn(d);
          const __nv_bfloat16 lo = __float2bfloat16_rn(d - __bfloat162float(hi));
          drow[gi] = hi;
          drow[G + gi] = lo;
        }
        for (int j = 2 * G + lane; j < ldx; j += 32) drow[j] = __float2bfloat16_rn(0.f);
      }
    }
  }
}

// The same fp16 copy, row exponent and (dext) group sums, one 256-thread block
// per row holding the row in registers (R 16-byte vectors a thread, K <= 2048 R):
// the row is read from memory once instead of twice.
template <int DT, int R>
__global__ void __launch_bounds__(256)
    row_prep_reg_kernel(const typename Elem<DT>::T *__restrict__ x1, int64_t M, int K,
                        int16_t *__restrict__ e_row, __half *__restrict__ x16,
                        __nv_bfloat16 *__restrict__ dext, int group, int G, int ldx) {
  __shared__ float red[8];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int64_t m = blockIdx.x; m < M; m += gridDim.x) {
    const typename Elem<DT>::T *row = x1 + m * K;
    uint4 v[R];
    float amax = 0.f;
#pragma unroll
    for (int j = 0; j < R; ++j) {
      const int k = (j * 256 + tid) * 8;  // K % 8 == 0
      v[j] = k < K ? *reinterpret_cast<const uint4 *>(row + k) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int j = 0; j < R; ++j) {
      const uint32_t w[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 f = unpack2<DT>(w[i]);
        amax = fmaxf(amax, fmaxf(fabsf(f.x), fabsf(f.y)));
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    if (lane == 0) red[warp] = amax;
    __syncthreads();
    amax = red[0];
#pragma unroll
    for (int i = 1; i < 8; ++i) amax = fmaxf(amax, red[i]);
    __syncthreads();  // red is rewritten for the next row only after every read
    const int e = row_exponent(amax);
    if (tid == 0) e_row[m] = (int16_t)e;
    __half *out = x16 + m * K;
#pragma unroll
    for (int j = 0; j < R; ++j) {
      const int k = (j * 256 + tid) * 8;
      if (k >= K) break;
      const uint32_t w[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
      uint32_t o[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 f = unpack2<DT>(w[i]);
        o[i] = pack2<WQ_F16>(scale_pow2(f.x, -e), scale_pow2(f.y, -e));
      }
      *reinterpret_cast<uint4 *>(out + k) = make_uint4(o[0], o[1], o[2], o[3]);
    }
    if (dext) {
      // per-group sums of the fp16 row just written, a thread per group, in
      // ascending k (the block's own stores: __syncthreads orders them first)
      __syncthreads();
      __nv_bfloat16 *drow = dext + m * ldx;
      for (int gi = tid; gi < G; gi += 256) {
        const int k0 = gi * group, k1 = k0 + group < K ? k0 + group : K;
        float d = 0.f;
        for (int k = k0; k < k1; k += 8) {  // group % 32 == 0 and K % 8 == 0
          const uint4 u = *reinterpret_cast<const uint4 *>(out + k);
          const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float2 f = unpack2<WQ_F16>(w[i]);
            d += f.x;
            d += f.y;
          }
        }
        // d = hi + lo to 2^-18, each bf16 (the difference d - hi is exact in fp32)
        const __nv_bfloat16 hi = __float2bfloat16_rn(d);
        const __nv_bfloat16 lo = __float2bfloat16_rn(d - __bfloat162float(hi));
        drow[gi] = hi;
        drow[G + gi] = lo;
      }
      for (int j = 2 * G + tid; j < ldx; j += 256) drow[j] = __float2bfloat16_rn(0.f);
    }
  }
}

template <int DT>
cudaError_t launch_row_prep_reg(const Problem &p, int16_t *e_row, __half *x16,
                                __nv_bfloat16 *dext, int ldx, cudaStream_t s) {
  using T = typename Elem<DT>::T;
  const T *x1 = static_cast<const T *>(p.x1);
  int64_t blocks = p.M < 1 ? 1 : p.M;
  const int64_t cap = (int64_t)device_info().sms * 8;
  if (blocks > cap) blocks = cap;
  const int K = (int)p.K, group = (int)p.group, G = (int)p.G;
  if (p.K <= 2048)
    row_prep_reg_kernel<DT, 1><<<(unsigned)blocks, 256, 0, s>>>(x1, p.M, K, e_row, x16, dext,
                                                                group, G, ldx);
  else if (p.K <= 4096)
    row_prep_reg_kernel<DT, 2><<<(unsigned)blocks, 256, 0, s>>>(x1, p.M, K, e_row, x16, dext,
                                                                group, G, ldx);
  else
    row_prep_reg_kernel<DT, 4><<<(unsigned)blocks, 256, 0, s>>>(x1, p.M, K, e_row, x16, dext,
                                                                group, G, ldx);
  return cudaGetLastError();
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
                   int G, int N, int ld, float qmax, int int4, int16_t *__restrict__ e_col,
                   uint32_t *__restrict__ S16, __nv_bfloat16 *__restrict__ Oext, int ldx) {
  using E = Elem<DT>;
  __shared__ float s_max[8][32];
  __shared__ int s_exp[32];
  const int cx = threadIdx.x & 31, gy = threadIdx.x >> 5;
  const int n = blockIdx.x * 32 + cx;
  float mx = 0.f;
  if (n < N) {
#pragma unroll 4
    for (int g = gy; g < G; g += 8) {
      mx = fmaxf(mx, qmax * fabsf(E::to_f(S[(int64_t)g * N + n])));
    }
  }
  s_max[gy][cx] = mx;
  __syncthreads();
  if (gy == 0) {
    float m = s_max[0][cx];
#pragma unroll
    for (int i = 1; i < 8; ++i) m = fmaxf(m, s_max[i][cx]);
    // m * 2^-e in [2^12, 2^13); 0 for an all-zero or non-finite column
    const int e = (m > 0.f && m <= FLT_MAX) ? ilog2f(m) - 12 : 0;
    if (n < N) e_col[n] = (int16_t)e;
    s_exp[cx] = e;
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
  if (int4 == 2) {
    // transposed INT4 weights: one word per (group, column), S16 in bits 15:0
    // for the even k of a byte and S16 / 16 in bits 31:16 for the odd k
    // (whose nibble is used in place at bits 7:4), plain column order
    if (n < N) {
      const int e = s_exp[cx];
#pragma unroll 4
      for (int g = gy; g < G; g += 8) {
        const float v = E::to_f(S[(int64_t)g * N + n]);
        const uint32_t lo = (uint32_t)__half_as_ushort(__float2half_rn(scale_pow2(v, -e)));
        const uint32_t hi = (uint32_t)__half_as_ushort(__float2half_rn(scale_pow2(v, -e - 4)));
        S16[(int64_t)g * N + n] = lo | (hi << 16);
      }
    }
    return;
  }
  if (n < ld) {
    const int e = s_exp[cx];
    const int es = (int4 && (n & 1)) ? -e - 4 : -e;  // odd INT4 columns: scale / 16 (exact)
#pragma unroll 4
    for (int g = gy; g < G; g += 8) {
      const bool live = n < N;
      S16[(int64_t)g * ld + dst] =
          live ? half_pair(scale_pow2(E::to_f(S[(int64_t)g * N + n]), es)) : 0u;
    }
  }
  if (O && n < N) {
    __nv_bfloat16 *orow = Oext + (int64_t)n * ldx;
    for (int g = gy; g < G; g += 8) {
      const __nv_bfloat16 o = __float2bfloat16_rn(scale_pow2(E::to_f(O[(int64_t)g * N + n]), -s_exp[cx]));
      orow[g] = o;
      orow[G + g] = o;
    }
    for (int j = 2 * G + gy; j < ldx; j += 8) orow[j] = __float2bfloat16_rn(0.f);
  }
}

}  // namespace

cudaError_t launch_row_prep(const Problem &p, float *rowsum, int16_t *e_row, __half *x16,
                            __nv_bfloat16 *dext, int ldx, cudaStream_t s) {
  if (x16 && !rowsum && p.K <= 8192)
    return p.dtype == WQ_BF16 ? launch_row_prep_reg<WQ_BF16>(p, e_row, x16, dext, ldx, s)
                              : launch_row_prep_reg<WQ_F16>(p, e_row, x16, dext, ldx, s);
  const int64_t warps_needed = p.M;
  int64_t blocks = (warps_needed * 32 + 255) / 256;
  const int64_t cap = (int64_t)device_info().sms * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  const int group = (int)p.group, G = (int)p.G;
  if (p.dtype == WQ_BF16)
    row_prep_kernel<WQ_BF16><<<(unsigned)blocks, 256, 0, s>>>(
        static_cast<const __nv_bfloat16 *>(p.x1), p.M, (int)p.K, rowsum, e_row, x16, dext, group,
        G, ldx);
  else
    row_prep_kernel<WQ_F16><<<(unsigned)blocks, 256, 0, s>>>(static_cast<const __half *>(p.x1), p.M,
                                                             (int)p.K, rowsum, e_row, x16, dext,
                                                             group, G, ldx);
  return cudaGetLastError();
}

cudaError_t launch_so_prep_t(const Problem &p, int16_t *e_col, uint32_t *S16T, cudaStream_t s) {
  const int N = (int)p.N;
  const int blocks = (N + 31) / 32;
  if (p.dtype == WQ_BF16)
    so_prep_kernel<WQ_BF16><<<blocks, 256, 0, s>>>(static_cast<const __nv_bfloat16 *>(p.scale), nullptr,
                                                   (int)p.G, N, N, 8.f, 2, e_col, S16T, nullptr, 0);
  else
    so_prep_kernel<WQ_F16><<<blocks, 256, 0, s>>>(static_cast<const __half *>(p.scale), nullptr,
                                                  (int)p.G, N, N, 8.f, 2, e_col, S16T, nullptr, 0);
  return cudaGetLastError();
}

cudaError_t launch_so_prep(const Problem &p, int64_t ld, int16_t *e_col, uint32_t *S16,
                           __nv_bfloat16 *Oext, int ldx, cudaStream_t s) {
  const int N = (int)p.N;
  const int blocks = (int)((ld + 31) / 32);
  const float qmax = p.wbits == 4 ? 8.f : 128.f;
  const int int4 = p.wbits == 4 ? 1 : 0;
  if (p.dtype == WQ_BF16)
    so_prep_kernel<WQ_BF16><<<blocks, 256, 0, s>>>(static_cast<const __nv_bfloat16 *>(p.scale),
                                                   static_cast<const __nv_bfloat16 *>(p.offset),
                                                   (int)p.G, N, (int)ld, qmax, int4, e_col, S16,
                                                   Oext, ldx);
  else
    so_prep_kernel<WQ_F16><<<blocks, 256, 0, s>>>(static_cast<const __half *>(p.scale),
                                                  static_cast<const __half *>(p.offset), (int)p.G,
                                                  N, (int)ld, qmax, int4, e_col, S16, Oext, ldx);
  return cudaGetLastError();
}

}  // namespace wq
