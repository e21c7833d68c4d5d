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
#include "wq_sm100.cuh"

namespace wq {
namespace {

using sm100::ldmatrix_x4;
using sm100::ldmatrix_x4_trans;
using sm100::mma_16816;
using sm100::smem_u32;

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

// ---------------------------------------------------------------- tensor-core form
//
// The same product with the slice sums on the tensor cores: E2M1 codes become
// fp16 exactly (cvt.rn.f16x2.e2m1x2), each 32-deep slice is two m16n8k16 MMAs
// with fp32 accumulation -- exact, as the slice sum of E2M1 products is a
// multiple of 1/4 below 2^11 -- and the slice is then scaled and added to the
// running fp32 sum: tot = fma(acc * 2^(e1 - 127), 2^(e2 - 127), tot). The
// first product is exact (acc has <= 13 significant bits above 2^-2, and
// 2^-127 is an fp32 subnormal, so acc * 2^-127 is a multiple of 2^-129); a row
// exponent above 117 could overflow it, so a slice whose scales reach 245
// takes a two-step path on the combined exponent instead. One rounding per
// slice (the add), against the exact kernel's fp64 sum.
//
// CTA tile 128 x 128 outputs, 8 warps as 2 (M) x 4 (N), warp tile 64 x 32
// (4 x 4 MMA tiles); a slice's codes are fetched into registers one slice
// ahead, decoded and stored into the other of two shared buffers: x2 and a
// transposed x1 as [k][128 + 8 pad] fp16 rows (ldmatrix.trans gives the
// fragments), an x1 given as (M, K) as [m][32 + 8 pad] rows (plain ldmatrix).

constexpr int kTcThreads = 256, kTcT = 128;
constexpr int kRowH = kTcT + 8;   // halves per [k][*] row (272 bytes: conflict-free ldmatrix)
constexpr int kRowA = kGs + 8;    // halves per [m][k] row (80 bytes)

// two fp16 values of the E2M1 codes in bits 3:0 (low half) and 7:4 (high half)
__device__ __forceinline__ uint32_t e2m1x2_to_f16x2(uint32_t byte) {
  uint32_t r;
  asm("{\n\t.reg .b8 t;\n\tcvt.u8.u32 t, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, t;\n\t}" : "=r"(r) : "r"(byte));
  return r;
}

// 2^(e - 127) for an E8M0 byte as an fp32 factor (e = 0 gives the subnormal
// 2^-127, e = 255 NaN)
__device__ __forceinline__ float e8m0_factor(uint32_t e) {
  return e == 255u ? __int_as_float(0x7fc00000) : (e ? __int_as_float((int)(e << 23)) : __int_as_float(0x00400000));
}

// acc * 2^e for e in [-254, 254] in two exact power-of-two steps
__device__ __forceinline__ float scale_two_step(float acc, int e) {
  const int a = e < -126 ? -126 : (e > 127 ? 127 : e);
  int b = e - a;
  b = b < -126 ? -126 : (b > 127 ? 127 : b);
  return acc * __int_as_float((a + 127) << 23) * __int_as_float((b + 127) << 23);
}

// One slice of a warp's (16 MTW) x 32 tile: two m16n8k16 MMAs deep from the
// fp16 tiles at a_base / b_base, then scaled by the slice's E8M0 bytes (e1s per
// tile row, e2s per tile column) and added to tot.
template <bool X1T, int MTW = 4>
__device__ __forceinline__ void mx_slice(uint32_t a_base, uint32_t b_base, const uint8_t *e1s,
                                         const uint8_t *e2s, bool huge, float (&tot)[MTW][4][4],
                                         int lane, int wm, int wn) {
  const int g = lane >> 2, t = lane & 3;
  constexpr int WR = 16 * MTW;  // the warp's rows
  float acc[MTW][4][4];
#pragma unroll
  for (int a = 0; a < MTW; ++a)
#pragma unroll
    for (int b = 0; b < 4; ++b)
#pragma unroll
      for (int c = 0; c < 4; ++c) acc[a][b][c] = 0.f;
#pragma unroll
  for (int kk = 0; kk < 2; ++kk) {
    uint32_t af[MTW][4], bf[4][2];
    const int sub = lane >> 3, r8 = lane & 7;
#pragma unroll
    for (int mt = 0; mt < MTW; ++mt) {
      const int mb = wm * WR + mt * 16;
      if constexpr (X1T) {
        const int k = kk * 16 + r8 + 8 * (sub >> 1), m = mb + 8 * (sub & 1);
        ldmatrix_x4_trans(a_base + (uint32_t)(k * kRowH + m) * 2u, af[mt][0], af[mt][1],
                          af[mt][2], af[mt][3]);
      } else {
        const int m = mb + r8 + 8 * (sub & 1), k = kk * 16 + 8 * (sub >> 1);
        ldmatrix_x4(a_base + (uint32_t)(m * kRowA + k) * 2u, af[mt][0], af[mt][1], af[mt][2],
                    af[mt][3]);
      }
    }
#pragma unroll
    for (int np = 0; np < 2; ++np) {
      const int k = kk * 16 + r8 + 8 * (sub & 1), n = wn * 32 + np * 16 + 8 * (sub >> 1);
      ldmatrix_x4_trans(b_base + (uint32_t)(k * kRowH + n) * 2u, bf[2 * np][0], bf[2 * np][1],
                        bf[2 * np + 1][0], bf[2 * np + 1][1]);
    }
#pragma unroll
    for (int mt = 0; mt < MTW; ++mt)
#pragma unroll
      for (int nt = 0; nt < 4; ++nt)
        mma_16816<false>(acc[mt][nt], af[mt][0], af[mt][1], af[mt][2], af[mt][3], bf[nt][0], bf[nt][1]);
  }
  // scale the slice and add it: element c of tile (mt, nt) is row g + 8 (c >> 1),
  // column 2t + (c & 1)
  if (!huge) {
    float hc[4][2];
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
      const int cb = wn * 32 + nt * 8 + 2 * t;
      hc[nt][0] = e8m0_factor(e2s[cb]);
      hc[nt][1] = e8m0_factor(e2s[cb + 1]);
    }
#pragma unroll
    for (int mt = 0; mt < MTW; ++mt) {
      const float f0 = e8m0_factor(e1s[wm * WR + mt * 16 + g]);
      const float f1 = e8m0_factor(e1s[wm * WR + mt * 16 + g + 8]);
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
        const float h0 = hc[nt][0], h1 = hc[nt][1];
        tot[mt][nt][0] = fmaf(acc[mt][nt][0] * f0, h0, tot[mt][nt][0]);
        tot[mt][nt][1] = fmaf(acc[mt][nt][1] * f0, h1, tot[mt][nt][1]);
        tot[mt][nt][2] = fmaf(acc[mt][nt][2] * f1, h0, tot[mt][nt][2]);
        tot[mt][nt][3] = fmaf(acc[mt][nt][3] * f1, h1, tot[mt][nt][3]);
      }
    }
  } else {
#pragma unroll
    for (int mt = 0; mt < MTW; ++mt)
#pragma unroll
      for (int nt = 0; nt < 4; ++nt)
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const uint32_t e1 = e1s[wm * WR + mt * 16 + g + 8 * (c >> 1)];
          const uint32_t e2 = e2s[wn * 32 + nt * 8 + 2 * t + (c & 1)];
          const float v = (e1 == 255u || e2 == 255u)
                              ? __int_as_float(0x7fc00000)
                              : scale_two_step(acc[mt][nt][c], (int)e1 + (int)e2 - 254);
          tot[mt][nt][c] += v;
        }
  }
}

template <bool X1T>
__global__ void __launch_bounds__(kTcThreads, 1)
    mx_mma_kernel(const uint8_t *__restrict__ x1, const uint8_t *__restrict__ s1,
                  const uint8_t *__restrict__ x2, const uint8_t *__restrict__ s2,
                  float *__restrict__ y, int64_t M, int64_t K, int64_t N) {
  constexpr int A_HALVES = X1T ? kGs * kRowH : kTcT * kRowA;
  __shared__ __align__(16) __half as[2][A_HALVES];
  __shared__ __align__(16) __half bs[2][kGs * kRowH];
  __shared__ uint8_t es1[2][kTcT], es2[2][kTcT];
  __shared__ int huge[2];  // a scale of this slice is 245..254

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int wm = warp & 1, wn = warp >> 1;
  const int g = lane >> 2, t = lane & 3;
  const int64_t m0 = (int64_t)blockIdx.y * kTcT, n0 = (int64_t)blockIdx.x * kTcT;
  const int64_t J = (K + kGs - 1) / kGs;

  // ---- one slice's global codes and scales in registers (8 + 8 bytes a thread)
  uint32_t ra[8], rb[8], rs = 0;
  auto fetch = [&](int64_t j) {
    const int64_t k0 = j * kGs;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int q = i * kTcThreads + tid;
      if constexpr (X1T) {  // (K, M/2): 32 k-rows x 64 bytes
        const int64_t k = k0 + q / 64, b = m0 / 2 + q % 64;
        ra[i] = (k < K && b < M / 2) ? x1[k * (M / 2) + b] : 0u;
      } else {              // (M, K/2): 128 rows x 16 bytes
        const int64_t m = m0 + q / 16, b = k0 / 2 + q % 16;
        ra[i] = (m < M && b < K / 2) ? x1[m * (K / 2) + b] : 0u;
      }
      const int64_t k = k0 + q / 64, b = n0 / 2 + q % 64;
      rb[i] = (k < K && b < N / 2) ? x2[k * (N / 2) + b] : 0u;
    }
    rs = 127u;
    if (tid < kTcT) {
      const int64_t m = m0 + tid;
      if (m < M) rs = X1T ? s1[j * M + m] : s1[m * J + j];
    } else {
      const int64_t n = n0 + tid - kTcT;
      if (n < N) rs = s2[j * N + n];
    }
  };
  auto store = [&](int buf) {
    uint32_t *aw = reinterpret_cast<uint32_t *>(as[buf]);
    uint32_t *bw = reinterpret_cast<uint32_t *>(bs[buf]);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int q = i * kTcThreads + tid;
      if constexpr (X1T) aw[((q / 64) * kRowH) / 2 + q % 64] = e2m1x2_to_f16x2(ra[i]);
      else aw[((q / 16) * kRowA) / 2 + q % 16] = e2m1x2_to_f16x2(ra[i]);
      bw[((q / 64) * kRowH) / 2 + q % 64] = e2m1x2_to_f16x2(rb[i]);
    }
    if (tid < kTcT) es1[buf][tid] = (uint8_t)rs;
    else es2[buf][tid - kTcT] = (uint8_t)rs;
    if (rs >= 245u && rs != 255u) huge[buf] = 1;
  };

  float tot[4][4][4];
#pragma unroll
  for (int a = 0; a < 4; ++a)
#pragma unroll
    for (int b = 0; b < 4; ++b)
#pragma unroll
      for (int c = 0; c < 4; ++c) tot[a][b][c] = 0.f;

  if (tid == 0) huge[0] = huge[1] = 0;
  __syncthreads();
  fetch(0);
  store(0);
  __syncthreads();
  for (int64_t j = 0; j < J; ++j) {
    const int buf = (int)(j & 1);
    const uint32_t a_base = smem_u32(as[0]) + (uint32_t)buf * (uint32_t)sizeof(as[0]);
    const uint32_t b_base = smem_u32(bs[0]) + (uint32_t)buf * (uint32_t)sizeof(bs[0]);
    if (j + 1 < J) fetch(j + 1);  // in flight during this slice's MMAs
    mx_slice<X1T>(a_base, b_base, es1[buf], es2[buf], huge[buf] != 0, tot, lane, wm, wn);
    if (j + 1 < J) {
      if (tid == 0) huge[buf ^ 1] = 0;  // the other buffer was last read a slice ago
      __syncthreads();                  // (and its flag with it)
      store(buf ^ 1);
    }
    __syncthreads();
  }
  // y += tot
#pragma unroll
  for (int mt = 0; mt < 4; ++mt)
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int64_t m = m0 + wm * 64 + mt * 16 + g + 8 * (c >> 1);
        const int64_t n = n0 + wn * 32 + nt * 8 + 2 * t + (c & 1);
        if (m < M && n < N) y[m * N + n] += tot[mt][nt][c];
      }
}

// The transposed-x1 form (the page's supported one) with x1, x2 and the scales
// copied a raw slice at a time by cp.async into a ring of kRing stages, three
// slices ahead of their use, then decoded into the fp16 tiles: the copies no
// longer wait on a single slice of compute. Needs M and N multiples of 32 and
// 16-byte aligned operands (16-byte copies that never straddle the edge).
constexpr int kRing = 4;
constexpr uint32_t kRawA = kGs * 64, kRawB = kGs * 64, kRawS = 2 * kTcT;
constexpr uint32_t kRawStage = kRawA + kRawB + kRawS;
constexpr uint32_t kF16Tile = kGs * kRowH * 2;
constexpr uint32_t kRingSmem = kRing * kRawStage + 4 * kF16Tile;
// 16 warps of 32 x 32 (the same 128 x 128 CTA tile): half the accumulator
// registers of a 64 x 32 warp, so twice the warps are resident
constexpr int kRingThreads = 512;

__device__ __forceinline__ void cp_async16_zfill(uint32_t dst, const void *src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
               "r"(valid ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit_group() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait_group() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__global__ void __launch_bounds__(kRingThreads, 1)
    mx_mma_ring_kernel(const uint8_t *__restrict__ x1, const uint8_t *__restrict__ s1,
                       const uint8_t *__restrict__ x2, const uint8_t *__restrict__ s2,
                       float *__restrict__ y, int64_t M, int64_t K, int64_t N) {
  extern __shared__ __align__(16) uint8_t mx_smem[];
  __shared__ int huge[2];
  const uint32_t raw = smem_u32(mx_smem);
  const uint32_t fa = raw + kRing * kRawStage;  // two A tiles, then two B tiles
  const uint32_t fb = fa + 2 * kF16Tile;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int wm = warp & 3, wn = warp >> 2;
  const int64_t m0 = (int64_t)blockIdx.y * kTcT, n0 = (int64_t)blockIdx.x * kTcT;
  const int64_t J = (K + kGs - 1) / kGs;

  // stage st of the ring: 32 rows x 64 bytes of x1 (threads 0..127) and of x2
  // (threads 128..255), 16 bytes a thread, and the slice's 128 + 128 scale bytes
  // (threads 0..15); copies past K, M or N read nothing and fill zeros. Every
  // thread commits one group per stage.
  auto issue = [&](int64_t st) {
    if (st < J && tid < 256) {
      const uint32_t slot = raw + (uint32_t)(st % kRing) * kRawStage;
      const int64_t k0 = st * kGs;
      const int row = (tid & 127) >> 2, c = tid & 3;
      const bool kin = k0 + row < K;
      if (tid < 128) {
        const bool ok = kin && m0 / 2 + 16 * c < M / 2;
        cp_async16_zfill(slot + (uint32_t)(row * 64 + 16 * c),
                         ok ? x1 + (k0 + row) * (M / 2) + m0 / 2 + 16 * c : x1, ok);
      } else {
        const bool ok = kin && n0 / 2 + 16 * c < N / 2;
        cp_async16_zfill(slot + kRawA + (uint32_t)(row * 64 + 16 * c),
                         ok ? x2 + (k0 + row) * (N / 2) + n0 / 2 + 16 * c : x2, ok);
      }
      if (tid < 8) {
        const bool ok = m0 + 16 * tid < M;
        cp_async16_zfill(slot + kRawA + kRawB + 16u * tid, ok ? s1 + st * M + m0 + 16 * tid : s1, ok);
      } else if (tid < 16) {
        const int q = tid - 8;
        const bool ok = n0 + 16 * q < N;
        cp_async16_zfill(slot + kRawA + kRawB + kTcT + 16u * q, ok ? s2 + st * N + n0 + 16 * q : s2, ok);
      }
    }
    cp_async_commit_group();  // one group per stage on every thread, empty or not
  };
  // raw stage st -> fp16 tiles b: 8 bytes of codes a thread, threads 0..255
  // for x1 and 256..511 for x2
  auto decode = [&](int64_t st, int b) {
    const uint32_t slot = raw + (uint32_t)(st % kRing) * kRawStage;
    const int row = (tid & 255) >> 3, off = (tid & 7) * 8;
    {
      const int op = tid >> 8;
      uint32_t lo, hi;
      asm volatile("ld.shared.v2.b32 {%0,%1}, [%2];"
                   : "=r"(lo), "=r"(hi)
                   : "r"(slot + (op ? kRawA : 0u) + (uint32_t)(row * 64 + off)));
      uint32_t w[8];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        w[i] = e2m1x2_to_f16x2((lo >> (8 * i)) & 0xFFu);
        w[4 + i] = e2m1x2_to_f16x2((hi >> (8 * i)) & 0xFFu);
      }
      const uint32_t dst = (op ? fb : fa) + (uint32_t)b * kF16Tile + (uint32_t)(row * kRowH * 2 + off * 4);
      asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(dst), "r"(w[0]), "r"(w[1]), "r"(w[2]),
                   "r"(w[3])
                   : "memory");
      asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(dst + 16), "r"(w[4]), "r"(w[5]),
                   "r"(w[6]), "r"(w[7])
                   : "memory");
    }
    if (tid < 256) {
      const uint32_t e = mx_smem[(st % kRing) * kRawStage + kRawA + kRawB + tid];
      if (e >= 245u && e != 255u) huge[b] = 1;
    }
  };

  float tot[2][4][4];
#pragma unroll
  for (int a = 0; a < 2; ++a)
#pragma unroll
    for (int b = 0; b < 4; ++b)
#pragma unroll
      for (int c = 0; c < 4; ++c) tot[a][b][c] = 0.f;

  if (tid == 0) huge[0] = huge[1] = 0;
#pragma unroll
  for (int st = 0; st < kRing - 1; ++st) issue(st);
  cp_async_wait_group<kRing - 2>();
  __syncthreads();
  decode(0, 0);
  __syncthreads();
  for (int64_t j = 0; j < J; ++j) {
    const int buf = (int)(j & 1);
    issue(j + kRing - 1);
    const uint8_t *es = mx_smem + (j % kRing) * kRawStage + kRawA + kRawB;
    mx_slice<true, 2>(fa + (uint32_t)buf * kF16Tile, fb + (uint32_t)buf * kF16Tile, es, es + kTcT,
                      huge[buf] != 0, tot, lane, wm, wn);
    if (j + 1 < J) {
      cp_async_wait_group<kRing - 2>();  // stage j + 1 has landed (this thread's copies)
      if (tid == 0) huge[buf ^ 1] = 0;   // last read a slice ago
      __syncthreads();                   // ... and everyone's, and tiles buf ^ 1 are free
      decode(j + 1, buf ^ 1);
    }
    __syncthreads();
  }
  cp_async_wait_group<0>();  // no copy in flight at exit (only empty groups remain)
#pragma unroll
  for (int mt = 0; mt < 2; ++mt)
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int64_t m = m0 + wm * 32 + mt * 16 + (lane >> 2) + 8 * (c >> 1);
        const int64_t n = n0 + wn * 32 + nt * 8 + 2 * (lane & 3) + (c & 1);
        if (m < M && n < N) y[m * N + n] += tot[mt][nt][c];
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

cudaError_t launch_mx_matmul_add_tc(const uint8_t *x1, const uint8_t *s1, bool x1t,
                                    const uint8_t *x2, const uint8_t *s2, float *y, int64_t M,
                                    int64_t K, int64_t N, cudaStream_t s) {
  const dim3 grid((unsigned)((N + kTcT - 1) / kTcT), (unsigned)((M + kTcT - 1) / kTcT), 1);
  auto a16 = [](const void *p) { return reinterpret_cast<uintptr_t>(p) % 16 == 0; };
  if (x1t && M % 32 == 0 && N % 32 == 0 && a16(x1) && a16(x2) && a16(s1) && a16(s2)) {
    static cudaError_t attr = cudaFuncSetAttribute(
        mx_mma_ring_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kRingSmem);
    if (attr != cudaSuccess) return attr;
    mx_mma_ring_kernel<<<grid, kRingThreads, kRingSmem, s>>>(x1, s1, x2, s2, y, M, K, N);
  } else if (x1t)
    mx_mma_kernel<true><<<grid, kTcThreads, 0, s>>>(x1, s1, x2, s2, y, M, K, N);
  else
    mx_mma_kernel<false><<<grid, kTcThreads, 0, s>>>(x1, s1, x2, s2, y, M, K, N);
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
