// Small device helpers shared by the kernels of libwq.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "../../include/wq.h"

namespace wq {

// Element type of the floating tensors, selected by the wq_dtype value.
template <int DT> struct Elem;
template <> struct Elem<WQ_F16> {
  using T = __half;
  __device__ static __forceinline__ float to_f(T v) { return __half2float(v); }
  __device__ static __forceinline__ T from_f(float v) { return __float2half_rn(v); }
};
template <> struct Elem<WQ_BF16> {
  using T = __nv_bfloat16;
  __device__ static __forceinline__ float to_f(T v) { return __bfloat162float(v); }
  __device__ static __forceinline__ T from_f(float v) { return __float2bfloat16_rn(v); }
};

// Two 16-bit floats of a 32-bit word -> two fp32 values (low half first).
template <int DT> __device__ __forceinline__ float2 unpack2(uint32_t w);
template <> __device__ __forceinline__ float2 unpack2<WQ_BF16>(uint32_t w) {
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}
template <> __device__ __forceinline__ float2 unpack2<WQ_F16>(uint32_t w) {
  __half2 h = *reinterpret_cast<__half2 *>(&w);
  return __half22float2(h);
}

// Two fp32 values -> one word of two 16-bit floats, each rounded to nearest even.
template <int DT> __device__ __forceinline__ uint32_t pack2(float lo, float hi);
template <> __device__ __forceinline__ uint32_t pack2<WQ_BF16>(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&v);
}
template <> __device__ __forceinline__ uint32_t pack2<WQ_F16>(float lo, float hi) {
  __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&v);
}

// Read-only streaming 128-bit load (not kept in L1).
__device__ __forceinline__ uint4 ld_stream_u4(const void *p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ void st_stream_u4(void *p, uint4 v) {
  asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}

// Packed pair subtraction in the operand dtype (exact here: small integers).
template <int DT>
__device__ __forceinline__ uint32_t sub2(uint32_t v, uint32_t c) {
  uint32_t r;
  if (DT == WQ_BF16)
    asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(v), "r"(c));
  else
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(v), "r"(c));
  return r;
}

// 4-bit value (0..15, two's complement nibble) of element (k, n) of a weight in
// the kernel-native tiled INT4 layout (64 k x 16 column tiles, 512 bytes each,
// tiles of a 64-row slab in column order; see wq_tiled.cu for the map).
__device__ __forceinline__ uint32_t tiled_nibble(const uint8_t *w, int64_t k, int64_t n, int64_t N) {
  const int64_t s = k >> 6, c = n >> 4;
  const int kk = (int)(k & 63), cc = (int)(n & 15);
  const int t = (kk >> 3) & 3, j = 2 * (kk >> 5) + ((kk >> 2) & 1), e = kk & 3;
  const int lane = 4 * (cc & 7) + t;
  const int p = (e < 2 ? 0 : 2) + (cc >> 3) + 4 * (e & 1);
  const uint32_t b = w[(s * (N >> 4) + c) * 512 + lane * 16 + j * 4 + (p >> 1)];
  return (b >> (4 * (p & 1))) & 0xFu;
}

// 2^e as an fp32 for e in [-126, 127].
__device__ __forceinline__ float exp2i(int e) { return __int_as_float((e + 127) << 23); }

// v * 2^e for e in [-252, 254], in two exact power-of-two steps (the result
// rounds only where it leaves the fp32 normal range).
__device__ __forceinline__ float scale_pow2(float v, int e) {
  const int a = e < -126 ? -126 : (e > 127 ? 127 : e);
  int b = e - a;
  b = b < -126 ? -126 : (b > 127 ? 127 : b);
  return v * exp2i(a) * exp2i(b);
}

}  // namespace wq
