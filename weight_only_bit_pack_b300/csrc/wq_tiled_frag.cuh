// Register-level helpers shared by the kernels that read the kernel-native
// tiled INT4 layout with mma.sync (wq_decode_tiled.cu, wq_decode_km.cu): the
// lane's 16 bytes of a 512-byte tile are its A fragments for four m16n8k16
// MMAs (A = W^T, 16 columns x 16 k-rows each), and the activations enter as the
// B operand.
#pragma once

#include <cstdint>

#include "../../include/wq.h"

namespace wq {
namespace tfrag {

// one cp.async of 16 bytes (global -> shared)
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Four A registers of one MMA from weight word w: register i holds nibbles i
// and i + 4 as the 16-bit floats 136 + q (bf16) or 1032 + q (fp16), exactly:
// (nibble ^ 8) = q + 8 lands in the low mantissa bits of 128.0 (1024.0).
template <int DT>
__device__ __forceinline__ void word_to_a(uint32_t w, uint32_t (&a)[4]) {
  constexpr uint32_t MAGIC = DT == WQ_BF16 ? 0x43084308u : 0x64086408u;
#pragma unroll
  for (int i = 0; i < 4; ++i) a[i] = ((i ? w >> (4 * i) : w) & 0x000F000Fu) ^ MAGIC;
}

// The same MMA without `volatile`, so the compiler may interleave it with the
// conversions around it.
template <bool BF>
__device__ __forceinline__ void mma_16816_f(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                            uint32_t b1) {
  if constexpr (BF)
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  else
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// mma_16816_f with a zero accumulator input.
template <bool BF>
__device__ __forceinline__ void mma_16816_z(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                            uint32_t b1) {
  const float z = 0.f;
  if constexpr (BF)
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%10,%10,%10,%10};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(z));
  else
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%10,%10,%10,%10};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(z));
}

}  // namespace tfrag
}  // namespace wq
