// INT32 -> dense INT4 weight pack (aclnnConvertWeightToINT4Pack, "Function
// description": re-lay 4-bit values held one per INT32 into two per byte).
//
// Layout: the input is (K, N) int32 row-major, the output (K, N/2) bytes; the
// element of even column 2j goes to bits 3:0 of byte j, column 2j+1 to bits
// 7:4, and a value keeps its low four bits. N is even, so a byte never spans
// two rows and the whole pack is a flat map from 2*i, 2*i+1 to byte i.
//
// The kernel is bound by HBM: 8 bytes read and 1 written per output byte. Each
// thread turns 8 int32 (two neighbouring 16-byte streaming loads, so a warp
// reads 1 KB contiguously) into one 4-byte store; a grid-stride loop over 4-byte
// units keeps every SM busy, and a scalar tail covers a byte count that is not
// a multiple of 4 or unaligned pointers.
#include "wq_internal.h"
#include "wq_common.cuh"

namespace wq {
namespace {

__device__ __forceinline__ uint32_t nib8(uint4 a, uint4 b) {
  // eight int32 (a = elements 0..3, b = 4..7) -> eight nibbles, element t at bits 4t+3:4t
  uint32_t w = (a.x & 0xFu) | ((a.y & 0xFu) << 4) | ((a.z & 0xFu) << 8) | ((a.w & 0xFu) << 12);
  w |= ((b.x & 0xFu) << 16) | ((b.y & 0xFu) << 20) | ((b.z & 0xFu) << 24) | ((b.w & 0xFu) << 28);
  return w;
}

__global__ void __launch_bounds__(256) pack_int4_kernel(const int32_t *__restrict__ in,
                                                       uint8_t *__restrict__ out, int64_t nvec,
                                                       int64_t tail_begin, int64_t nbytes) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  for (int64_t i = tid; i < nvec; i += stride) {
    const int32_t *src = in + i * 8;
    const uint4 a = ld_stream_u4(src), b = ld_stream_u4(src + 4);
    __stcs(reinterpret_cast<unsigned int *>(out) + i, nib8(a, b));
  }
  for (int64_t b = tail_begin + tid; b < nbytes; b += stride) {
    const uint32_t lo = (uint32_t)in[2 * b] & 0xFu;
    const uint32_t hi = (uint32_t)in[2 * b + 1] & 0xFu;
    out[b] = (uint8_t)(lo | (hi << 4));
  }
}

}  // namespace

cudaError_t launch_pack_int4(const int32_t *in, uint8_t *out, int64_t K, int64_t N, cudaStream_t s) {
  const int64_t nbytes = K * (N / 2);
  const bool aligned = ((uintptr_t)in % 16 == 0) && ((uintptr_t)out % 4 == 0);
  const int64_t nvec = aligned ? nbytes / 4 : 0;
  const int64_t tail = nvec * 4;
  const int64_t work = nvec > 0 ? nvec : (nbytes - tail);
  const int threads = 256;
  int64_t blocks = (work + threads - 1) / threads;
  const int64_t cap = (int64_t)device_info().sms * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  pack_int4_kernel<<<(unsigned)blocks, threads, 0, s>>>(in, out, nvec, tail, nbytes);
  return cudaGetLastError();
}

}  // namespace wq
