// Kernel-native tiled INT4 layout: the pack into it and the conversions between
// the INT4 layouts of a weight (dense, transposed, tiled).
//
// aclnnConvertWeightToINT4Pack, "Function description": besides the dense ND
// output, the pack can emit the same 4-bit values in a layout tiled for the
// matrix unit. The pages do not fix such a layout for this GPU; the library's
// is built around the m16n8k16 MMA fragments of the small-M decode kernel:
//
//   A (K, N) weight (N % 16 == 0) is cut into tiles of 64 k-rows x 16 columns.
//   Tile (s, c) -- k-rows 64s.., columns 16c.. -- takes the 512 bytes at
//   (s * N/16 + c) * 512: the tiles of one 64-row slab follow each other in
//   column order, slab after slab. K is padded with zero nibbles to a multiple
//   of 64. Inside a tile, element (kk, cc) = (k - 64s, n - 16c) sits in
//     lane = 4 g + t, word j = 2 h + jl, nibble p = (e < 2 ? 0 : 2) + u + 4 (e % 2)
//   with h = kk/32, t = (kk%32)/8, jl = (kk%8)/4, e = kk%4, g = cc%8, u = cc/8:
//   byte lane*16 + j*4 + p/2, bits 4(p%2)+3 : 4(p%2).
//
// So lane l's 16 bytes are its A fragments (A = W^T) of the tile's four MMAs:
// word j is MMA j, and its register i = (word >> 4i) & 0x000F000F holds
// nibbles i and i+4, i.e. a0 = columns g (rows 2t, 2t+1 of A), a1 = column
// g+8, a2 / a3 the same columns two k-rows on. MMA j covers the k-rows
// 32(j/2) + 4(j%2) + 8t + {0..3}: all inside one aligned 32-row block, so no
// MMA straddles a quantization group (group sizes are multiples of 32), and a
// lane's activations for the whole tile are the 16-byte runs at 8t and 32 + 8t.
//
// The pack reads a 64 x 128 block of int32 through shared memory (coalesced
// loads, conflict-free column reads with a 129-word pitch) and writes whole
// 512-byte tiles; the dense <-> tiled conversions use the same block shape, and
// a plain one-byte-per-thread remap covers the pairs with the transposed layout
// (an offline, once-per-weight step).
#include "wq_common.cuh"
#include "wq_internal.h"

namespace wq {
namespace {

constexpr int kTK = 64, kTC = 16, kTileBytes = 512;
constexpr int kBlockCols = 128;            // 8 tiles of a slab per block
constexpr int kPitch = kBlockCols + 1;     // shared-memory row pitch (words)

// Position (row kk, column cc) of nibble p of word j of lane (g, t) in its tile.
__device__ __forceinline__ void tiled_element(int g, int t, int j, int p, int &kk, int &cc) {
  const int e = ((p & 3) >= 2 ? 2 : 0) + (p >> 2);
  kk = 32 * (j >> 1) + 8 * t + 4 * (j & 1) + e;
  cc = g + 8 * (p & 1);
}

// Source of the 4-bit values: unpacked int32 (K, N), or dense INT4 bytes (K, N/2).
struct FromInt32 {
  const int32_t *v;
  __device__ int32_t at(int64_t k, int64_t n, int64_t N) const { return v[k * N + n]; }
};
struct FromNd {
  const uint8_t *b;
  __device__ int32_t at(int64_t k, int64_t n, int64_t N) const {
    const uint32_t byte = b[k * (N / 2) + n / 2];
    return (int32_t)((n & 1) ? (byte >> 4) : (byte & 0xFu));
  }
};

// grid (ceil(N / 128), ceil(K / 64)); 256 threads: thread = (tile of the block, lane)
template <typename Src>
__global__ void __launch_bounds__(256)
    to_tiled_kernel(Src src, uint8_t *__restrict__ out, int64_t K, int64_t N) {
  __shared__ uint8_t sv[kTK * kPitch];
  const int64_t s = blockIdx.y, n0 = (int64_t)blockIdx.x * kBlockCols;
  for (int i = threadIdx.x; i < kTK * kBlockCols; i += 256) {
    const int r = i / kBlockCols, c = i % kBlockCols;
    const int64_t k = s * kTK + r, n = n0 + c;
    sv[r * kPitch + c] = (k < K && n < N) ? (uint8_t)(src.at(k, n, N) & 0xF) : 0;
  }
  __syncthreads();
  const int tile = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t cg = n0 / kTC + tile;
  if (cg * kTC >= N) return;
  const int g = lane >> 2, t = lane & 3;
  uint32_t w[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    uint32_t word = 0;
#pragma unroll
    for (int p = 0; p < 8; ++p) {
      int kk, cc;
      tiled_element(g, t, j, p, kk, cc);
      word |= (uint32_t)sv[kk * kPitch + tile * kTC + cc] << (4 * p);
    }
    w[j] = word;
  }
  uint8_t *dst = out + ((s * (N / kTC) + cg) * kTileBytes + lane * 16);
  *reinterpret_cast<uint4 *>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
}

// Tiled -> dense INT4 bytes (K, N/2). Same grid and block shape.
__global__ void __launch_bounds__(256)
    to_nd_kernel(const uint8_t *__restrict__ in, uint8_t *__restrict__ out, int64_t K, int64_t N) {
  __shared__ uint8_t sv[kTK * kPitch];
  const int64_t s = blockIdx.y, n0 = (int64_t)blockIdx.x * kBlockCols;
  const int tile = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t cg = n0 / kTC + tile;
  if (cg * kTC < N) {
    const uint4 v = *reinterpret_cast<const uint4 *>(in + (s * (N / kTC) + cg) * kTileBytes + lane * 16);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    const int g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int p = 0; p < 8; ++p) {
        int kk, cc;
        tiled_element(g, t, j, p, kk, cc);
        sv[kk * kPitch + tile * kTC + cc] = (uint8_t)((w[j] >> (4 * p)) & 0xFu);
      }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < kTK * (kBlockCols / 2); i += 256) {
    const int r = i / (kBlockCols / 2), c2 = i % (kBlockCols / 2);
    const int64_t k = s * kTK + r, n = n0 + 2 * c2;
    if (k < K && n < N)
      out[k * (N / 2) + n / 2] = (uint8_t)(sv[r * kPitch + 2 * c2] | (sv[r * kPitch + 2 * c2 + 1] << 4));
  }
}

// Nibble of logical element (k, n) of a (K, N) weight in layout `lay`.
__device__ __forceinline__ uint32_t nibble_at(const uint8_t *w, int lay, int64_t k, int64_t n,
                                              int64_t K, int64_t N) {
  if (lay == WQ_INT4_TILED) return tiled_nibble(w, k, n, N);
  const uint32_t b = lay == WQ_INT4 ? w[k * (N / 2) + n / 2] : w[n * (K / 2) + k / 2];
  const int odd = lay == WQ_INT4 ? (int)(n & 1) : (int)(k & 1);
  return odd ? (b >> 4) : (b & 0xFu);
}

// Logical element (k, n) held by nibble h (0 = bits 3:0) of byte i of a
// (K, N) weight in layout `lay`; false for a padding nibble of the tiled layout.
__device__ __forceinline__ bool element_of(int lay, int64_t i, int h, int64_t K, int64_t N,
                                           int64_t &k, int64_t &n) {
  if (lay == WQ_INT4) {
    k = i / (N / 2);
    n = 2 * (i % (N / 2)) + h;
  } else if (lay == WQ_INT4_T) {
    n = i / (K / 2);
    k = 2 * (i % (K / 2)) + h;
  } else {
    const int64_t tile = i / kTileBytes, r = i % kTileBytes;
    const int lane = (int)(r / 16), j = (int)((r % 16) / 4), p = 2 * (int)(r % 4) + h;
    int kk, cc;
    tiled_element(lane >> 2, lane & 3, j, p, kk, cc);
    k = (tile / (N / kTC)) * kTK + kk;
    n = (tile % (N / kTC)) * kTC + cc;
  }
  return k < K;
}

// One thread per output byte: each of its two nibbles is fetched from the
// source layout (any pair of WQ_INT4, WQ_INT4_T, WQ_INT4_TILED).
__global__ void __launch_bounds__(256)
    remap_kernel(const uint8_t *__restrict__ in, int in_lay, uint8_t *__restrict__ out,
                 int out_lay, int64_t K, int64_t N, int64_t nbytes) {
  for (int64_t i = (int64_t)blockIdx.x * 256 + threadIdx.x; i < nbytes;
       i += (int64_t)gridDim.x * 256) {
    uint32_t byte = 0;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      int64_t k, n;
      if (element_of(out_lay, i, h, K, N, k, n)) byte |= nibble_at(in, in_lay, k, n, K, N) << (4 * h);
    }
    out[i] = (uint8_t)byte;
  }
}

dim3 tiled_grid(int64_t K, int64_t N) {
  return dim3((unsigned)((N + kBlockCols - 1) / kBlockCols), (unsigned)((K + kTK - 1) / kTK), 1);
}

}  // namespace

uint64_t tiled_int4_bytes(int64_t K, int64_t N) {
  return (uint64_t)((K + kTK - 1) / kTK) * kTK * (uint64_t)N / 2;
}

cudaError_t launch_pack_int4_tiled(const int32_t *in, uint8_t *out, int64_t K, int64_t N,
                                   cudaStream_t s) {
  to_tiled_kernel<FromInt32><<<tiled_grid(K, N), 256, 0, s>>>(FromInt32{in}, out, K, N);
  return cudaGetLastError();
}

cudaError_t launch_int4_nd_to_tiled(const uint8_t *in, uint8_t *out, int64_t K, int64_t N,
                                    cudaStream_t s) {
  to_tiled_kernel<FromNd><<<tiled_grid(K, N), 256, 0, s>>>(FromNd{in}, out, K, N);
  return cudaGetLastError();
}

cudaError_t launch_int4_tiled_to_nd(const uint8_t *in, uint8_t *out, int64_t K, int64_t N,
                                    cudaStream_t s) {
  to_nd_kernel<<<tiled_grid(K, N), 256, 0, s>>>(in, out, K, N);
  return cudaGetLastError();
}

cudaError_t launch_int4_remap(const uint8_t *in, int in_layout, uint8_t *out, int out_layout,
                              int64_t K, int64_t N, cudaStream_t s) {
  const int64_t nbytes = out_layout == WQ_INT4_TILED ? (int64_t)tiled_int4_bytes(K, N) : K * N / 2;
  int64_t blocks = (nbytes + 255) / 256;
  const int64_t cap = (int64_t)device_info().sms * 16;
  if (blocks > cap) blocks = cap;
  remap_kernel<<<(unsigned)blocks, 256, 0, s>>>(in, in_layout, out, out_layout, K, N, nbytes);
  return cudaGetLastError();
}

}  // namespace wq
