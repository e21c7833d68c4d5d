// Split-K reduction + bias + residual add + RMSNorm
// (aclnnWeightQuantMatmulAllReduceAddRmsNorm, "Function description":
//   y = mm_out + residual;  normOut = y / sqrt(mean_n(y^2) + epsilon) * gamma).
//
// Input: `parts` fp32 partial products x1 @ W of shape (M, N) in the workspace
// (written by the generic or decode matmul kernel). One thread-block cluster
// of C blocks owns one row: each block sums the partials of its n-range in a
// fixed order, adds bias and residual, writes y, keeps y in registers, and
// reduces sum(y^2) over its range; the C block sums are exchanged through
// distributed shared memory (no global atomics), so every block gets the row's
// total, computes rstd and writes normOut from the registers. y is never read
// back from memory, and the result does not depend on timing.
#include <cooperative_groups.h>

#include "wq_internal.h"
#include "wq_common.cuh"

namespace cg = cooperative_groups;

namespace wq {
namespace {

constexpr int kEpiThreads = 512;
constexpr int kEpiItems = 16;                           // values held per thread
constexpr int64_t kEpiChunk = kEpiThreads * kEpiItems;  // max columns per block

template <int DT, int VEC>
__global__ void __launch_bounds__(kEpiThreads)
    epilogue_kernel(const float *__restrict__ part, int parts, const typename Elem<DT>::T *bias,
                    const typename Elem<DT>::T *residual, const typename Elem<DT>::T *__restrict__ gamma,
                    typename Elem<DT>::T *y, typename Elem<DT>::T *__restrict__ normOut, int64_t M,
                    int64_t N, int64_t chunk, int C, int64_t row_step, float eps) {
  using E = Elem<DT>;
  using T = typename E::T;
  __shared__ float s_warp[kEpiThreads / 32];
  __shared__ float s_block;

  // With programmatic dependent launch this waits for the producing matmul
  // grid; launched normally it returns at once.
  cudaGridDependencySynchronize();

  const int crank = (int)(blockIdx.x % C);
  const int64_t n_begin = crank * chunk;
  const int64_t n_end = (n_begin + chunk < N) ? n_begin + chunk : N;
  const int tid = threadIdx.x;
  constexpr int ITER = kEpiItems / VEC;

  for (int64_t m = blockIdx.x / C; m < M; m += row_step) {
    float v[kEpiItems];
    float ss = 0.f;
#pragma unroll
    for (int it = 0; it < ITER; ++it) {
      const int64_t n = n_begin + ((int64_t)it * kEpiThreads + tid) * VEC;
      if (VEC == 8) {
        if (n < n_end) {
          float a[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) a[j] = 0.f;
          for (int pidx = 0; pidx < parts; ++pidx) {
            const float4 *src = reinterpret_cast<const float4 *>(part + ((int64_t)pidx * M + m) * N + n);
            const float4 p0 = src[0], p1 = src[1];
            a[0] += p0.x; a[1] += p0.y; a[2] += p0.z; a[3] += p0.w;
            a[4] += p1.x; a[5] += p1.y; a[6] += p1.z; a[7] += p1.w;
          }
          const uint4 rr = *reinterpret_cast<const uint4 *>(residual + m * N + n);
          const uint32_t rw[4] = {rr.x, rr.y, rr.z, rr.w};
          uint32_t bw[4] = {0u, 0u, 0u, 0u};
          if (bias) {
            const uint4 bb = *reinterpret_cast<const uint4 *>(bias + n);
            bw[0] = bb.x; bw[1] = bb.y; bw[2] = bb.z; bw[3] = bb.w;
          }
          uint32_t yw[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float2 r2 = unpack2<DT>(rw[j]);
            const float2 b2 = unpack2<DT>(bw[j]);
            const float y0 = a[2 * j] + b2.x + r2.x;
            const float y1 = a[2 * j + 1] + b2.y + r2.y;
            v[it * 8 + 2 * j] = y0;
            v[it * 8 + 2 * j + 1] = y1;
            ss = fmaf(y0, y0, ss);
            ss = fmaf(y1, y1, ss);
            yw[j] = pack2<DT>(y0, y1);
          }
          *reinterpret_cast<uint4 *>(y + m * N + n) = make_uint4(yw[0], yw[1], yw[2], yw[3]);
        }
      } else {
        if (n < n_end) {
          float a = 0.f;
          for (int pidx = 0; pidx < parts; ++pidx) a += part[((int64_t)pidx * M + m) * N + n];
          float yv = a + (bias ? E::to_f(bias[n]) : 0.f) + E::to_f(residual[m * N + n]);
          v[it] = yv;
          ss = fmaf(yv, yv, ss);
          y[m * N + n] = E::from_f(yv);
        }
      }
    }
    // block reduction of ss in a fixed order
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if ((tid & 31) == 0) s_warp[tid >> 5] = ss;
    __syncthreads();
    if (tid == 0) {
      float t = 0.f;
#pragma unroll
      for (int w = 0; w < kEpiThreads / 32; ++w) t += s_warp[w];
      s_block = t;
    }
    float total;
    if (C > 1) {
      cg::cluster_group cluster = cg::this_cluster();
      cluster.sync();  // every block's s_block is written
      total = 0.f;
      for (int r = 0; r < C; ++r) total += *cluster.map_shared_rank(&s_block, r);
      cluster.sync();  // nobody overwrites s_block / exits while others read it
    } else {
      __syncthreads();
      total = s_block;
      __syncthreads();
    }
    const float rstd = rsqrtf(total / (float)N + eps);
#pragma unroll
    for (int it = 0; it < ITER; ++it) {
      const int64_t n = n_begin + ((int64_t)it * kEpiThreads + tid) * VEC;
      if (n >= n_end) continue;
      if (VEC == 8) {
        const uint4 gg = *reinterpret_cast<const uint4 *>(gamma + n);
        const uint32_t gw[4] = {gg.x, gg.y, gg.z, gg.w};
        uint32_t ow[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float2 g2 = unpack2<DT>(gw[j]);
          ow[j] = pack2<DT>(v[it * 8 + 2 * j] * rstd * g2.x, v[it * 8 + 2 * j + 1] * rstd * g2.y);
        }
        *reinterpret_cast<uint4 *>(normOut + m * N + n) = make_uint4(ow[0], ow[1], ow[2], ow[3]);
      } else {
        normOut[m * N + n] = E::from_f(v[it] * rstd * E::to_f(gamma[n]));
      }
    }
  }
}

}  // namespace

void plan_epilogue(const Problem &p, Plan &plan) {
  int64_t C = (p.N + kEpiChunk - 1) / kEpiChunk;
  if (C < 1) C = 1;
  // vector path: 8 columns per access, 16-byte aligned rows and pointers
  bool vec = (p.N % 8 == 0);
  const void *ptrs[] = {p.bias, p.residual, p.gamma, p.y, p.normOut};
  for (const void *q : ptrs)
    if (q && ((uintptr_t)q % 16) != 0) vec = false;
  plan.epi_cluster = (int)C;
  plan.epi_vec = vec;
}

cudaError_t launch_epilogue(const Problem &p, const Plan &plan, const void *ws, bool pdl,
                            cudaStream_t s) {
  const int C = plan.epi_cluster;
  int64_t chunk = (p.N + C - 1) / C;
  if (plan.epi_vec) chunk = (chunk + 7) / 8 * 8;
  int64_t rows = p.M;
  const int64_t max_rows = (int64_t)(0x7fffffff / C);
  if (rows > max_rows) rows = max_rows;
  if (rows > 65536) rows = 65536;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(rows * C), 1, 1);
  cfg.blockDim = dim3(kEpiThreads, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attrs[2];
  int na = 0;
  if (C > 1) {
    attrs[na].id = cudaLaunchAttributeClusterDimension;
    attrs[na].val.clusterDim.x = C;
    attrs[na].val.clusterDim.y = 1;
    attrs[na].val.clusterDim.z = 1;
    ++na;
  }
  if (pdl) {
    attrs[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  cfg.attrs = attrs;
  cfg.numAttrs = na;
  const float *part = reinterpret_cast<const float *>(static_cast<const char *>(ws) + plan.part_off);
  const float eps = p.eps;
#define WQ_EPI_LAUNCH(DT, V)                                                                     \
  cudaLaunchKernelEx(&cfg, epilogue_kernel<DT, V>, part, plan.parts,                            \
                     static_cast<const Elem<DT>::T *>(p.bias),                                  \
                     static_cast<const Elem<DT>::T *>(p.residual),                              \
                     static_cast<const Elem<DT>::T *>(p.gamma), static_cast<Elem<DT>::T *>(p.y), \
                     static_cast<Elem<DT>::T *>(p.normOut), p.M, p.N, chunk, C, rows, eps)
  cudaError_t e;
  if (p.dtype == WQ_BF16)
    e = plan.epi_vec ? WQ_EPI_LAUNCH(WQ_BF16, 8) : WQ_EPI_LAUNCH(WQ_BF16, 1);
  else
    e = plan.epi_vec ? WQ_EPI_LAUNCH(WQ_F16, 8) : WQ_EPI_LAUNCH(WQ_F16, 1);
#undef WQ_EPI_LAUNCH
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace wq
