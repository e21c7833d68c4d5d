// Large-M kernel of the fused operator for transposed INT4 weights
// (aclnnWeightQuantMatmulAllReduceAddRmsNorm, "Function description" and the
// constraint that x2 may be given transposed: x2 stored as (N, K), packed two
// per byte along K) with bf16 per-group scales and no offset.
//
// The product is computed transposed, D^T = W^T x1^T: the dequantized weight
// is the MMA's A operand and lives in tensor memory, where the dequant warps
// store it with tcgen05.st; only x1 (the B operand) passes through shared
// memory. Per 64-deep k-step a CTA moves 32 KB of x1 and 4 KB of packed
// weights into shared memory and the MMAs read the x1 tile once -- against
// ~190 KB of shared-memory traffic per k-step of the same work when the
// dequantized weight is the B operand in shared memory.
//
// Output tile: 128 weight columns (the 128 TMEM lanes, MMA M = 128) x 256
// rows of x1 (MMA N = 256), tiles in row-block-major order, one persistent CTA
// per SM; each dequantized weight element serves 256 rows. Warp roles (16):
//   warp 0       TMA producer, per k-step: x1 tile (256 rows x 64, fp16 copy
//                with a per-row power of two, 128-byte swizzle, K-major), the
//                tile's 128 packed weight rows (32 bytes each, 32-byte swizzle)
//                and two rows of scale words.
//   warp 1       TMEM owner (512 columns: D at 0, eight A stages of 32 columns
//                at 256 + 32 s) and MMA issuer (kind::f16, A from TMEM, B from
//                shared memory, M = 128, N = 256, K = 16).
//   warps 4-11   dequant: warp (k half p, lane quarter q) owns weight row
//                n = 32 q + lane of the tile and k 32 p .. 32 p + 31 of each
//                k-step: it reads those 16 bytes from the stage, forms q * S16
//                in fp16 (exact) as 16 columns of (k even, k odd) pairs and
//                stores them to its TMEM lane. The odd k's nibble is used in
//                place at bits 7:4 (as 1152 + 16 q, with S16 / 16), the even
//                k's at bits 3:0 (1032 + q, with S16).
//   warps 12-15  epilogue, lane quarter q: thread = weight column n, TMEM
//                columns = rows m. y = acc * 2^(e_m + e_n) + bias + residual,
//                the residual read as 32 x 32 TMA boxes ([m][n], two ahead), y
//                written column-wise into a shared box and stored as coalesced
//                box rows; each warp forms per-row sums of y^2 over its 32
//                columns of the tile (a butterfly over the lanes leaves row j's
//                sum in lane j) in shared memory, and once all four warps have
//                (an mbarrier, bounded wait) warp q adds the four in a fixed
//                order for rows 64 q .. 64 q + 63 and publishes one partial per
//                row and n-tile; the accumulator is handed back once read.
//                Then the previous tile's rows (64 per warp) are normalised a
//                row per warp instruction once every partial of their row
//                block is published.
// Every wait is bounded; on timeout the kernel records the place in the
// status word, drains its copies and MMAs, frees TMEM and exits.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "wq_common.cuh"
#include "wq_internal.h"
#include "wq_sm100.cuh"
#include "wq_sync.cuh"

namespace wq {
namespace {

using namespace sm100;

constexpr int TM = 256, TN = 128, TK = 64;
constexpr int NRX = 4;  // x1 + weight stages in shared memory
constexpr int NRA = 8;  // weight stages in tensor memory (32 columns each)
constexpr int kThreadsT = 512;
constexpr int kDq0 = 4, kDqN = 8, kEpi0 = 12, kEpiN = 4;
constexpr uint32_t kTmemColsT = 512, kColA = 256;
constexpr int kNRes = 3;           // residual boxes per epilogue warp
constexpr uint32_t kBox = 32 * 64; // 32 rows x 32 columns x 2 bytes
constexpr int kPartsPerLaneT = 10; // row partials read by a normalising lane: one per n-tile, <= 296 n-tiles

enum WhereT : uint32_t {
  kTWProducer = 1, kTWMma = 2, kTWDequant = 3, kTWEpi = 4, kTWRowBlock = 5
};

struct TArgs {
  const int16_t *e_row, *e_col;
  const void *bias, *gamma;
  void *y, *normOut;
  uint32_t *status, *counters;
  float *rowpart;
  long long M;
  int K, N, group, nTilesN, kTiles;
  long long nTiles;
  float eps;
  long long budget;
  uint32_t extra;
};

// A stage: x1 tile (32 KB, 128-byte swizzle), the tile's packed weight rows
// (128 rows x 32 bytes, 32-byte swizzle) and two rows of scale words (1 KB).
struct LayoutT {
  static constexpr uint32_t X_BYTES = TM * TK * 2;                  // 32 KB
  static constexpr uint32_t W_BYTES = TN * TK / 2;                  // 4 KB
  static constexpr uint32_t S_BYTES = 2 * TN * 4;                   // 1 KB
  static constexpr uint32_t STAGE = X_BYTES + W_BYTES + S_BYTES;    // 37 KB, 1024-aligned
  static constexpr uint32_t X_OFF = 0;
  static constexpr uint32_t EPI_OFF = X_OFF + NRX * STAGE;          // 1024-aligned
  // per-warp sums of y^2 of the tile's rows, two buffers: float [2][kEpiN][TM]
  static constexpr uint32_t PART_OFF = EPI_OFF + kEpiN * (kNRes + 1) * kBox;
  static constexpr uint32_t BAR_OFF = PART_OFF + 2 * kEpiN * TM * 4;
  static constexpr int NBARS = 2 * NRX + 2 * NRA + 2 + 1 + kEpiN * kNRes + 2;
  static constexpr uint32_t SMEM = BAR_OFF + 8 * NBARS + 16 + 1024;
  static_assert(SMEM <= 232448, "shared memory per CTA");
};

#define TXFULL(s) (s)
#define TXEMPTY(s) (NRX + (s))
#define TAFULL(s) (2 * NRX + (s))
#define TAEMPTY(s) (2 * NRX + NRA + (s))
#define TACCFULL() (2 * NRX + 2 * NRA)
#define TACCEMPTY() (2 * NRX + 2 * NRA + 1)
#define TDRAIN() (2 * NRX + 2 * NRA + 2)
#define TRESFULL(q, b) (2 * NRX + 2 * NRA + 3 + kNRes * (q) + (b))
#define TPARTFULL(b) (2 * NRX + 2 * NRA + 3 + kNRes * kEpiN + (b))

// D[tmem] (+)= A[tmem] * B[smem]^T, kind::f16, A read from tensor memory.
__device__ __forceinline__ void mma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc,
                                           uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// 32 lanes x 16 columns of 32-bit TMEM words from registers.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15])
      : "memory");
}

__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// (v - c) * s on fp16 pairs, each step one IEEE rounding (exact here)
__device__ __forceinline__ uint32_t sub_mul2_h(uint32_t v, uint32_t c, uint32_t s) {
  uint32_t r;
  asm("{\n\t.reg .b32 t;\n\t"
      "sub.rn.f16x2 t, %1, %2;\n\t"
      "mul.rn.f16x2 %0, t, %3;\n\t}"
      : "=r"(r)
      : "r"(v), "r"(c), "r"(s));
  return r;
}

__global__ void __launch_bounds__(kThreadsT, 1)
    prefill_t_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w,
                     const __grid_constant__ CUtensorMap tm_s, const __grid_constant__ CUtensorMap tm_r,
                     const TArgs a) {
  using L = LayoutT;
  using T = __nv_bfloat16;
  extern __shared__ uint8_t smem_raw_t[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw_t) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  auto BAR = [&](int i) -> uint32_t { return sbase + L::BAR_OFF + 8u * i; };
  uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + L::BAR_OFF + 8 * L::NBARS);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_holder + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NRX; ++s) {
      mbar_init(BAR(TXFULL(s)), 1);
      mbar_init(BAR(TXEMPTY(s)), 1);
    }
    for (int s = 0; s < NRA; ++s) {
      mbar_init(BAR(TAFULL(s)), kDqN);
      mbar_init(BAR(TAEMPTY(s)), 1);
    }
    mbar_init(BAR(TACCFULL()), 1);
    mbar_init(BAR(TACCEMPTY()), kEpiN);
    mbar_init(BAR(TDRAIN()), 1);
    for (int q = 0; q < kEpiN; ++q)
      for (int b = 0; b < kNRes; ++b) mbar_init(BAR(TRESFULL(q, b)), 1);
    mbar_init(BAR(TPARTFULL(0)), kEpiN);
    mbar_init(BAR(TPARTFULL(1)), kEpiN);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tm_x);
    prefetch_tmap(&tm_w);
    prefetch_tmap(&tm_s);
    prefetch_tmap(&tm_r);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_holder), kTmemColsT);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA producer
    const uint64_t pol_w = policy_evict_last();  // weights are re-read by every row block
    long long it = 0;
    for (long long t = blockIdx.x; t < a.nTiles; t += gridDim.x) {
      const int rb = (int)(t / a.nTilesN), nt = (int)(t % a.nTilesN);
      for (int ks = 0; ks < a.kTiles; ++ks, ++it) {
        const int s = (int)(it % NRX);
        if (!wait_bar_warp(BAR(TXEMPTY(s)), (uint32_t)(((it / NRX) & 1) ^ 1), abort_flag, a.status,
                           kTWProducer))
          goto pdone;
        if (lane == 0) {
          const uint32_t st = sbase + L::X_OFF + s * L::STAGE;
          mbar_arrive_expect_tx(BAR(TXFULL(s)), L::STAGE);
          tma_load_2d(st, &tm_x, ks * TK, rb * TM, BAR(TXFULL(s)));
          tma_load_2d_hint(st + L::X_BYTES, &tm_w, ks * (TK / 2), nt * TN, BAR(TXFULL(s)), pol_w);
          tma_load_2d(st + L::X_BYTES + L::W_BYTES, &tm_s, nt * TN, (ks * TK) / a.group, BAR(TXFULL(s)));
        }
        __syncwarp();
      }
    }
  pdone:
    for (long long j = (it > NRX ? it - NRX : 0); j < it; ++j)
      drain_bar(BAR(TXFULL((int)(j % NRX))), (uint32_t)((j / NRX) & 1));
    __syncwarp();
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    {
      const uint32_t idesc = idesc_f16(0u, 128, TM);  // fp16 x fp16, M = 128 (weight columns), N = 256
      long long it = 0;
      int lt = 0;
      for (long long t = blockIdx.x; t < a.nTiles; t += gridDim.x, ++lt) {
        if (!wait_bar_warp(BAR(TACCEMPTY()), (uint32_t)((lt & 1) ^ 1), abort_flag, a.status, kTWMma))
          goto mdone;
        tc_fence_after();
        for (int ks = 0; ks < a.kTiles; ++ks, ++it) {
          const int s = (int)(it % NRX), sa = (int)(it % NRA);
          if (!wait_bar_warp(BAR(TXFULL(s)), (uint32_t)((it / NRX) & 1), abort_flag, a.status, kTWMma))
            goto mdone;
          if (!wait_bar_warp(BAR(TAFULL(sa)), (uint32_t)((it / NRA) & 1), abort_flag, a.status, kTWMma))
            goto mdone;
          tc_fence_after();
          if (lane == 0) {
            const uint32_t xaddr = sbase + L::X_OFF + s * L::STAGE;
#pragma unroll
            for (int kk = 0; kk < TK / 16; ++kk)
              mma_f16_ts(tmem_base, tmem_base + kColA + (uint32_t)(sa * 32 + kk * 8),
                         desc_kmajor_sw128(xaddr + kk * 32), idesc, (ks | kk) != 0 ? 1u : 0u);
            mma_commit(BAR(TXEMPTY(s)));
            mma_commit(BAR(TAEMPTY(sa)));
          }
          __syncwarp();
        }
        if (lane == 0) mma_commit(BAR(TACCFULL()));
        __syncwarp();
      }
    mdone:
      if (lane == 0) mma_commit(BAR(TDRAIN()));
      __syncwarp();
      drain_bar(BAR(TDRAIN()), 0);
      __syncwarp();
    }
  } else if (warp >= kDq0 && warp < kDq0 + kDqN) {
    // ---------------------------------------------------------------- dequant
    const int hp = (warp - kDq0) >> 2, q = warp & 3;  // k half, lane quarter
    const uint32_t lane_base = tmem_base + ((uint32_t)(32 * q) << 16) + kColA + (uint32_t)(hp * 16);
    const int r = 32 * q + lane;  // weight row of the tile
    // this thread's 16-byte chunk hp of the row in the 32-byte-swizzled weight
    // block: chunk c of row r at r * 32 + 16 (c ^ ((r >> 2) & 1))
    const uint32_t woff = (uint32_t)(r * 32 + 16 * (hp ^ ((r >> 2) & 1)));
    long long it = 0;
    for (long long t = blockIdx.x; t < a.nTiles; t += gridDim.x) {
      for (int ks = 0; ks < a.kTiles; ++ks, ++it) {
        const int s = (int)(it % NRX), sa = (int)(it % NRA);
        if (!wait_bar_warp(BAR(TXFULL(s)), (uint32_t)((it / NRX) & 1), abort_flag, a.status, kTWDequant))
          goto ddone;
        const uint32_t st = sbase + L::X_OFF + s * L::STAGE;
        uint32_t w[4];
        asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                     : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
                     : "r"(st + L::X_BYTES + woff));
        // the scale word of this 32-deep half: row (k0 + 32 hp) / group of the
        // copied pair, whose first row is k0 / group
        const int k0 = ks * TK;
        const uint32_t srow = (uint32_t)((k0 + 32 * hp) / a.group - k0 / a.group);
        uint32_t sc;
        asm volatile("ld.shared.b32 %0, [%1];"
                     : "=r"(sc)
                     : "r"(st + L::X_BYTES + L::W_BYTES + 4u * (srow * TN + r)));
        if (!wait_bar_warp(BAR(TAEMPTY(sa)), (uint32_t)(((it / NRA) & 1) ^ 1), abort_flag, a.status,
                           kTWDequant))
          goto ddone;
        tc_fence_after();
        {
          uint32_t out[16];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
#pragma unroll
            for (int p = 0; p < 4; ++p) {
              // byte p of word i holds k = 8i + 2p (bits 3:0) and 8i + 2p + 1 (bits 7:4)
              // of this half
              const uint32_t x = __byte_perm(w[i], 0u, (uint32_t)(p | (p << 8)));
              const uint32_t v = (x & 0x00F0000Fu) ^ 0x64806408u;
              out[4 * i + p] = sub_mul2_h(v, 0x64806408u, sc);
            }
          }
          tmem_st16(lane_base + (uint32_t)(sa * 32), out);
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(BAR(TAFULL(sa)));
      }
    }
  ddone:;
  } else if (warp >= kEpi0) {
    // ---------------------------------------------------------------- epilogue
    const int q = warp & 3;  // TMEM lane quarter
    const T *bias = static_cast<const T *>(a.bias);
    const T *gam = static_cast<const T *>(a.gamma);
    const T *yin = static_cast<const T *>(a.y);
    T *yout = static_cast<T *>(a.y);
    T *nout = static_cast<T *>(a.normOut);
    const uint32_t lane_addr = tmem_base + ((uint32_t)(32 * q) << 16);
    const uint32_t rbox = sbase + L::EPI_OFF + (uint32_t)q * (kNRes + 1) * kBox;
    const uint32_t ybox = rbox + (uint32_t)kNRes * kBox;
    float *part = reinterpret_cast<float *>(smem + L::PART_OFF);
    uint32_t rc = 0, issued = 0;
    int lt = 0;
    long long prev_t = -1;
    bool ok = true;

    auto normalize = [&](long long t) -> bool {
      const int rb = (int)(t / a.nTilesN), nt = (int)(t % a.nTilesN);
      {
        const uint32_t target = (uint32_t)(kEpiN * a.nTilesN) + a.extra;
        bool done = false;
        if (lane == 0) {
          const long long t0 = clock64();
          while (true) {
            done = ld_acquire_u32(a.counters + rb) >= target;
            if (done || *abort_flag) break;
            if (clock64() - t0 > a.budget) {
              *abort_flag = 1;
              record_timeout(a.status, kTWRowBlock);
              break;
            }
            __nanosleep(64);
          }
        }
        done = __shfl_sync(0xffffffffu, done, 0);
        __syncwarp();
        if (!done) return false;
      }
      // lane l: columns 4 l .. 4 l + 3 of the 128-column tile (8 bytes)
      const int n = nt * TN + 4 * lane;
      const bool col_ok = n < a.N;
      uint2 g = make_uint2(0u, 0u);
      if (col_ok) g = *reinterpret_cast<const uint2 *>(gam + n);
      const uint32_t gw[2] = {g.x, g.y};
      const long long mbase = (long long)rb * TM + 64 * q;
#pragma unroll 1
      for (int r0 = 0; r0 < 64; r0 += 4) {
        float pv[4][kPartsPerLaneT];
        uint2 yv[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const long long m = mbase + r0 + u;
          const bool live = m < a.M;
          const float *rp = a.rowpart + m * a.nTilesN;
#pragma unroll
          for (int i = 0; i < kPartsPerLaneT; ++i) {
            const int j = lane + 32 * i;
            pv[u][i] = live && j < a.nTilesN ? __ldcg(rp + j) : 0.f;
          }
          yv[u] = make_uint2(0u, 0u);
          if (live && col_ok) yv[u] = __ldcg(reinterpret_cast<const uint2 *>(yin + m * a.N + n));
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const long long m = mbase + r0 + u;
          float tot = 0.f;
#pragma unroll
          for (int i = 0; i < kPartsPerLaneT; ++i) tot += pv[u][i];
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, o);
          if (m < a.M && col_ok) {
            const float rstd = rsqrtf(tot / (float)a.N + a.eps);
            const uint32_t yw[2] = {yv[u].x, yv[u].y};
            uint32_t o2[2];
#pragma unroll
            for (int i = 0; i < 2; ++i) {
              const float2 y2 = unpack2<WQ_BF16>(yw[i]), g2 = unpack2<WQ_BF16>(gw[i]);
              o2[i] = pack2<WQ_BF16>(y2.x * rstd * g2.x, y2.y * rstd * g2.y);
            }
            *reinterpret_cast<uint2 *>(nout + m * a.N + n) = make_uint2(o2[0], o2[1]);
          }
        }
      }
      return true;
    };

    // residual box k of a tile: rows 32 (k % 8) of the row block, this warp's
    // 32 columns of the tile (each tile takes exactly 8 boxes)
    auto load_res = [&](uint32_t k, long long t) {
      issued = k + 1;
      if (lane == 0) {
        const int rb = (int)(t / a.nTilesN), nt = (int)(t % a.nTilesN);
        const int c = (int)(k % 8);
        fence_proxy_async_smem();
        const uint32_t bar = BAR(TRESFULL(q, (int)(k % kNRes)));
        mbar_arrive_expect_tx(bar, kBox);
        tma_load_2d(rbox + (k % kNRes) * kBox, &tm_r, nt * TN + 32 * q, rb * TM + 32 * c, bar);
      }
    };

    for (long long t = blockIdx.x; t < a.nTiles && ok; t += gridDim.x, ++lt) {
      const int rb = (int)(t / a.nTilesN), nt = (int)(t % a.nTilesN);
      const uint32_t rc0 = rc;  // boxes rc0 .. rc0 + 7 belong to this tile
      load_res(rc0, t);
      load_res(rc0 + 1, t);
      // per-row exponents of this row block: lane j of chunk c holds row 32 c + j
      int erow[8];
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const long long m = (long long)rb * TM + 32 * c + lane;
        erow[c] = m < a.M ? (int)a.e_row[m] : 0;
      }
      const long long n = (long long)nt * TN + 32 * q + lane;
      const bool col_ok = n < a.N;
      const int en = col_ok ? (int)a.e_col[n] : 0;
      const float bv = (bias && col_ok) ? __bfloat162float(bias[n]) : 0.f;
      if (!wait_bar_warp(BAR(TACCFULL()), (uint32_t)(lt & 1), abort_flag, a.status, kTWEpi)) {
        ok = false;
        break;
      }
      tc_fence_after();
#pragma unroll 1
      for (int c = 0; c < 8; ++c, ++rc) {
        if (c + 2 < 8) load_res(rc0 + (uint32_t)(c + 2), t);
        uint32_t r[32];
        tmem_ld32(lane_addr + (uint32_t)(32 * c), r);
        tmem_wait_ld();
        if (!wait_bar_warp(BAR(TRESFULL(q, (int)(rc % kNRes))), (rc / kNRes) & 1u, abort_flag,
                           a.status, kTWEpi)) {
          ok = false;
          break;
        }
        const uint32_t rbx = rbox + (rc % kNRes) * kBox;
        int erc = erow[0];
#pragma unroll
        for (int i = 1; i < 8; ++i) erc = c == i ? erow[i] : erc;
        float sq[32];
        __syncwarp();  // every lane has read the previous y box
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const int em = __shfl_sync(0xffffffffu, erc, j);
          uint16_t rr;
          asm volatile("ld.shared.u16 %0, [%1];" : "=h"(rr) : "r"(rbx + (uint32_t)(j * 64 + 2 * lane)));
          const float yv = scale_pow2(__uint_as_float(r[j]), em + en) + bv +
                           __bfloat162float(__ushort_as_bfloat16(rr));
          const long long m = (long long)rb * TM + 32 * c + j;
          sq[j] = (col_ok && m < a.M) ? yv * yv : 0.f;
          const uint16_t yb = __bfloat16_as_ushort(__float2bfloat16_rn(yv));
          asm volatile("st.shared.u16 [%0], %1;" ::"r"(ybox + (uint32_t)(j * 64 + 2 * lane)), "h"(yb)
                       : "memory");
        }
        // sums over the warp's 32 columns: a butterfly leaves row j's sum in lane j
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) {
#pragma unroll
          for (int k = 0; k < o; ++k) {
            const bool upper = (lane & o) != 0;
            const float send = upper ? sq[k] : sq[k + o];
            const float keep = upper ? sq[k + o] : sq[k];
            sq[k] = keep + __shfl_xor_sync(0xffffffffu, send, o);
          }
        }
        part[((lt & 1) * kEpiN + q) * TM + 32 * c + lane] = sq[0];
        __syncwarp();
        // whole box rows: lanes 4i .. 4i+3 store row 8u + i
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int rr = 8 * u + (lane >> 2), jj = lane & 3;
          const long long my = (long long)rb * TM + 32 * c + rr;
          const long long ny = (long long)nt * TN + 32 * q + 8 * jj;
          uint32_t q0, q1, q2, q3;
          asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                       : "=r"(q0), "=r"(q1), "=r"(q2), "=r"(q3)
                       : "r"(ybox + (uint32_t)(rr * 64 + jj * 16)));
          if (my < a.M && ny < a.N)
            *reinterpret_cast<uint4 *>(yout + my * a.N + ny) = make_uint4(q0, q1, q2, q3);
        }
      }
      if (!ok) break;
      // the accumulator has been read: hand it back to the MMA issuer; this
      // warp's partial of every row of the tile is published with the count
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(BAR(TACCEMPTY()));
      // the four warps' sums of each row, added in warp order; warp q takes
      // rows 64 q .. 64 q + 63 and publishes them
      if (lane == 0) mbar_arrive(BAR(TPARTFULL(lt & 1)));
      if (!wait_bar_warp(BAR(TPARTFULL(lt & 1)), (uint32_t)((lt >> 1) & 1), abort_flag, a.status,
                         kTWEpi)) {
        ok = false;
        break;
      }
      {
        const float *pb = part + (lt & 1) * kEpiN * TM;
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int ml = 64 * q + 32 * u + lane;
          const float tot = ((pb[ml] + pb[TM + ml]) + pb[2 * TM + ml]) + pb[3 * TM + ml];
          const long long m = (long long)rb * TM + ml;
          if (m < a.M) a.rowpart[m * a.nTilesN + nt] = tot;
        }
      }
      __syncwarp();
      if (lane == 0) {
        __threadfence();
        red_release_add(a.counters + rb, 1u);
      }
      __syncwarp();
      if (prev_t >= 0) {
        if (!normalize(prev_t)) {
          ok = false;
          break;
        }
      }
      prev_t = t;
    }
    if (lane == 0) {
      for (uint32_t k = rc; k < issued; ++k)
        drain_bar(BAR(TRESFULL(q, (int)(k % kNRes))), (k / kNRes) & 1u);
    }
    __syncwarp();
    if (ok && prev_t >= 0) normalize(prev_t);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemColsT);
  }
}

using EncodeTiledFnT = PFN_cuTensorMapEncodeTiled_v12000;

EncodeTiledFnT encode_fn_t() {
  static EncodeTiledFnT fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFnT>(p);
    else
      cudaGetLastError();
  });
  return fn;
}

bool a16(const void *p) { return p == nullptr || (reinterpret_cast<uintptr_t>(p) % 16) == 0; }
uint64_t al256(uint64_t v) { return (v + 255) / 256 * 256; }

}  // namespace

bool prefill_t_applicable(const Problem &p) {
  if (!p.transposed || p.wbits != 4 || p.dtype != WQ_BF16) return false;
  if (p.smode != kPerGroup || p.offset) return false;
  if (p.M < 1 || p.N < 1 || p.K % TK != 0 || p.N % 32 != 0) return false;
  if (p.group % 32 != 0 || p.G < 2) return false;  // a stage copies two scale rows
  const void *ptrs[] = {p.x1, p.x2, p.scale, p.bias, p.residual, p.gamma, p.y, p.normOut};
  for (const void *q : ptrs)
    if (!a16(q)) return false;
  // row-block waits: a CTA normalises tile t - 1 after publishing tile t, so every
  // wait depends only on smaller tile indices while n-tiles per row <= 2 x grid
  const int64_t nt = (p.N + TN - 1) / TN;
  if (nt > 2 * device_info().sms || nt > 32 * kPartsPerLaneT) return false;
  return true;
}

bool plan_prefill_t(const Problem &p, Plan &plan) {
  if (!prefill_t_applicable(p)) return false;
  plan.kernel = WQ_KERNEL_PREFILL;
  plan.mode = 2;  // transposed operands
  plan.n_tiles = (p.N + TN - 1) / TN;
  plan.m_tiles = (p.M + TM - 1) / TM;
  plan.m_halves = 1;
  const int64_t tiles = plan.n_tiles * plan.m_tiles;
  const int64_t sms = device_info().sms;
  plan.grid = (int)(tiles < sms ? tiles : sms);
  uint64_t off = kWsHeader;
  plan.cnt_off = off;
  off += al256((uint64_t)plan.m_tiles * 4);
  plan.rowpart_off = off;
  off += al256((uint64_t)p.M * (uint64_t)plan.n_tiles * sizeof(float));
  plan.erow_off = off;
  off += al256((uint64_t)p.M * sizeof(int16_t));
  plan.ecol_off = off;
  off += al256((uint64_t)p.N * sizeof(int16_t));
  plan.s16_off = off;
  off += al256((uint64_t)p.G * (uint64_t)p.N * 4);
  plan.x16_off = off;
  off += al256((uint64_t)p.M * (uint64_t)p.K * 2);
  plan.ws_bytes = off;
  return true;
}

cudaError_t launch_prefill_t(const Problem &p, const Plan &plan, void *ws, cudaStream_t s) {
  using L = LayoutT;
  static std::once_flag attr_once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(attr_once, [] {
    attr_err = cudaFuncSetAttribute(prefill_t_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)L::SMEM);
  });
  if (attr_err != cudaSuccess) return attr_err;
  EncodeTiledFnT enc = encode_fn_t();
  if (!enc) return cudaErrorNotSupported;
  char *wsb = static_cast<char *>(ws);

  TArgs args = {};
  args.bias = p.bias; args.gamma = p.gamma; args.y = p.y; args.normOut = p.normOut;
  args.status = reinterpret_cast<uint32_t *>(ws);
  args.counters = reinterpret_cast<uint32_t *>(wsb + plan.cnt_off);
  args.rowpart = reinterpret_cast<float *>(wsb + plan.rowpart_off);
  args.M = p.M; args.K = (int)p.K; args.N = (int)p.N; args.group = (int)p.group;
  args.nTilesN = (int)plan.n_tiles;
  args.kTiles = (int)(p.K / TK);
  args.nTiles = plan.n_tiles * plan.m_tiles;
  args.eps = p.eps;
  args.budget = wait_budget();
  args.extra = wait_extra_arrivals();

  // status word and row-block counters start at zero on every call
  cudaError_t e = cudaMemsetAsync(ws, 0, plan.rowpart_off, s);
  if (e != cudaSuccess) return e;
  int16_t *e_row = reinterpret_cast<int16_t *>(wsb + plan.erow_off);
  int16_t *e_col = reinterpret_cast<int16_t *>(wsb + plan.ecol_off);
  uint32_t *S16T = reinterpret_cast<uint32_t *>(wsb + plan.s16_off);
  __half *x16 = reinterpret_cast<__half *>(wsb + plan.x16_off);
  e = launch_row_prep(p, nullptr, e_row, x16, nullptr, 0, s);
  if (e != cudaSuccess) return e;
  e = launch_so_prep_t(p, e_col, S16T, s);
  if (e != cudaSuccess) return e;
  args.e_row = e_row; args.e_col = e_col;

  CUtensorMap tm_x, tm_w, tm_s, tm_r;
  {
    const cuuint64_t dims[2] = {(cuuint64_t)p.K, (cuuint64_t)p.M};
    const cuuint64_t strides[1] = {(cuuint64_t)p.K * 2};
    const cuuint32_t box[2] = {TK, TM};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(&tm_x, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, x16, dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  }
  {
    // packed weight rows: (N, K/2) bytes, boxes of 32 bytes x 256 rows, 32-byte swizzle
    const cuuint64_t dims[2] = {(cuuint64_t)p.K / 2, (cuuint64_t)p.N};
    const cuuint64_t strides[1] = {(cuuint64_t)p.K / 2};
    const cuuint32_t box[2] = {TK / 2, TN};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(&tm_w, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(p.x2), dims, strides,
                     box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_32B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  }
  {
    // scale words: (G, N), boxes of 256 columns x 2 rows
    const cuuint64_t dims[2] = {(cuuint64_t)p.N, (cuuint64_t)p.G};
    const cuuint64_t strides[1] = {(cuuint64_t)p.N * 4};
    const cuuint32_t box[2] = {TN, 2};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(&tm_s, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, S16T, dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  }
  {
    const cuuint64_t dims[2] = {(cuuint64_t)p.N, (cuuint64_t)p.M};
    const cuuint64_t strides[1] = {(cuuint64_t)p.N * 2};
    const cuuint32_t box[2] = {32, 32};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(&tm_r, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(p.residual), dims,
                     strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  }
  prefill_t_kernel<<<plan.grid, kThreadsT, L::SMEM, s>>>(tm_x, tm_w, tm_s, tm_r, args);
  return cudaGetLastError();
}

}  // namespace wq
