// Prefill (large-M) kernel of the weight-only quantized matmul with the fused
// residual-add + RMSNorm epilogue (aclnnWeightQuantMatmulAllReduceAddRmsNorm,
// "Function description": mm_out = x1 @ (x2*antiquantScale + antiquantOffset)
// + bias; y = mm_out + residual; normOut = y / RMS(y) * gamma).
//
// One persistent CTA per SM walks output tiles of (128 MH) x 256, row blocks
// in pairs with their tiles interleaved (tile_coords), MH = 1 or (INT4 weights, M > 128) 2: with two 128-row
// halves one dequantized INT4 weight tile feeds twice the MMAs (INT8 weights
// are cheap to dequantize and gain nothing from it). Warp roles (16 warps):
//   warp 0       TMA producer: x1 tile (128 MH x 64, 128-byte swizzle) and the
//                packed weight tile (64 k-rows x 256 n, INT4 or INT8) per k-step.
//   warp 1       TMEM owner (512 columns: two 128 x 256 fp32 accumulators, or
//                the two halves of one) and tcgen05.mma issuer (M=128, N=256,
//                K=16, kind::f16; one MMA per half).
//   warps 4-11   dequant: packed weight -> B operand (W^T, 256 x 64, K-major,
//                128-byte swizzle), in one of two forms (below).
//   warps 12-15  epilogue (one per TMEM lane quarter): y = acc + bias +
//                residual, with the residual read and y written as 32 x 32
//                boxes through shared memory by the TMA (the next residual box
//                is in flight while one is used); per-row partial sum(y^2) (of
//                the fp32 y) published to the workspace; the accumulator is
//                handed back to the MMA as soon as it has been read. Then, for
//                the previous tile, wait until every n-tile of its row block
//                has published and write normOut = y * rstd * gamma a row per
//                warp instruction (coalesced), rstd from the partials summed in
//                a fixed order, y from L2 (a row block of y is 128 MH x N x 2 bytes).
// Operand modes:
//   RAWQ   per-tensor / per-channel scales: B holds the integer q itself (exact
//          in fp16 and bf16), the MMA accumulates x1*q in fp32, and the epilogue
//          applies mm = S[n]*acc + O[n]*rowsum(x1[m,:]) + bias.
//   F16EMU bf16 per-group scales: A is an fp16 copy of x1 scaled by a per-row
//          power of two 2^-e_m that puts the row maximum in [2^13, 2^14) (exact
//          for every element within 2^27 of the row maximum) and B = q*S16 in
//          fp16, where S16 is the scale times a per-column power of two 2^-e_n.
//          For INT4, q*S16 is exact (8-bit significand x 3-bit q <= 11 bits);
//          for INT8 it rounds once, at 2^-11. An offset is not added to B (that
//          sum would round): its term sum_g O[g][n] * sum_{k in g} x1[m][k]
//          runs as kTilesX extra k-steps of bf16 MMAs into the same
//          accumulator, A = the per-group row sums of the fp16 copy split into
//          bf16 hi + lo (to 2^-18), B = O * 2^-e_n in bf16 (exact), both loaded by
//          TMA straight into the MMA's operand layout. The epilogue multiplies
//          by 2^(e_m + e_n). Rounding W to bf16 instead (2^-9) would put the
//          result outside the operator's stated tolerance at these K.
// Pipelines: NR raw stages (x1 + packed weight) and NB dequantized-weight
// stages, each guarded by full/empty mbarriers. With MH = 1 two accumulator
// buffers let the epilogue of tile j overlap the main loop of tile j+1; with
// MH = 2 the single accumulator is handed back as soon as the epilogue has
// read it. The wait for a row block never holds an accumulator.
//
// Cross-CTA row reduction: all CTAs are co-resident (grid <= SMs, 1 CTA/SM)
// and a CTA publishes tile j before it waits for the row block of tile j-1;
// with n-tiles per row <= grid size every wait depends only on tiles with a
// smaller index, so the waits always end. Every wait is bounded anyway: on
// timeout the kernel sets the workspace status word, stops waiting and exits
// after draining its own copies and MMAs, leaving the context usable.
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

constexpr int BM = 128, BN = 256, BK = 64;
// Stage counts: NR raw stages (x1 tile + packed weight tile + scale/offset
// rows) and NB dequantized-weight stages, within 227 KB of shared memory next
// to the epilogue's 32 KB of residual and y boxes: INT8 tiles are twice as
// large, and a 256-row x1 tile twice as large again.
template <int WBITS, int MH, int MODE> struct Stages {
  static constexpr int NR = MH == 2 ? 3 : (WBITS == 4 && MODE == 0 ? 4 : 3);
  static constexpr int NB = MH == 2 || (WBITS == 8 && MODE == 1) ? 2 : 3;
};
constexpr int SO_ROWS = 3;  // group rows a 64-deep k-stage can touch (group >= 32)
constexpr int kThreads = 512;
constexpr int kDqWarp0 = 4, kDqWarps = 8;
constexpr int kEpiWarp0 = 12, kEpiWarps = 4;
constexpr uint32_t kTmemCols = 512;
// n-tiles per row are at most the grid (<= SMs): 5 per lane cover 160
constexpr int kPartsPerLane = 5;

// Where a bounded wait gave up (upper bits of the status word).
enum Where : uint32_t {
  kWhereProducer = 1, kWhereMma = 2, kWhereDequant = 3, kWhereEpiAcc = 4, kWhereRowBlock = 5
};

enum Mode : int { kRawQ = 0, kF16Emu = 1 };

struct PrefillArgs {
  const void *scale, *offset, *bias, *residual, *gamma;
  void *y, *normOut;
  uint32_t *status;
  uint32_t *counters;
  float *rowpart;
  const float *rowsum;       // RAWQ with offset: sum_k x1[m, k]
  const int16_t *e_row;      // F16EMU: row exponents
  const int16_t *e_col;      // F16EMU: column exponents
  const uint32_t *S16;       // F16EMU: scaled fp16 scale pairs (G x ld words)
  long long M;
  int K, N, group, Ns, nTilesN, kTiles;
  int kTilesX;               // F16EMU with offset: extra k-steps of the offset term (else 0)
  long long nTiles;
  int mTiles;                // row blocks (TM rows each)
  float eps;
  uint32_t so_bytes;         // F16EMU: bytes of one scale/offset row box (rows x 256 x 4)
  long long budget;          // cycles a row-block wait lasts before it gives up
  uint32_t extra;            // arrivals a row-block wait needs beyond its own (0; > 0 only in tests)
};

// Tile t -> (row block rb, n-tile nt). Row blocks go in pairs: within a pair
// the tiles alternate between its two row blocks at the same n-tile, so the
// two CTAs that run tiles 2i and 2i+1 side by side read one weight tile and
// the second read hits L2 (the whole INT4 weight nearly fills L2 by itself, so
// a row-block-major order re-reads most of it from DRAM for every row block).
// A last unpaired row block runs its n-tiles in order. The tiles of one row
// block lie within 2 * nTilesN consecutive indices, so with nTilesN <= grid a
// CTA that has published its current tile only ever waits for a row block
// whose tiles precede its own next tile, which keeps the waits deadlock-free.
__device__ __forceinline__ void tile_coords(const PrefillArgs &a, long long t, int &rb, int &nt) {
  const long long span = 2LL * a.nTilesN;
  const long long pair = t / span, r = t - pair * span;
  const int rb0 = (int)(2 * pair);
  if (rb0 + 1 < a.mTiles) {
    rb = rb0 + (int)(r & 1);
    nt = (int)(r >> 1);
  } else {
    rb = rb0;
    nt = (int)r;
  }
}

template <int WBITS, int MH, int MODE>
struct Layout {
  static_assert(MH == 1 || (MH == 2 && WBITS == 4), "256-row tiles with INT4 weights only");
  static constexpr int NR = Stages<WBITS, MH, MODE>::NR, NB = Stages<WBITS, MH, MODE>::NB;
  static constexpr uint32_t A_HALF = BM * BK * 2;             // 16 KB: one 128-row half
  static constexpr uint32_t A_BYTES = MH * A_HALF;
  static constexpr uint32_t BQ_BYTES = BK * BN * WBITS / 8;   // 8 or 16 KB
  static constexpr uint32_t B_BYTES = BN * BK * 2;            // 32 KB
  // F16EMU: rows of S16 pairs (3 KB); RAWQ reads scales in the epilogue
  static constexpr uint32_t SO_BYTES = MODE == kF16Emu ? SO_ROWS * BN * 4 : 0;
  // epilogue boxes of 32 rows x 32 columns (64-byte rows, 64-byte swizzle): per
  // epilogue warp three residual boxes and one y box
  static constexpr uint32_t EPI_BOX = 32 * 64;
  static constexpr int NRES = 3;
  static constexpr uint32_t A_OFF = 0;
  static constexpr uint32_t BQ_OFF = A_OFF + NR * A_BYTES;
  static constexpr uint32_t B_OFF = BQ_OFF + NR * BQ_BYTES;
  static constexpr uint32_t EPI_OFF = B_OFF + NB * B_BYTES;   // 1024-byte aligned
  static constexpr uint32_t S_OFF = EPI_OFF + (NRES + 1) * 4 * EPI_BOX;
  static constexpr uint32_t BAR_OFF = S_OFF + NR * SO_BYTES;
  static constexpr int NBARS = 2 * NR + 2 * NB + 4 + 1 + 4 * NRES;
  static constexpr uint32_t SMEM = BAR_OFF + 8 * NBARS + 16 + 1024;
  static_assert(SMEM <= 232448, "shared memory per CTA");
};

// barrier indices (NR, NB are the kernel's stage counts)
#define FULL(s) (s)
#define RAWEMPTY(s) (NR + (s))
#define BFULL(s) (2 * NR + (s))
#define BEMPTY(s) (2 * NR + NB + (s))
#define ACCFULL(b) (2 * NR + 2 * NB + (b))
#define ACCEMPTY(b) (2 * NR + 2 * NB + 2 + (b))
#define DRAIN() (2 * NR + 2 * NB + 4)
#define RESFULL(q, b) (2 * NR + 2 * NB + 5 + 3 * (q) + (b))

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
               : "memory");
}

__device__ __forceinline__ uint32_t ld_shared_u32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}

// Packed fp16 pair arithmetic: (v - c) * s, exact here (small integers times
// a scale whose product fits the fp16 significand) or rounded once (INT8).
__device__ __forceinline__ uint32_t sub_mul2_f16(uint32_t v, uint32_t c, uint32_t s) {
  uint32_t r;
  asm("{\n\t.reg .b32 t;\n\t"
      "sub.rn.f16x2 t, %1, %2;\n\t"
      "mul.rn.f16x2 %0, t, %3;\n\t}"
      : "=r"(r)
      : "r"(v), "r"(c), "r"(s));
  return r;
}

// Reads the S16 pairs (both halves hold the value) of CNT columns in group
// row `row` of the stage's scale rows: four columns per 16-byte chunk, chunk q
// at word w + QSTRIDE * q of the row. Rows past the last group were zero-filled
// by the copy (callers skip k-rows past K, whose rows may be stale).
template <int CNT, int QSTRIDE>
__device__ __forceinline__ void smem_s(uint32_t s_base, int row, int w, uint32_t (&s2)[CNT]) {
  const uint32_t off = (uint32_t)(row * BN + w) * 4u;
#pragma unroll
  for (int q = 0; q < CNT / 4; ++q)
    asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(s2[4 * q]), "=r"(s2[4 * q + 1]), "=r"(s2[4 * q + 2]), "=r"(s2[4 * q + 3])
                 : "r"(s_base + off + 4u * QSTRIDE * q));
}

// Byte offset of the 16-byte chunk (row r, k-octet c) in a K-major 128-byte
// swizzled tile with 64 elements per row.
__device__ __forceinline__ uint32_t sw128_chunk(int r, int c) {
  return (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4));
}

template <int DT, int WBITS, int MODE, int MH>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w,
                   const __grid_constant__ CUtensorMap tm_s, const __grid_constant__ CUtensorMap tm_dx,
                   const __grid_constant__ CUtensorMap tm_ox, const __grid_constant__ CUtensorMap tm_r,
                   const PrefillArgs a) {
  using L = Layout<WBITS, MH, MODE>;
  constexpr int NACC = 2 / MH;   // accumulator buffers of MH x 256 TMEM columns
  constexpr int TM = BM * MH;    // output rows per tile
  using E = Elem<DT>;
  using T = typename E::T;
  constexpr int MDT = MODE == kF16Emu ? WQ_F16 : DT;  // operand dtype of the MMA
  constexpr int NR = L::NR, NB = L::NB;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  auto BAR = [&](int i) -> uint32_t { return sbase + L::BAR_OFF + 8u * i; };
  uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + L::BAR_OFF + 8 * L::NBARS);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_holder + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NR; ++s) {
      mbar_init(BAR(FULL(s)), 1);
      mbar_init(BAR(RAWEMPTY(s)), kDqWarps + 1);
    }
    for (int s = 0; s < NB; ++s) {
      mbar_init(BAR(BFULL(s)), kDqWarps);
      mbar_init(BAR(BEMPTY(s)), 1);
    }
    for (int b = 0; b < NACC; ++b) {
      mbar_init(BAR(ACCFULL(b)), 1);
      mbar_init(BAR(ACCEMPTY(b)), kEpiWarps);
    }
    mbar_init(BAR(DRAIN()), 1);
    for (int q = 0; q < 4; ++q)
      for (int b = 0; b < L::NRES; ++b) mbar_init(BAR(RESFULL(q, b)), 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tm_x);
    prefetch_tmap(&tm_w);
    prefetch_tmap(&tm_r);
    if (MODE == kF16Emu) {
      prefetch_tmap(&tm_s);
      if (a.kTilesX) {
        prefetch_tmap(&tm_dx);
        prefetch_tmap(&tm_ox);
      }
    }
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_holder), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA producer
    // packed weights are re-read by every row block: keep them in L2
    const uint64_t pol_w = policy_evict_last();
    long long it = 0;
    const int kAll = a.kTiles + a.kTilesX;
    for (long long t = blockIdx.x; t < a.nTiles; t += gridDim.x) {
      int rb, nt;
      tile_coords(a, t, rb, nt);
      for (int ks = 0; ks < kAll; ++ks, ++it) {
        const int s = (int)(it % NR);
        const uint32_t ph = (uint32_t)((it / NR) & 1);
        if (!wait_bar_warp(BAR(RAWEMPTY(s)), ph ^ 1u, abort_flag, a.status, kWhereProducer)) goto pdone;
        if (MODE == kF16Emu && ks >= a.kTiles) {
          // offset-term k-step: A = row sums of the groups (bf16 parts), B = the
          // offsets, both straight into the MMA's operand layout; the B slot is
          // this stage's, once the MMA has released it
          const int sb = (int)(it % NB);
          if (!wait_bar_warp(BAR(BEMPTY(sb)), (uint32_t)(((it / NB) & 1) ^ 1), abort_flag, a.status,
                             kWhereProducer))
            goto pdone;
          if (lane == 0) {
            const int kx = (ks - a.kTiles) * BK;
            mbar_arrive_expect_tx(BAR(FULL(s)), L::A_BYTES + L::B_BYTES);
            tma_load_2d(sbase + L::A_OFF + s * L::A_BYTES, &tm_dx, kx, rb * TM, BAR(FULL(s)));
            tma_load_2d(sbase + L::B_OFF + sb * L::B_BYTES, &tm_ox, kx, nt * BN, BAR(FULL(s)));
          }
          __syncwarp();
          continue;
        }
        if (lane == 0) {
          uint32_t bytes = L::A_BYTES + L::BQ_BYTES;
          if (MODE == kF16Emu) bytes += a.so_bytes;
          mbar_arrive_expect_tx(BAR(FULL(s)), bytes);
          tma_load_2d(sbase + L::A_OFF + s * L::A_BYTES, &tm_x, ks * BK, rb * TM, BAR(FULL(s)));
          tma_load_2d_hint(sbase + L::BQ_OFF + s * L::BQ_BYTES, &tm_w, nt * (BN * WBITS / 8),
                           ks * BK, BAR(FULL(s)), pol_w);
          if (MODE == kF16Emu) {
            // the group rows this k-stage touches: (ks*BK)/group .. +SO_ROWS-1
            const int r0 = (ks * BK) / a.group;
            tma_load_2d(sbase + L::S_OFF + s * L::SO_BYTES, &tm_s, nt * BN, r0, BAR(FULL(s)));
          }
        }
        __syncwarp();
      }
    }
  pdone:
    // every copy this warp issued has landed before the CTA may exit
    for (long long j = (it > NR ? it - NR : 0); j < it; ++j)
      drain_bar(BAR(FULL((int)(j % NR))), (uint32_t)((j / NR) & 1));
    __syncwarp();
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    {
      const uint32_t idesc = idesc_f16(MDT == WQ_BF16 ? 1u : 0u, BM, BN);
      const uint32_t idesc_x = idesc_f16(1u, BM, BN);  // offset-term k-steps: bf16 x bf16
      const int kAll = a.kTiles + a.kTilesX;
      long long it = 0;
      int lt = 0;
      for (long long t = blockIdx.x; t < a.nTiles; t += gridDim.x, ++lt) {
        const int buf = lt % NACC;
        if (!wait_bar_warp(BAR(ACCEMPTY(buf)), (uint32_t)(((lt / NACC) & 1) ^ 1), abort_flag,
                           a.status, kWhereMma))
          goto mdone;
        tc_fence_after();
        const uint32_t d = tmem_base + (uint32_t)(buf * BN);  // half h at + h * BN
        for (int ks = 0; ks < kAll; ++ks, ++it) {
          const int s = (int)(it % NR), sb = (int)(it % NB);
          const bool xstep = ks >= a.kTiles;  // offset-term step: both operands came by TMA
          if (!wait_bar_warp(BAR(FULL(s)), (uint32_t)((it / NR) & 1), abort_flag, a.status, kWhereMma))
            goto mdone;
          if (!wait_bar_warp(BAR(BFULL(sb)), (uint32_t)((it / NB) & 1), abort_flag, a.status,
                             kWhereMma))
            goto mdone;
          tc_fence_after();
          if (lane == 0) {
            const uint32_t aaddr = sbase + L::A_OFF + s * L::A_BYTES;
            const uint32_t baddr = sbase + L::B_OFF + sb * L::B_BYTES;
            const uint32_t id = xstep ? idesc_x : idesc;
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk)
#pragma unroll
              for (int h = 0; h < MH; ++h)
                mma_f16(d + (uint32_t)(h * BN), desc_kmajor_sw128(aaddr + h * L::A_HALF + kk * 32),
                        desc_kmajor_sw128(baddr + kk * 32), id, (ks | kk) != 0 ? 1u : 0u);
            mma_commit(BAR(BEMPTY(sb)));
            mma_commit(BAR(RAWEMPTY(s)));
          }
          __syncwarp();
        }
        if (lane == 0) mma_commit(BAR(ACCFULL(buf)));
        __syncwarp();
      }
    mdone:
      if (lane == 0) mma_commit(BAR(DRAIN()));
      __syncwarp();
      drain_bar(BAR(DRAIN()), 0);
      __syncwarp();
    }
  } else if (warp >= kDqWarp0 && warp < kDqWarp0 + kDqWarps) {
    // ---------------------------------------------------------------- dequant
    // Each thread owns one k-octet (8 k-rows) of 8 (INT4) or 2 x 4 (INT8)
    // consecutive columns per stage. The k-octet is rotated by lane so that
    // both the packed-word loads and the 16-byte swizzled stores are free of
    // shared-memory bank conflicts.
    const int dw = warp - kDqWarp0;
    const int ko = (dw + lane) & 7;
    // INT4: this thread's eight swizzled 16-byte stores of a B stage (row 8*lane + j, chunk ko)
    uint32_t sto[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) sto[j] = sw128_chunk(8 * lane + j, ko);
    // INT4: nibble r, u = r ^ 8 = q + 8, and (magic | u) is the 16-bit float
    // 128 + u (bf16) or 1024 + u (fp16); subtracting `magic` gives q exactly.
    const uint32_t magic4 = MDT == WQ_BF16 ? 0x43084308u : 0x64086408u;
    long long it = 0;
    const int kAll = a.kTiles + a.kTilesX;
    for (long long t = blockIdx.x; t < a.nTiles; t += gridDim.x) {
      // (ks * BK) % group, kept without a division; the stage's first group row
      // is (ks * BK) / group, and this thread's k-octet lies in that row or the
      // next ones: srow = (kmod + 8 ko) / group, at most 2 (group >= 32)
      int kmod = 0;
      for (int ks = 0; ks < kAll; ++ks, ++it, kmod += BK) {
        while (kmod >= a.group && a.group > 0) kmod -= a.group;
        const int s = (int)(it % NR), sb = (int)(it % NB);
        const int k = ks * BK + 8 * ko;
        const int kk8 = kmod + 8 * ko;
        const int srow = kk8 < a.group ? 0 : (kk8 < 2 * a.group ? 1 : 2);
        if (ks >= a.kTiles) {
          // offset-term step: no weight to dequantize (the producer copied both
          // operands). The warps still arrive on the raw slot's and the B slot's
          // barriers, so that every barrier completes exactly once per step and
          // the parity waits of later steps stay in step. They arrive only after
          // the copies landed: the producer issued them after the B slot's
          // previous use was released, so no arrival counts towards that use.
          if (!wait_bar_warp(BAR(FULL(s)), (uint32_t)((it / NR) & 1), abort_flag, a.status,
                             kWhereDequant))
            goto ddone;
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(BAR(RAWEMPTY(s)));
            mbar_arrive(BAR(BFULL(sb)));
          }
          continue;
        }
        const uint32_t bq = sbase + L::BQ_OFF + s * L::BQ_BYTES;
        const uint32_t bst = sbase + L::B_OFF + sb * L::B_BYTES;
        if constexpr (WBITS == 4) {
          uint32_t s2[8];
          if (!wait_bar_warp(BAR(FULL(s)), (uint32_t)((it / NR) & 1), abort_flag, a.status,
                             kWhereDequant))
            goto ddone;
          if (!wait_bar_warp(BAR(BEMPTY(sb)), (uint32_t)(((it / NB) & 1) ^ 1), abort_flag, a.status,
                             kWhereDequant))
            goto ddone;
          if constexpr (MODE == kF16Emu) {
            if (k < a.K) {
              // columns 8 lane .. 8 lane + 7, stored as words 4 lane .. and 128 + 4 lane ..
              smem_s<8, 128>(sbase + L::S_OFF + s * L::SO_BYTES, srow, 4 * lane, s2);
            } else {
#pragma unroll
              for (int j = 0; j < 8; ++j) s2[j] = 0u;
            }
          }
          uint32_t wr[8], wsh[8];
#pragma unroll
          for (int tt = 0; tt < 8; ++tt) wr[tt] = ld_shared_u32(bq + (8 * ko + tt) * 128 + 4 * lane);
          __syncwarp();
          if (lane == 0) mbar_arrive(BAR(RAWEMPTY(s)));
          if constexpr (MODE != kF16Emu) {
#pragma unroll
            for (int tt = 0; tt < 8; ++tt) wsh[tt] = wr[tt] >> 4;
          }
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const uint32_t b = (uint32_t)(j >> 1);
            const uint32_t sel = b | ((b + 4u) << 8);
            uint32_t c[4];
#pragma unroll
            for (int p = 0; p < 4; ++p) {
              if constexpr (MODE == kF16Emu) {
                // fp16 operands: an odd column's nibble is used in place at bits
                // 7:4, as 1152 + 16 q; its S16 was stored divided by 16
                const uint32_t x = __byte_perm(wr[2 * p], wr[2 * p + 1], sel);
                const uint32_t mg = (j & 1) ? 0x64806480u : magic4;
                const uint32_t v = (x & ((j & 1) ? 0x00F000F0u : 0x000F000Fu)) ^ mg;
                c[p] = sub_mul2_f16(v, mg, s2[j]);
              } else {
                const uint32_t x = (j & 1) ? __byte_perm(wsh[2 * p], wsh[2 * p + 1], sel)
                                           : __byte_perm(wr[2 * p], wr[2 * p + 1], sel);
                const uint32_t v = (x & 0x000F000Fu) ^ magic4;
                c[p] = sub2<MDT>(v, magic4);
              }
            }
            st_shared_v4(bst + sto[j], c[0], c[1], c[2], c[3]);
          }
        } else {
          uint32_t s2a[4], s2b[4];
          if (!wait_bar_warp(BAR(FULL(s)), (uint32_t)((it / NR) & 1), abort_flag, a.status,
                             kWhereDequant))
            goto ddone;
          if (!wait_bar_warp(BAR(BEMPTY(sb)), (uint32_t)(((it / NB) & 1) ^ 1), abort_flag, a.status,
                             kWhereDequant))
            goto ddone;
          if constexpr (MODE == kF16Emu) {
            if (k < a.K) {
              const int rr = srow;
              const uint32_t sa = sbase + L::S_OFF + s * L::SO_BYTES;
              smem_s<4, 4>(sa, rr, 4 * lane, s2a);
              smem_s<4, 4>(sa, rr, 4 * (lane + 32), s2b);
            } else {
#pragma unroll
              for (int j = 0; j < 4; ++j) s2a[j] = s2b[j] = 0u;
            }
          }
          uint32_t wa[8], wb[8];
#pragma unroll
          for (int tt = 0; tt < 8; ++tt) {
            wa[tt] = ld_shared_u32(bq + (8 * ko + tt) * 256 + 4 * lane);
            wb[tt] = ld_shared_u32(bq + (8 * ko + tt) * 256 + 4 * (lane + 32));
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(BAR(RAWEMPTY(s)));
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            const uint32_t *w = half ? wb : wa;
            const int nq = lane + 32 * half;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const uint32_t sel = (uint32_t)j | ((uint32_t)(j + 4) << 8);
              uint32_t c[4];
#pragma unroll
              for (int p = 0; p < 4; ++p) {
                const uint32_t x = __byte_perm(w[2 * p], w[2 * p + 1], sel);
                if constexpr (MDT == WQ_F16) {
                  // byte b, (b ^ 0x80) | 0x6400 is the fp16 value 1152 + q
                  const uint32_t v = (x & 0x00FF00FFu) ^ 0x64806480u;
                  if constexpr (MODE == kF16Emu)
                    c[p] = sub_mul2_f16(v, 0x64806480u, half ? s2b[j] : s2a[j]);
                  else
                    c[p] = sub2<WQ_F16>(v, 0x64806480u);
                } else {
                  // bf16 operand, raw q: |q| <= 128 is exact in bf16
                  c[p] = pack2<WQ_BF16>((float)(int8_t)(x & 0xFFu), (float)(int8_t)((x >> 16) & 0xFFu));
                }
              }
              st_shared_v4(bst + sw128_chunk(4 * nq + j, ko), c[0], c[1], c[2], c[3]);
            }
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(BAR(BFULL(sb)));
      }
    }
  ddone:;
  } else if (warp >= kEpiWarp0) {
    // ---------------------------------------------------------------- epilogue
    // Thread = TMEM lane = output row. Global traffic goes through 32 x 32
    // boxes in shared memory (64-byte rows, 64-byte swizzle: 16-byte chunk j of
    // row r sits at r*64 + ((j ^ ((r >> 1) & 3)) << 4), so a row read or
    // written by its thread is free of bank conflicts): the TMA loads the
    // residual boxes two ahead of their use, and each y box, written a row per
    // thread, leaves as coalesced 16-byte stores of whole box rows.
    const int qd = warp & 3;  // TMEM lane quarter
    const int rit = 32 * qd + lane;
    const T *bias = static_cast<const T *>(a.bias);
    const T *gam = static_cast<const T *>(a.gamma);
    const T *yout = static_cast<const T *>(a.y);
    T *nout = static_cast<T *>(a.normOut);
    const uint32_t lane_addr = tmem_base + ((uint32_t)(32 * qd) << 16);
    constexpr int NRES = L::NRES;
    const uint32_t rbox = sbase + L::EPI_OFF + (uint32_t)qd * (NRES + 1) * L::EPI_BOX;
    const uint32_t ybox = rbox + (uint32_t)NRES * L::EPI_BOX;
    const uint32_t row_off = (uint32_t)lane * 64u;
    const uint32_t swz = (uint32_t)((lane >> 1) & 3);
    T *yst = static_cast<T *>(a.y);
    uint32_t rc = 0;      // residual boxes used so far: box rc % NRES, phase (rc / NRES) & 1
    uint32_t issued = 0;  // residual box loads issued (those in [rc, issued) are in flight)
    int lt = 0;
    long long prev_t = -1;
    bool ok = true;

    // Normalises the previous tile's rows: warp = row (32 lanes x 8 columns
    // cover a 256-column tile row with 16-byte accesses), rows of this warp's
    // lane quarter only, whose y this warp stored.
    auto normalize = [&](long long t) -> bool {
      int rb, nt;
      tile_coords(a, t, rb, nt);
      // wait until every n-tile of this row block published its partial sums
      {
        const uint32_t target = (uint32_t)(kEpiWarps * a.nTilesN) + a.extra;
        bool done = false;
        if (lane == 0) {
          const long long t0 = clock64();
          while (true) {
            done = ld_acquire_u32(a.counters + rb) >= target;
            if (done || *abort_flag) break;
            if (clock64() - t0 > a.budget) {
              *abort_flag = 1;
              record_timeout(a.status, kWhereRowBlock);
              break;
            }
            __nanosleep(64);
          }
        }
        done = __shfl_sync(0xffffffffu, done, 0);
        __syncwarp();  // the lanes' reads below come after lane 0's acquire
        if (!done) return false;
      }
      const int n = nt * BN + 8 * lane;
      const bool col_ok = n < a.N;  // N % 16 == 0 keeps every 8-column group whole
      uint4 g = make_uint4(0u, 0u, 0u, 0u);
      if (col_ok) g = *reinterpret_cast<const uint4 *>(gam + n);
      const uint32_t gw[4] = {g.x, g.y, g.z, g.w};
      const int nparts = a.nTilesN;
#pragma unroll 1
      for (int h = 0; h < MH; ++h) {
        const long long mbase = (long long)rb * TM + h * BM + 32 * qd;
#pragma unroll 1
        for (int r0 = 0; r0 < 32; r0 += 4) {
          float tot[4];
          uint4 yv[4];
          // all loads of the four rows first (kPartsPerLane partial sums per
          // lane cover the row's n-tiles), then the sums
          float pv[4][kPartsPerLane];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const long long m = mbase + r0 + u;
            yv[u] = make_uint4(0u, 0u, 0u, 0u);
            const bool live = m < a.M;
            const float *rp = a.rowpart + m * nparts;
#pragma unroll
            for (int i = 0; i < kPartsPerLane; ++i) {
              const int j = lane + 32 * i;
              pv[u][i] = live && j < nparts ? __ldcg(rp + j) : 0.f;
            }
            if (live && col_ok) yv[u] = __ldcg(reinterpret_cast<const uint4 *>(yout + m * a.N + n));
          }
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            tot[u] = 0.f;
#pragma unroll
            for (int i = 0; i < kPartsPerLane; ++i) tot[u] += pv[u][i];
          }
#pragma unroll
          for (int u = 0; u < 4; ++u) {
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) tot[u] += __shfl_xor_sync(0xffffffffu, tot[u], o);
            const long long m = mbase + r0 + u;
            if (m < a.M && col_ok) {
              const float rstd = rsqrtf(tot[u] / (float)a.N + a.eps);
              const uint32_t yw[4] = {yv[u].x, yv[u].y, yv[u].z, yv[u].w};
              uint32_t o4[4];
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const float2 y2 = unpack2<DT>(yw[i]), g2 = unpack2<DT>(gw[i]);
                o4[i] = pack2<DT>(y2.x * rstd * g2.x, y2.y * rstd * g2.y);
              }
              *reinterpret_cast<uint4 *>(nout + m * a.N + n) = make_uint4(o4[0], o4[1], o4[2], o4[3]);
            }
          }
        }
      }
      return true;
    };

    // Pulls this warp's residual rows of tile t into L2 (lane = row), a whole
    // main loop before the y pass's boxes read them.
    auto prefetch_residual = [&](long long t) {
      if (t >= a.nTiles) return;
      int rb, nt;
      tile_coords(a, t, rb, nt);
      const int n0 = nt * BN;
      const T *res = static_cast<const T *>(a.residual);
#pragma unroll
      for (int h = 0; h < MH; ++h) {
        const long long m = (long long)rb * TM + h * BM + rit;
        if (m >= a.M) break;
        const char *rowp = reinterpret_cast<const char *>(res + m * a.N + n0);
        const int bytes = (n0 + BN < a.N ? BN : a.N - n0) * (int)sizeof(T);
        for (int b = 0; b < bytes; b += 128)
          asm volatile("prefetch.global.L2 [%0];" ::"l"(rowp + b));
      }
    };
    // lane 0: load residual box k (32 rows from m0, 32 columns from n) into box k % NRES
    auto load_residual = [&](uint32_t k, int n, long long m0) {
      issued = k + 1;
      if (lane == 0) {
        fence_proxy_async_smem();  // the lanes' earlier reads of this box come first
        const uint32_t bar = BAR(RESFULL(qd, (int)(k % NRES)));
        mbar_arrive_expect_tx(bar, L::EPI_BOX);
        tma_load_2d(rbox + (k % NRES) * L::EPI_BOX, &tm_r, n, (int)m0, bar);
      }
    };
    constexpr int CPH = BN / 32;  // 32-column chunks per tile row
    prefetch_residual(blockIdx.x);
    for (long long t = blockIdx.x; t < a.nTiles && ok; t += gridDim.x, ++lt) {
      const int buf = lt % NACC;
      int rb, nt;
      tile_coords(a, t, rb, nt);
      const int n0 = nt * BN;
      // this tile's per-column parameters, 8 columns a lane (lane l holds
      // columns n0 + 8l ..), handed to the lanes that need them by shuffles
      uint4 cb = make_uint4(0u, 0u, 0u, 0u), cs = cb, co = cb;  // bias, scale or e_col, offset
      {
        const int nl = n0 + 8 * lane;
        if (nl < a.N) {
          if (bias) cb = *reinterpret_cast<const uint4 *>(bias + nl);
          if constexpr (MODE == kRawQ) {
            if (a.Ns != 1) {
              cs = *reinterpret_cast<const uint4 *>(static_cast<const T *>(a.scale) + nl);
              if (a.offset) co = *reinterpret_cast<const uint4 *>(static_cast<const T *>(a.offset) + nl);
            }
          } else {
            cs = *reinterpret_cast<const uint4 *>(a.e_col + nl);
          }
        }
      }
      // boxes of this tile inside the output: nch column boxes for each half
      // whose 32 rows of this warp start before M
      const int nch = (a.N - n0 + 31) / 32 < CPH ? (a.N - n0 + 31) / 32 : CPH;
      auto half_live = [&](int h) { return (long long)rb * TM + h * BM + 32 * qd < a.M; };
      int nlive = 0;
      while (nlive < MH && half_live(nlive)) ++nlive;
      const int nbox = nlive * nch;  // this warp's boxes of the tile, half-major
      const uint32_t rc0 = rc;
      // box i of the tile: half i / nch, columns n0 + 32 (i % nch)
      auto load_box = [&](int i) {
        if (i < nbox)
          load_residual(rc0 + (uint32_t)i, n0 + 32 * (i % nch),
                        (long long)rb * TM + (i / nch) * BM + 32 * qd);
      };
      load_box(0);
      load_box(1);
      if (!wait_bar_warp(BAR(ACCFULL(buf)), (uint32_t)((lt / NACC) & 1), abort_flag, a.status,
                         kWhereEpiAcc)) {
        ok = false;
        break;
      }
      tc_fence_after();
#pragma unroll 1
      for (int h = 0; h < nlive && ok; ++h) {
        const long long mrow0 = (long long)rb * TM + h * BM + 32 * qd;  // the warp's first row
        const long long m = mrow0 + lane;
        const bool row_ok = m < a.M;
        const uint32_t taddr = lane_addr + (uint32_t)((buf + h) * BN);
        float ss = 0.f;
        // per-row factor of this thread's row
        float rs = 0.f;   // RAWQ + offset: sum_k x1[m, k]
        int em = 0;       // F16EMU: row exponent
        if (row_ok) {
          if constexpr (MODE == kRawQ) {
            if (a.offset) rs = a.rowsum[m];
          } else {
            em = a.e_row[m];
          }
        }
#pragma unroll 1
        for (int c = 0; c < nch; ++c, ++rc) {
          load_box(h * nch + c + 2);  // two boxes ahead
          uint32_t r[32];
          tmem_ld32(taddr + 32 * c, r);
          tmem_wait_ld();
          if (!wait_bar_warp(BAR(RESFULL(qd, (int)(rc % NRES))), (rc / NRES) & 1u, abort_flag,
                             a.status, kWhereEpiAcc)) {
            ok = false;
            break;
          }
          const uint32_t rb_addr = rbox + (rc % NRES) * L::EPI_BOX + row_off;
          uint32_t yo[16];
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            const int n = n0 + 32 * c + 8 * v;
            // mm = the operator's x1 @ W for these 8 columns (held by lane g)
            const int g = 4 * c + v;
            auto bcast = [&](uint4 q, uint32_t (&w)[4]) {
              w[0] = __shfl_sync(0xffffffffu, q.x, g);
              w[1] = __shfl_sync(0xffffffffu, q.y, g);
              w[2] = __shfl_sync(0xffffffffu, q.z, g);
              w[3] = __shfl_sync(0xffffffffu, q.w, g);
            };
            uint32_t bw[4], cw[4];
            bcast(cb, bw);
            bcast(cs, cw);
            float mmv[8];
            if (n < a.N) {
              if constexpr (MODE == kRawQ) {
                uint32_t sw[4], ow[4] = {0u, 0u, 0u, 0u};
                if (a.Ns == 1) {
                  const uint32_t sb = *reinterpret_cast<const uint16_t *>(a.scale);
                  sw[0] = sw[1] = sw[2] = sw[3] = sb | (sb << 16);
                  if (a.offset) {
                    const uint32_t ob = *reinterpret_cast<const uint16_t *>(a.offset);
                    ow[0] = ow[1] = ow[2] = ow[3] = ob | (ob << 16);
                  }
                } else {
                  sw[0] = cw[0]; sw[1] = cw[1]; sw[2] = cw[2]; sw[3] = cw[3];
                  if (a.offset) bcast(co, ow);
                }
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                  const float2 s2 = unpack2<DT>(sw[i]);
                  const float2 o2 = unpack2<DT>(ow[i]);
                  mmv[2 * i] = fmaf(s2.x, __uint_as_float(r[8 * v + 2 * i]), o2.x * rs);
                  mmv[2 * i + 1] = fmaf(s2.y, __uint_as_float(r[8 * v + 2 * i + 1]), o2.y * rs);
                }
              } else {
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                  const int en = (int)(int16_t)((cw[i >> 1] >> (16 * (i & 1))) & 0xFFFFu);
                  mmv[i] = scale_pow2(__uint_as_float(r[8 * v + i]), em + en);
                }
              }
            } else {
#pragma unroll
              for (int i = 0; i < 8; ++i) mmv[i] = 0.f;
            }
            uint32_t rw[4];
            asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                         : "=r"(rw[0]), "=r"(rw[1]), "=r"(rw[2]), "=r"(rw[3])
                         : "r"(rb_addr + ((((uint32_t)v) ^ swz) << 4)));
            float yv[8];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const float2 b2 = unpack2<DT>(bw[i]);
              const float2 r2 = unpack2<DT>(rw[i]);
              yv[2 * i] = mmv[2 * i] + b2.x + r2.x;
              yv[2 * i + 1] = mmv[2 * i + 1] + b2.y + r2.y;
              yo[4 * v + i] = pack2<DT>(yv[2 * i], yv[2 * i + 1]);
            }
            if (row_ok && n < a.N) {
#pragma unroll
              for (int i = 0; i < 8; ++i) ss = fmaf(yv[i], yv[i], ss);
            }
          }
          // the y box: every lane has read the previous one; write this thread's
          // row, then store whole box rows (lanes 4i..4i+3 cover row 8u + i)
          __syncwarp();
#pragma unroll
          for (int v = 0; v < 4; ++v)
            st_shared_v4(ybox + row_off + ((((uint32_t)v) ^ swz) << 4), yo[4 * v], yo[4 * v + 1],
                         yo[4 * v + 2], yo[4 * v + 3]);
          __syncwarp();
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int rr = 8 * u + (lane >> 2), j = lane & 3;
            const long long my = mrow0 + rr;
            const int ny = n0 + 32 * c + 8 * j;
            uint32_t q0, q1, q2, q3;
            asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                         : "=r"(q0), "=r"(q1), "=r"(q2), "=r"(q3)
                         : "r"(ybox + (uint32_t)rr * 64u +
                               ((((uint32_t)j) ^ (((uint32_t)rr >> 1) & 3u)) << 4)));
            if (my < a.M && ny < a.N)
              *reinterpret_cast<uint4 *>(yst + my * a.N + ny) = make_uint4(q0, q1, q2, q3);
          }
        }
        if (row_ok && ok) a.rowpart[m * a.nTilesN + nt] = ss;
      }  // halves
      if (!ok) break;
      // the accumulator has been read: hand it back to the MMA issuer
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(BAR(ACCEMPTY(buf)));
      // each epilogue warp publishes its 32 rows; the row block is complete
      // when all kEpiWarps warps of all n-tiles have published
      __syncwarp();
      if (lane == 0) {
        __threadfence();
        red_release_add(a.counters + rb, 1u);
      }
      __syncwarp();
      prefetch_residual(t + gridDim.x);
      if (prev_t >= 0) {
        if (!normalize(prev_t)) {
          ok = false;
          break;
        }
      }
      prev_t = t;
    }
    if (lane == 0) {
      // no copy of this warp may still be in flight when the CTA exits
      for (uint32_t k = rc; k < issued; ++k)
        drain_bar(BAR(RESFULL(qd, (int)(k % NRES))), (k / NRES) & 1u);
    }
    __syncwarp();
    if (ok && prev_t >= 0) normalize(prev_t);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

// ------------------------------------------------------------------ host side

using EncodeTiledFn = PFN_cuTensorMapEncodeTiled_v12000;

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
    else
      cudaGetLastError();
  });
  return fn;
}

bool aligned16(const void *p) { return p == nullptr || (reinterpret_cast<uintptr_t>(p) % 16) == 0; }

}  // namespace

static uint64_t align256(uint64_t v) { return (v + 255) / 256 * 256; }

// Words per S16/O16 row: INT4 rows are padded to whole n-tiles (their columns
// are stored in the dequant's interleaved order, see so_prep_kernel).
static int64_t so_ld(const Problem &p, const Plan &plan) {
  return p.wbits == 4 ? plan.n_tiles * BN : p.N;
}

bool prefill_applicable(const Problem &p) {
  if (p.M < 1 || p.N < 1) return false;
  if (p.K % 8 != 0) return false;                       // x1 row stride: 16-byte multiple for TMA
  if (p.wbits == 4 ? (p.N % 32 != 0) : (p.N % 16 != 0)) return false;  // packed row stride
  // fp16 activations with per-group scales have no exact single-operand form
  // (an 11-bit fp16 scale times q needs more than 11 bits): other kernels.
  if (p.smode == kPerGroup && p.dtype == WQ_F16) return false;
  const void *ptrs[] = {p.x1, p.x2, p.scale, p.offset, p.bias, p.residual, p.gamma, p.y, p.normOut};
  for (const void *q : ptrs)
    if (!aligned16(q)) return false;
  const int64_t nTilesN = (p.N + BN - 1) / BN;
  if (nTilesN > device_info().sms) return false;        // row-block waits need n-tiles <= CTAs
  if (nTilesN > 32 * kPartsPerLane) return false;       // partial sums a normalising warp reads
  return true;
}

bool plan_prefill(const Problem &p, Plan &plan) {
  if (!prefill_applicable(p)) return false;
  plan.kernel = WQ_KERNEL_PREFILL;
  plan.mode = p.smode == kPerGroup ? kF16Emu : kRawQ;
  plan.n_tiles = (p.N + BN - 1) / BN;
  // 256-row tiles (INT4): one dequantized weight tile feeds two MMAs, which
  // makes a row cost about kHalvesCost of a 128-row tile's; taken when that
  // outweighs the coarser last wave of tiles over the SMs.
  const int64_t sms = device_info().sms;
  auto waves = [&](int64_t rows) {
    const int64_t tiles = plan.n_tiles * ((p.M + rows - 1) / rows);
    return (tiles + sms - 1) / sms;
  };
  constexpr double kHalvesCost = 0.75;
  plan.m_halves = (p.wbits == 4 && p.M > BM &&
                   (double)waves(2 * BM) * 2.0 * kHalvesCost < (double)waves(BM))
                      ? 2
                      : 1;
  plan.m_tiles = (p.M + BM * plan.m_halves - 1) / (BM * plan.m_halves);
  const int64_t tiles = plan.n_tiles * plan.m_tiles;
  plan.grid = (int)(tiles < sms ? tiles : sms);
  uint64_t off = kWsHeader;
  plan.cnt_off = off;
  off += align256((uint64_t)plan.m_tiles * 4);
  plan.rowpart_off = off;
  off += align256((uint64_t)p.M * (uint64_t)plan.n_tiles * sizeof(float));
  if (plan.mode == kRawQ) {
    if (p.offset) {
      plan.rowsum_off = off;
      off += align256((uint64_t)p.M * sizeof(float));
    }
  } else {
    plan.erow_off = off;
    off += align256((uint64_t)p.M * sizeof(int16_t));
    plan.ecol_off = off;
    off += align256((uint64_t)p.N * sizeof(int16_t));
    const uint64_t ld = (uint64_t)so_ld(p, plan);
    plan.s16_off = off;
    off += align256((uint64_t)p.G * ld * 4);
    plan.x16_off = off;
    off += align256((uint64_t)p.M * p.K * 2);
    if (p.offset) {
      // offset term: (M, ldx) group row sums (hi | lo) and (N, ldx) offsets, bf16
      plan.ldx = (int)((2 * p.G + BK - 1) / BK * BK);
      plan.dext_off = off;
      off += align256((uint64_t)p.M * plan.ldx * 2);
      plan.oext_off = off;
      off += align256((uint64_t)p.N * plan.ldx * 2);
    }
  }
  plan.ws_bytes = off;
  return true;
}

template <int DT, int WBITS, int MODE, int MH>
static cudaError_t launch_prefill_t(const Problem &p, const Plan &plan, void *ws, cudaStream_t s) {
  using L = Layout<WBITS, MH, MODE>;
  constexpr int TMROWS = BM * MH;
  static std::once_flag attr_once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(attr_once, [] {
    attr_err = cudaFuncSetAttribute(prefill_kernel<DT, WBITS, MODE, MH>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L::SMEM);
  });
  if (attr_err != cudaSuccess) return attr_err;
  EncodeTiledFn enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  char *wsb = static_cast<char *>(ws);

  PrefillArgs args = {};
  args.scale = p.scale; args.offset = p.offset; args.bias = p.bias; args.residual = p.residual;
  args.gamma = p.gamma; args.y = p.y; args.normOut = p.normOut;
  args.status = reinterpret_cast<uint32_t *>(ws);
  args.counters = reinterpret_cast<uint32_t *>(wsb + plan.cnt_off);
  args.rowpart = reinterpret_cast<float *>(wsb + plan.rowpart_off);
  args.M = p.M; args.K = (int)p.K; args.N = (int)p.N; args.group = (int)p.group; args.Ns = (int)p.Ns;
  args.nTilesN = (int)plan.n_tiles;
  args.kTiles = (int)((p.K + BK - 1) / BK);
  args.kTilesX = MODE == kF16Emu && p.offset ? plan.ldx / BK : 0;
  args.nTiles = plan.n_tiles * plan.m_tiles;
  args.mTiles = (int)plan.m_tiles;
  args.eps = p.eps;
  args.budget = wait_budget();
  args.extra = wait_extra_arrivals();

  // status word and row-block counters start at zero on every call
  cudaError_t e = cudaMemsetAsync(ws, 0, plan.rowpart_off, s);
  if (e != cudaSuccess) return e;

  const void *a_src = p.x1;
  const void *x_ext = nullptr, *o_ext = nullptr;  // offset-term operands (F16EMU with offset)
  CUtensorMapDataType a_type =
      DT == WQ_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  if constexpr (MODE == kRawQ) {
    if (p.offset) {
      float *rowsum = reinterpret_cast<float *>(wsb + plan.rowsum_off);
      e = launch_row_prep(p, rowsum, nullptr, nullptr, nullptr, 0, s);
      if (e != cudaSuccess) return e;
      args.rowsum = rowsum;
    }
  } else {
    int16_t *e_row = reinterpret_cast<int16_t *>(wsb + plan.erow_off);
    int16_t *e_col = reinterpret_cast<int16_t *>(wsb + plan.ecol_off);
    uint32_t *S16 = reinterpret_cast<uint32_t *>(wsb + plan.s16_off);
    __half *x16 = reinterpret_cast<__half *>(wsb + plan.x16_off);
    __nv_bfloat16 *dext = p.offset ? reinterpret_cast<__nv_bfloat16 *>(wsb + plan.dext_off) : nullptr;
    __nv_bfloat16 *oext = p.offset ? reinterpret_cast<__nv_bfloat16 *>(wsb + plan.oext_off) : nullptr;
    e = launch_row_prep(p, nullptr, e_row, x16, dext, plan.ldx, s);
    if (e != cudaSuccess) return e;
    e = launch_so_prep(p, so_ld(p, plan), e_col, S16, oext, plan.ldx, s);
    if (e != cudaSuccess) return e;
    args.e_row = e_row; args.e_col = e_col; args.S16 = S16;
    x_ext = dext;
    o_ext = oext;
    a_src = x16;
    a_type = CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  }

  CUtensorMap tm_x, tm_w;
  {
    const cuuint64_t dims[2] = {(cuuint64_t)p.K, (cuuint64_t)p.M};
    const cuuint64_t strides[1] = {(cuuint64_t)p.K * 2};
    const cuuint32_t box[2] = {BK, BM * MH};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(&tm_x, a_type, 2, const_cast<void *>(a_src), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  }
  {
    const cuuint64_t row_bytes = (cuuint64_t)p.N * WBITS / 8;
    const cuuint64_t dims[2] = {row_bytes, (cuuint64_t)p.K};
    const cuuint64_t strides[1] = {row_bytes};
    const cuuint32_t box[2] = {(cuuint32_t)(BN * WBITS / 8), BK};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(&tm_w, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(p.x2), dims, strides,
                     box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  }
  CUtensorMap tm_s = tm_w, tm_dx = tm_w, tm_ox = tm_w;  // placeholders unless F16EMU
  args.so_bytes = 0;
  if constexpr (MODE == kF16Emu) {
    const int64_t ld = so_ld(p, plan);
    const cuuint64_t dims[2] = {(cuuint64_t)ld, (cuuint64_t)p.G};
    const cuuint64_t strides[1] = {(cuuint64_t)ld * 4};
    // group rows a 64-deep k-stage touches: one when groups are whole multiples of it
    const cuuint32_t rows =
        p.group % BK == 0 ? 1u : (cuuint32_t)(p.G < SO_ROWS ? p.G : SO_ROWS);
    const cuuint32_t box[2] = {BN, rows};
    const cuuint32_t estr[2] = {1, 1};
    args.so_bytes = rows * BN * 4;
    CUresult r = enc(&tm_s, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<uint32_t *>(args.S16), dims,
                     strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    if (args.kTilesX > 0) {
      // A: (M, ldx) group row sums, 64 x (128 MH) boxes; B: (N, ldx) offsets,
      // 64 x 256 boxes; both bf16, K-major with the 128-byte swizzle of the MMA
      const cuuint64_t sx[1] = {(cuuint64_t)plan.ldx * 2};
      const cuuint32_t estr1[2] = {1, 1};
      const cuuint64_t dxd[2] = {(cuuint64_t)plan.ldx, (cuuint64_t)p.M};
      const cuuint32_t dxb[2] = {BK, (cuuint32_t)TMROWS};
      r = enc(&tm_dx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(x_ext), dxd, sx, dxb,
              estr1, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
      if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
      const cuuint64_t oxd[2] = {(cuuint64_t)plan.ldx, (cuuint64_t)p.N};
      const cuuint32_t oxb[2] = {BK, BN};
      r = enc(&tm_ox, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(o_ext), oxd, sx, oxb,
              estr1, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
      if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    }
  }
  // the residual, read in 32 x 32 boxes by the epilogue
  CUtensorMap tm_r;
  {
    const cuuint64_t dims[2] = {(cuuint64_t)p.N, (cuuint64_t)p.M};
    const cuuint64_t strides[1] = {(cuuint64_t)p.N * 2};
    const cuuint32_t box[2] = {32, 32};
    const cuuint32_t estr[2] = {1, 1};
    const CUtensorMapDataType t =
        DT == WQ_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    CUresult r = enc(&tm_r, t, 2, const_cast<void *>(p.residual), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  }
  prefill_kernel<DT, WBITS, MODE, MH>
      <<<plan.grid, kThreads, L::SMEM, s>>>(tm_x, tm_w, tm_s, tm_dx, tm_ox, tm_r, args);
  return cudaGetLastError();
}

template <int DT, int WBITS, int MODE>
static cudaError_t launch_prefill_h(const Problem &p, const Plan &plan, void *ws, cudaStream_t s) {
  if constexpr (WBITS == 4) {
    if (plan.m_halves == 2) return launch_prefill_t<DT, WBITS, MODE, 2>(p, plan, ws, s);
  }
  if (plan.m_halves != 1) return cudaErrorNotSupported;
  return launch_prefill_t<DT, WBITS, MODE, 1>(p, plan, ws, s);
}

template <int DT, int WBITS>
static cudaError_t launch_prefill_m(const Problem &p, const Plan &plan, void *ws, cudaStream_t s) {
  if (plan.mode == kF16Emu) {
    if constexpr (DT == WQ_BF16) return launch_prefill_h<DT, WBITS, kF16Emu>(p, plan, ws, s);
    return cudaErrorNotSupported;
  }
  return launch_prefill_h<DT, WBITS, kRawQ>(p, plan, ws, s);
}

cudaError_t launch_prefill(const Problem &p, const Plan &plan, void *ws, cudaStream_t s) {
  if (p.dtype == WQ_BF16)
    return p.wbits == 4 ? launch_prefill_m<WQ_BF16, 4>(p, plan, ws, s)
                        : launch_prefill_m<WQ_BF16, 8>(p, plan, ws, s);
  return p.wbits == 4 ? launch_prefill_m<WQ_F16, 4>(p, plan, ws, s)
                      : launch_prefill_m<WQ_F16, 8>(p, plan, ws, s);
}

}  // namespace wq
