// Decode (small-M) kernel of the weight-only quantized matmul with the fused
// residual-add + RMSNorm epilogue (aclnnWeightQuantMatmulAllReduceAddRmsNorm,
// "Function description": mm_out = x1 @ (x2*antiquantScale + antiquantOffset)
// + bias; y = mm_out + residual; normOut = y / RMS(y) * gamma).
//
// With M <= 16 rows the operator is a stream over the packed INT4 weight: every
// weight byte is read once and used for at most 16 products, so the kernel is
// built to keep HBM busy on every SM and to spend few instructions per weight.
//
// Work split (stream-K). Output columns come in n-tiles of 256 (128 bytes of
// packed INT4 per k-row); K comes in 64-row stages. The nTiles x kst units
// (tile, stage), in tile-major order, are cut into G equal contiguous runs of
// `per` units, one per CTA, G <= SM count, one CTA per SM. A run covers the end
// of one tile and the start of the next (or more), so each CTA produces one
// partial sum per tile it touches (a "segment").
//
// Warp roles (4*KH consumer warps + 1 producer warp):
//   producer   one elected lane streams the run through an NS-deep ring of
//              stages: the 64 x 128-byte box of packed weights and the 64 x MP
//              box of x1 (both 128-byte swizzled), plus the scale (and offset)
//              rows of the groups the stage touches, all by TMA, completion on
//              the stage's full mbarrier.
//   consumers  warp w takes the 64 columns 64*(w%4) .. +63 and the stages j
//              with j % KH == w / 4 (j counts the run's units). Per 16 k-rows it
//              turns four 32-bit words of nibbles into the A fragments of four
//              m16n8k16 MMAs (A = W^T, 16 columns x 16 k, exact integers q in
//              bf16/fp16), loads B = x1^T (16 k x 8 rows) with ldmatrix and
//              accumulates fp32. The scale is applied to each group's fp32 sum
//              when the group ends (the offset to the group's x1 row sum, from
//              the same MMA with an all-ones A), so the dequantized weight is
//              exact and only fp32 accumulation rounds.
// Segment end. The KH k-phases add in shared memory (fixed order) and the CTA
// writes the segment's M x 256 fp32 partial to the workspace, then counts it on
// the tile's counter. The CTA that brings the counter to the number of
// segments of the tile finishes the tile: it sums the segments in CTA order,
// adds bias and residual, writes y (and an fp32 copy to the workspace) and the
// tile's per-row sum of y^2, and clears the counter for the next call.
// RMSNorm. Every CTA then arrives at a grid-wide counter; once all have, each
// sums the tiles' row sums in tile order, forms 1/RMS per row and writes normOut
// for the tiles it finished. The last CTA to leave clears the counter. All
// reductions run in a fixed order: results are bitwise reproducible.
//
// Co-residency: G CTAs of one per SM are all resident, so the grid barrier
// cannot deadlock; every wait is bounded anyway, and a wait that gives up
// records WQ_ERR_DEVICE_TIMEOUT in the status word and lets the kernel finish.
//
// Programmatic dependent launch: before the dependency wait a CTA only warms
// L2 with the first stages of its run (a prefetch moves no data into the CTA
// and cannot observe a stale value); activations, weights, counters and
// outputs are touched only after it.
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

constexpr int DNT = 256;                    // columns per n-tile
constexpr int DKB = 64;                     // k-rows per stage
constexpr uint32_t DW = DKB * DNT / 2;      // 8 KB of packed INT4 per stage
constexpr uint32_t DSO = 2 * DNT * 2;       // 1 KB: the two group rows a stage can touch
constexpr int NS = 8;                       // pipeline depth (stages)
constexpr int kTileCounters = 256;          // N <= 65535 gives at most 256 tiles
constexpr uint32_t kGbarOff = 128;          // header: grid counters (arrive, depart)
constexpr uint32_t kTcntOff = 1024;         // header: per-tile segment counters

template <int MT>
struct DCfg {
  static constexpr int MP = 8 * MT;                // rows held (x1 box height)
  static constexpr int KH = MT == 1 ? 4 : 2;       // k-phases
  static constexpr int CW = 4 * KH;                // consumer warps
  static constexpr int CT = CW * 32;               // consumer threads
  static constexpr int THREADS = CT + 32;          // + producer warp
  static constexpr uint32_t XB = MP * 128;         // x1 box bytes per stage
  static constexpr uint32_t OFF_X = DW;            // slot: W | X | S | O
  static constexpr uint32_t OFF_S = DW + (XB + 1023) / 1024 * 1024;
  static constexpr uint32_t OFF_O = OFF_S + DSO;
  static constexpr uint32_t SLOT = OFF_O + DSO;    // a multiple of 1024
  static constexpr uint32_t OFF_RED = NS * SLOT;   // KH x MP x 256 fp32
  static constexpr uint32_t OFF_MISC = OFF_RED + KH * MP * DNT * 4;
  static constexpr uint32_t OFF_BAR = OFF_MISC + 2048;  // misc: 1/RMS, per-warp row sums, flags
  static_assert((16 + CW * 16 + 2) * 4 <= 2048, "misc area");
  static constexpr uint32_t SMEM = OFF_BAR + 8 * 2 * NS + 1024;  // + base alignment slack
  static_assert(SLOT % 1024 == 0, "stage slots keep the 128-byte swizzle atoms aligned");
};

enum DWhere : uint32_t { kDWhereProducer = 11, kDWhereConsumer = 12, kDWhereGrid = 15 };

struct DecodeArgs {
  const void *scale, *offset, *bias, *residual, *gamma;
  void *y, *normOut;
  uint32_t *status;   // header word 0
  uint32_t *gbar;     // header: [0] arrive, [1] depart
  uint32_t *tcnt;     // header: segments counted per tile
  float *part;        // G x SMAX x MP x 256 segment partials
  float *y32;         // nTiles x MP x 256 fp32 y
  float *ss;          // nTiles x 16 per-row sums of y^2
  int M, K, N, group, Ns;
  int nTiles, kst, U, per, G, SMAX, npf;
  float eps;
};

// Four nibble pairs -> two A-fragment registers of exact integers q: `lo` holds
// the low nibbles of byte i of wa (k) and wb (k+1), `hi` the high nibbles.
// (nib ^ 8) | magic is the 16-bit float 128 + q + 8 (bf16) or 1024 + q + 8
// (fp16); subtracting 136 / 1032 leaves q exactly.
template <int DT>
__device__ __forceinline__ void nib_pairs(uint32_t wa, uint32_t wb, int i, uint32_t &lo,
                                          uint32_t &hi) {
  constexpr uint32_t MAGIC = DT == WQ_BF16 ? 0x43084308u : 0x64086408u;
  const uint32_t sel = (uint32_t)i | ((uint32_t)i << 4) | ((uint32_t)(4 + i) << 8) |
                       ((uint32_t)(4 + i) << 12);
  const uint32_t x = __byte_perm(wa, wb, sel);
  lo = sub2<DT>((x & 0x000F000Fu) ^ MAGIC, MAGIC);
  hi = sub2<DT>(((x >> 4) & 0x000F000Fu) ^ MAGIC, MAGIC);
}

__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}

template <int DT>
__device__ __forceinline__ void lds8f(uint32_t addr, float (&f)[8]) {
  uint32_t v[4];
  asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3])
               : "r"(addr));
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float2 p = unpack2<DT>(v[q]);
    f[2 * q] = p.x;
    f[2 * q + 1] = p.y;
  }
}

template <int DT, int MT, bool HAS_O>
__global__ void __launch_bounds__(DCfg<MT>::THREADS, 1)
    decode_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_x,
                  const __grid_constant__ CUtensorMap tm_s, const __grid_constant__ CUtensorMap tm_o,
                  const DecodeArgs a) {
  using C = DCfg<MT>;
  using E = Elem<DT>;
  using T = typename E::T;
  constexpr int MP = C::MP, KH = C::KH, CT = C::CT;
  constexpr bool BF = DT == WQ_BF16;
  extern __shared__ uint8_t dsm_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(dsm_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_u32(smem);
  auto FULL = [&](int s) { return sb + C::OFF_BAR + 8u * s; };
  auto EMPTY = [&](int s) { return sb + C::OFF_BAR + 8u * (NS + s); };
  float *red = reinterpret_cast<float *>(smem + C::OFF_RED);
  float *misc = reinterpret_cast<float *>(smem + C::OFF_MISC);
  float *s_rstd = misc;                                              // [16]
  float *s_ssw = misc + 16;                                          // [CW][16]
  volatile int *abort_flag = reinterpret_cast<volatile int *>(misc + 16 + C::CW * 16);
  volatile int *s_fin = reinterpret_cast<volatile int *>(misc + 17 + C::CW * 16);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cta = blockIdx.x;
  const int u0 = cta * a.per;
  const int u1 = u0 + a.per < a.U ? u0 + a.per : a.U;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(FULL(s), 1);
      mbar_init(EMPTY(s), 4);  // the four column warps of the stage's k-phase
    }
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tm_w);
    prefetch_tmap(&tm_x);
    if (a.Ns != 1) {
      prefetch_tmap(&tm_s);
      if (HAS_O) prefetch_tmap(&tm_o);
    }
  }
  if (warp == C::CW && lane == 0) {
    const int npf = u1 - u0 < a.npf ? u1 - u0 : a.npf;
    for (int j = 0; j < npf; ++j) {
      const int u = u0 + j, tile = u / a.kst, st = u - tile * a.kst;
      tma_prefetch_l2_2d(&tm_w, tile * (DNT / 2), st * DKB);
    }
  }
  __syncthreads();
  griddep_wait();  // the previous grid on the stream has finished and flushed
  griddep_launch_dependents();

  if (warp == C::CW) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();  // each weight byte is used once per call
      const uint32_t so_bytes = a.Ns != 1 ? (a.group ? 2u : 1u) * DNT * 2u : 0u;
      const uint32_t bytes = DW + C::XB + (HAS_O ? 2u : 1u) * so_bytes;
      int slot = 0;
      uint32_t ph = 0;
      int issued = 0;
      for (int u = u0; u < u1; ++u) {
        if (!wait_bar(EMPTY(slot), ph ^ 1u, abort_flag, a.status, kDWhereProducer)) break;
        const int tile = u / a.kst, st = u - tile * a.kst;
        const int row0 = st * DKB;
        const uint32_t dst = sb + (uint32_t)slot * C::SLOT;
        mbar_arrive_expect_tx(FULL(slot), bytes);
        tma_load_2d_hint(dst, &tm_w, tile * (DNT / 2), row0, FULL(slot), pol);
        tma_load_2d(dst + C::OFF_X, &tm_x, row0, 0, FULL(slot));
        if (a.Ns != 1) {
          // the scale (and offset) rows of the groups this stage touches
          const int g0 = a.group ? row0 / a.group : 0;
          tma_load_2d(dst + C::OFF_S, &tm_s, tile * DNT, g0, FULL(slot));
          if (HAS_O) tma_load_2d(dst + C::OFF_O, &tm_o, tile * DNT, g0, FULL(slot));
        }
        ++issued;
        if (++slot == NS) { slot = 0; ph ^= 1u; }
      }
      // every copy issued has landed before the CTA may exit
      for (int j = (issued > NS ? issued - NS : 0); j < issued; ++j)
        drain_bar(FULL(j % NS), (uint32_t)((j / NS) & 1));
    }
    __syncwarp();
    return;
  }

  // ------------------------------------------------------------------ consumers
  const int ctid = threadIdx.x;
  const int wc = warp & 3, kh = warp >> 2;
  const int g = lane >> 2, t = lane & 3;
  const uint32_t ones = BF ? 0x3F803F80u : 0x3C003C00u;  // 1.0 in both halves
  const T *bias = static_cast<const T *>(a.bias);
  const T *res = static_cast<const T *>(a.residual);
  const T *gam = static_cast<const T *>(a.gamma);
  T *yout = static_cast<T *>(a.y);
  T *nout = static_cast<T *>(a.normOut);

  // ldmatrix row of this lane in an x1 box (rows m at 128-byte pitch, swizzled)
  int ldm_m, ldm_c;
  {
    const int l = MT == 2 ? lane : (lane & 15);
    const int jj = l >> 3;
    ldm_m = (l & 7) + 8 * (jj >> 1);
    ldm_c = jj & 1;
  }
  float sscal = 0.f, oscal = 0.f;  // per-tensor scale / offset
  if (a.Ns == 1) {
    sscal = E::to_f(static_cast<const T *>(a.scale)[0]);
    if (HAS_O) oscal = E::to_f(static_cast<const T *>(a.offset)[0]);
  }

  const int t0c = u0 / a.kst;                   // first tile of this CTA's run
  const int t1c = u1 > u0 ? (u1 - 1) / a.kst : t0c - 1;
  int fin_tiles[4];
  int nfin = 0;
  int j = 0, slot = 0;
  uint32_t ph = 0;

  for (int tile = t0c; tile <= t1c; ++tile) {
    const int sbeg = (u0 > tile * a.kst ? u0 - tile * a.kst : 0);
    const int send = (u1 < (tile + 1) * a.kst ? u1 - tile * a.kst : a.kst);
    float tot[MT][4][4], acc[MT][4][4], d1[MT][2];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int c = 0; c < 4; ++c) tot[mt][i][c] = acc[mt][i][c] = 0.f;
      d1[mt][0] = d1[mt][1] = 0.f;
    }
    float sf[8], of[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) { sf[q] = sscal; of[q] = oscal; }
    int cur = -1;
    auto flush = [&]() {
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float sl = sf[2 * i], sh = sf[2 * i + 1];
          if constexpr (HAS_O) {
            const float ol = of[2 * i], oh = of[2 * i + 1];
            tot[mt][i][0] += fmaf(sl, acc[mt][i][0], ol * d1[mt][0]);
            tot[mt][i][1] += fmaf(sl, acc[mt][i][1], ol * d1[mt][1]);
            tot[mt][i][2] += fmaf(sh, acc[mt][i][2], oh * d1[mt][0]);
            tot[mt][i][3] += fmaf(sh, acc[mt][i][3], oh * d1[mt][1]);
          } else {
            tot[mt][i][0] = fmaf(sl, acc[mt][i][0], tot[mt][i][0]);
            tot[mt][i][1] = fmaf(sl, acc[mt][i][1], tot[mt][i][1]);
            tot[mt][i][2] = fmaf(sh, acc[mt][i][2], tot[mt][i][2]);
            tot[mt][i][3] = fmaf(sh, acc[mt][i][3], tot[mt][i][3]);
          }
#pragma unroll
          for (int c = 0; c < 4; ++c) acc[mt][i][c] = 0.f;
        }
        d1[mt][0] = d1[mt][1] = 0.f;
      }
    };

    for (int st = sbeg; st < send; ++st) {
      if ((j & (KH - 1)) == kh) {
        const bool ok = wait_bar_warp(FULL(slot), ph, abort_flag, a.status, kDWhereConsumer);
        if (ok) {
          const uint32_t base = sb + (uint32_t)slot * C::SLOT;
          const int srow = st * DKB;
          const int gs = a.group ? srow / a.group : 0;  // group of the stage's first row
          const int gnext = a.group ? (gs + 1) * a.group : 0x7fffffff;
#pragma unroll
          for (int kb = 0; kb < DKB / 16; ++kb) {
            const int row0 = srow + 16 * kb;
            // a 64-row stage crosses at most one group boundary per 32 rows
            const int grp = row0 >= gnext ? row0 / a.group : gs;
            if (grp != cur) {
              if (cur >= 0) flush();
              cur = grp;
              if (a.Ns != 1) {
                const uint32_t so = base + C::OFF_S + (uint32_t)((grp - gs) * DNT + 64 * wc + 8 * g) * 2u;
                lds8f<DT>(so, sf);
                if constexpr (HAS_O) lds8f<DT>(so + DSO, of);
              }
            }
            // four words of nibbles: stage rows 16kb + 2t + {0, 1, 8, 9}, bytes
            // 4g..4g+3 of this warp's 32-byte column span, through the swizzle
            uint32_t w[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const int rl = 16 * kb + 2 * t + (q & 1) + 8 * (q >> 1);
              const uint32_t chunk = (uint32_t)((2 * wc + (g >> 2)) ^ (rl & 7));
              w[q] = lds32(base + (uint32_t)rl * 128u + (chunk << 4) + (uint32_t)((g & 3) << 2));
            }
            // B = x1^T for these 16 k (x1 box: row m at m*128, 16-byte chunk c at c ^ (m & 7))
            uint32_t b[MT][2];
            {
              const int cidx = 2 * kb + ldm_c;
              const uint32_t baddr =
                  base + C::OFF_X + (uint32_t)ldm_m * 128u + ((uint32_t)(cidx ^ (ldm_m & 7)) << 4);
              if constexpr (MT == 2)
                ldmatrix_x4(baddr, b[0][0], b[0][1], b[1][0], b[1][1]);
              else
                ldmatrix_x2(baddr, b[0][0], b[0][1]);
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              uint32_t a0, a1, a2, a3;
              nib_pairs<DT>(w[0], w[1], i, a0, a1);
              nib_pairs<DT>(w[2], w[3], i, a2, a3);
#pragma unroll
              for (int mt = 0; mt < MT; ++mt)
                mma_16816<BF>(acc[mt][i], a0, a1, a2, a3, b[mt][0], b[mt][1]);
            }
            if constexpr (HAS_O) {
#pragma unroll
              for (int mt = 0; mt < MT; ++mt) {
                float dd[4] = {d1[mt][0], d1[mt][1], d1[mt][0], d1[mt][1]};
                mma_16816<BF>(dd, ones, ones, ones, ones, b[mt][0], b[mt][1]);
                d1[mt][0] = dd[0];
                d1[mt][1] = dd[1];
              }
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(EMPTY(slot));
      }
      ++j;
      if (++slot == NS) { slot = 0; ph ^= 1u; }
    }
    if (cur >= 0) flush();

    // ---- segment end: k-phases add in shared memory, the partial goes to the workspace
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int c = 0; c < 4; ++c)
          red[(kh * MP + 8 * mt + 2 * t + (c & 1)) * DNT + 64 * wc + 8 * g + 2 * i + (c >> 1)] =
              tot[mt][i][c];
    named_bar_sync(1, CT);
    float4 *dstp = reinterpret_cast<float4 *>(
        a.part + ((int64_t)cta * a.SMAX + (tile - t0c)) * (MP * DNT));
    for (int q = ctid; q < MP * DNT / 4; q += CT) {
      float4 v = reinterpret_cast<const float4 *>(red)[q];
#pragma unroll
      for (int h = 1; h < KH; ++h) {
        const float4 w4 = reinterpret_cast<const float4 *>(red + h * MP * DNT)[q];
        v.x += w4.x; v.y += w4.y; v.z += w4.z; v.w += w4.w;
      }
      __stcg(dstp + q, v);
    }
    __threadfence();
    named_bar_sync(1, CT);
    if (ctid == 0) {
      const int c_first = (tile * a.kst) / a.per;
      const int c_last = ((tile + 1) * a.kst - 1) / a.per;
      const uint32_t old = atomicAdd(a.tcnt + tile, 1u);
      const int last = old == (uint32_t)(c_last - c_first);
      if (last) __threadfence();
      *s_fin = last;
    }
    named_bar_sync(1, CT);
    const bool finisher = *s_fin != 0;
    if (finisher) {
      // ---- finish the tile: segments in CTA order + bias + residual -> y, sum(y^2)
      const int c_first = (tile * a.kst) / a.per;
      const int c_last = ((tile + 1) * a.kst - 1) / a.per;
      for (int q = ctid; q < C::CW * 16; q += CT) s_ssw[q] = 0.f;
      named_bar_sync(1, CT);
      for (int idx = ctid; idx < MP * DNT; idx += CT) {
        const int m = idx / DNT, col = idx - m * DNT;  // a warp shares one row m
        const int n = tile * DNT + col;
        float v = 0.f;
#pragma unroll 4
        for (int cc = c_first; cc <= c_last; ++cc) {
          const int seg = tile - (cc * a.per) / a.kst;
          v += __ldcg(a.part + ((int64_t)cc * a.SMAX + seg) * (MP * DNT) + idx);
        }
        float yv = 0.f;
        if (m < a.M && n < a.N) {
          yv = v + (bias ? E::to_f(bias[n]) : 0.f) + E::to_f(res[(int64_t)m * a.N + n]);
          yout[(int64_t)m * a.N + n] = E::from_f(yv);
        }
        __stcg(a.y32 + (int64_t)tile * (MP * DNT) + idx, yv);
        float sq = yv * yv;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, o);
        if (lane == 0) s_ssw[warp * 16 + m] += sq;
      }
      named_bar_sync(1, CT);
      if (ctid < MP) {
        float v = 0.f;
        for (int w = 0; w < C::CW; ++w) v += s_ssw[w * 16 + ctid];
        __stcg(a.ss + tile * 16 + ctid, v);
      }
      if (ctid == 0) a.tcnt[tile] = 0u;  // the last user of this counter in this call
      if (nfin < 4) fin_tiles[nfin] = tile;
      ++nfin;
      __threadfence();
    }
  }

  // ---- grid barrier, then 1/RMS per row and normOut of the tiles this CTA finished
  named_bar_sync(1, CT);
  if (ctid == 0) {
    red_release_add(a.gbar, 1u);
    const long long t0 = clock64();
    while (ld_acquire_u32(a.gbar) < (uint32_t)a.G) {
      if (*abort_flag) break;
      if (clock64() - t0 > kWaitBudget) {
        *abort_flag = 1;
        record_timeout(a.status, kDWhereGrid);
        break;
      }
      __nanosleep(32);
    }
  }
  named_bar_sync(1, CT);
  if (ctid < a.M && nfin > 0) {
    float tot = 0.f;
#pragma unroll 8
    for (int tl = 0; tl < a.nTiles; ++tl) tot += __ldcg(a.ss + tl * 16 + ctid);
    s_rstd[ctid] = rsqrtf(tot / (float)a.N + a.eps);
  }
  named_bar_sync(1, CT);
  if (ctid == 0) {
    // the last CTA through clears the grid counters for the next call
    if (atomicAdd(a.gbar + 1, 1u) == (uint32_t)a.G - 1u) {
      atomicExch(a.gbar, 0u);
      atomicExch(a.gbar + 1, 0u);
    }
  }
  for (int f = 0; f < nfin && f < 4; ++f) {
    const int tile = fin_tiles[f];
    for (int idx = ctid; idx < MP * DNT; idx += CT) {
      const int m = idx / DNT, col = idx - m * DNT;
      const int n = tile * DNT + col;
      if (m < a.M && n < a.N)
        nout[(int64_t)m * a.N + n] =
            E::from_f(__ldcg(a.y32 + (int64_t)tile * (MP * DNT) + idx) * s_rstd[m] * E::to_f(gam[n]));
    }
  }
}

// ------------------------------------------------------------------ host side

using EncodeTiledFn = PFN_cuTensorMapEncodeTiled_v12000;

EncodeTiledFn dencode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
    else
      cudaGetLastError();
  });
  return fn;
}

bool daligned16(const void *p) { return p == nullptr || (reinterpret_cast<uintptr_t>(p) % 16) == 0; }

// Geometry of one call, from the problem and the SM count alone (so the first
// phase, without a GPU, sizes the workspace exactly as the launch uses it).
struct DecodeGeom {
  int MP, kst, nTiles, U, per, G, SMAX;
  uint64_t part_off, y32_off, ss_off, ws_bytes;
};

uint64_t dalign256(uint64_t v) { return (v + 255) / 256 * 256; }

DecodeGeom decode_geom(const Problem &p) {
  DecodeGeom gm;
  gm.MP = p.M <= 8 ? 8 : 16;
  gm.kst = (int)((p.K + DKB - 1) / DKB);
  gm.nTiles = (int)((p.N + DNT - 1) / DNT);
  gm.U = gm.nTiles * gm.kst;
  const int sms = device_info().sms > 0 ? device_info().sms : 148;
  gm.per = (gm.U + sms - 1) / sms;
  gm.G = (gm.U + gm.per - 1) / gm.per;
  gm.SMAX = (gm.per + gm.kst - 1) / gm.kst + 1;  // tiles a run of `per` units can touch
  gm.part_off = kWsHeader;
  gm.y32_off = gm.part_off + dalign256((uint64_t)gm.G * gm.SMAX * gm.MP * DNT * 4);
  gm.ss_off = gm.y32_off + dalign256((uint64_t)gm.nTiles * gm.MP * DNT * 4);
  gm.ws_bytes = gm.ss_off + dalign256((uint64_t)gm.nTiles * 16 * 4);
  return gm;
}

}  // namespace

bool decode_applicable(const Problem &p) {
  if (p.M < 1 || p.M > 16 || p.N < 1) return false;
  if (p.wbits != 4) return false;
  if (p.N % 32 != 0) return false;  // packed row = N/2 bytes, a multiple of 16 for TMA
  if (p.K % 8 != 0) return false;   // x1 row pitch, a multiple of 16 bytes for TMA
  if ((p.N + DNT - 1) / DNT > kTileCounters) return false;
  const void *ptrs[] = {p.x1, p.x2, p.scale, p.offset};
  for (const void *q : ptrs)
    if (!daligned16(q)) return false;
  const DecodeGeom gm = decode_geom(p);
  return gm.SMAX <= 4;  // a CTA finishes at most four tiles
}

bool plan_decode(const Problem &p, Plan &plan) {
  if (!decode_applicable(p)) return false;
  plan.kernel = WQ_KERNEL_DECODE;
  plan.ws_bytes = decode_geom(p).ws_bytes;
  return true;
}

template <int DT, int MT, bool HAS_O>
static cudaError_t launch_decode_t(const Problem &p, const Plan &plan, void *ws, cudaStream_t s) {
  (void)plan;
  using C = DCfg<MT>;
  EncodeTiledFn enc = dencode_fn();
  if (!enc) return cudaErrorNotSupported;
  static std::once_flag attr_once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(attr_once, [] {
    attr_err = cudaFuncSetAttribute(decode_kernel<DT, MT, HAS_O>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::SMEM);
  });
  if (attr_err != cudaSuccess) return attr_err;
  const DecodeGeom gm = decode_geom(p);
  if (gm.G > device_info().sms) return cudaErrorInvalidConfiguration;

  const CUtensorMapDataType fty =
      DT == WQ_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  CUtensorMap tm_w, tm_x, tm_s, tm_o;
  {
    const cuuint64_t row_bytes = (cuuint64_t)p.N / 2;
    const cuuint64_t dims[2] = {row_bytes, (cuuint64_t)p.K};
    const cuuint64_t strides[1] = {row_bytes};
    const cuuint32_t box[2] = {DNT / 2, DKB};
    const cuuint32_t estr[2] = {1, 1};
    if (enc(&tm_w, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(p.x2), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  {
    const cuuint64_t dims[2] = {(cuuint64_t)p.K, (cuuint64_t)p.M};
    const cuuint64_t strides[1] = {(cuuint64_t)p.K * 2};
    const cuuint32_t box[2] = {DKB, (cuuint32_t)C::MP};
    const cuuint32_t estr[2] = {1, 1};
    if (enc(&tm_x, fty, 2, const_cast<void *>(p.x1), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  tm_s = tm_w;  // placeholders unless the scale has N columns
  tm_o = tm_w;
  if (p.Ns != 1) {
    const cuuint64_t dims[2] = {(cuuint64_t)p.N, (cuuint64_t)p.G};
    const cuuint64_t strides[1] = {(cuuint64_t)p.N * 2};
    const cuuint32_t box[2] = {DNT, p.smode == kPerGroup ? 2u : 1u};
    const cuuint32_t estr[2] = {1, 1};
    if (enc(&tm_s, fty, 2, const_cast<void *>(p.scale), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
    if (HAS_O &&
        enc(&tm_o, fty, 2, const_cast<void *>(p.offset), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  char *wsb = static_cast<char *>(ws);
  DecodeArgs args = {};
  args.scale = p.scale; args.offset = p.offset; args.bias = p.bias;
  args.residual = p.residual; args.gamma = p.gamma; args.y = p.y; args.normOut = p.normOut;
  args.status = reinterpret_cast<uint32_t *>(ws);
  args.gbar = reinterpret_cast<uint32_t *>(wsb + kGbarOff);
  args.tcnt = reinterpret_cast<uint32_t *>(wsb + kTcntOff);
  args.part = reinterpret_cast<float *>(wsb + gm.part_off);
  args.y32 = reinterpret_cast<float *>(wsb + gm.y32_off);
  args.ss = reinterpret_cast<float *>(wsb + gm.ss_off);
  args.M = (int)p.M; args.K = (int)p.K; args.N = (int)p.N;
  args.group = (int)p.group; args.Ns = (int)p.Ns;
  args.nTiles = gm.nTiles; args.kst = gm.kst; args.U = gm.U; args.per = gm.per; args.G = gm.G;
  args.SMAX = gm.SMAX;
  args.npf = gm.per < 16 ? gm.per : 16;
  args.eps = p.eps;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)gm.G, 1, 1);
  cfg.blockDim = dim3(C::THREADS, 1, 1);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, decode_kernel<DT, MT, HAS_O>, tm_w, tm_x, tm_s, tm_o, args);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_decode(const Problem &p, const Plan &plan, void *ws, cudaStream_t s) {
  const bool o = p.offset != nullptr;
  const int MT = p.M <= 8 ? 1 : 2;
  if (p.dtype == WQ_BF16) {
    if (MT == 1) return o ? launch_decode_t<WQ_BF16, 1, true>(p, plan, ws, s)
                          : launch_decode_t<WQ_BF16, 1, false>(p, plan, ws, s);
    return o ? launch_decode_t<WQ_BF16, 2, true>(p, plan, ws, s)
             : launch_decode_t<WQ_BF16, 2, false>(p, plan, ws, s);
  }
  if (MT == 1) return o ? launch_decode_t<WQ_F16, 1, true>(p, plan, ws, s)
                        : launch_decode_t<WQ_F16, 1, false>(p, plan, ws, s);
  return o ? launch_decode_t<WQ_F16, 2, true>(p, plan, ws, s)
           : launch_decode_t<WQ_F16, 2, false>(p, plan, ws, s);
}

}  // namespace wq
