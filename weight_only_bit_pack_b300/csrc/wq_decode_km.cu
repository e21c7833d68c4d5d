// k-major decode kernel of the fused operator for weights in the kernel-native
// tiled INT4 layout, 9..64 rows (aclnnWeightQuantMatmulAllReduceAddRmsNorm,
// "Function description": mm_out = x1 @ (x2*antiquantScale + antiquantOffset)
// + bias; y = mm_out + residual; normOut = y / RMS(y) * gamma; the tiled
// weight is the pack's matrix-unit output, aclnnConvertWeightToINT4Pack).
//
// With 9..64 rows x1 no longer fits in shared memory whole (8192 k-rows x 32
// rows is 512 KB), so every CTA walks K in slices of 128 k-rows and all its
// warps work on the same slice: the slice of x1 (all rows, 128 k-rows) is
// copied once per CTA by the TMA into a ring of shared-memory stages and read
// by every warp.
//
// Work split. Column groups of 16 (one tile column) are dealt to the CTAs in
// contiguous, balanced ranges (at most 14 per CTA); warp w < 14 owns column
// group w of its CTA for the whole of K, so no partial sum crosses warps or
// CTAs. Warp 15 is the producer (two 64 x MP boxes of x1 per slice, 128-byte
// swizzle); warp 14 forms each slice's x1 row sums d (MMAs with an all-ones
// A operand) into a small ring beside it.
//
// Per slice a consumer warp has the two 512-byte tiles of its column group
// (k-steps 2j, 2j+1), loaded TD slices ahead into registers: each word gives
// four A registers (136 + q, or 1032 + q in fp16, exactly) of m16n8k16 MMAs
// with B = x1^T from the staged slice (eight row blocks: two passes of four
// over the same weight words, converted again per pass). A scale group is a whole number of
// slices (group % 128 == 0), or the scale is per-channel or per-tensor, so the
// warp folds every slice's sums at once: tot += S acc + (O - 136 S) d, with the
// scale (offset) values of its two columns loaded a slice ahead.
//
// Epilogue: each consumer warp adds bias and residual to its 16 columns, writes
// y and keeps it in registers, and puts its per-row sums of y^2 in shared
// memory; the CTA adds them in warp order and publishes one partial per row;
// after a grid-wide counter (one CTA per SM, all resident) every CTA sums the
// partials in CTA order, forms 1/RMS per row and writes normOut for its columns.
// Every reduction runs in a fixed order, so results are bitwise reproducible.
// Every wait is bounded; a wait that gives up records WQ_ERR_DEVICE_TIMEOUT and
// the kernel writes no normOut.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "wq_common.cuh"
#include "wq_internal.h"
#include "wq_sm100.cuh"
#include "wq_sync.cuh"
#include "wq_tiled_frag.cuh"

namespace wq {
namespace {

using namespace sm100;
using namespace tfrag;

constexpr int KW = 16;                   // warps per CTA
constexpr int KTHREADS = KW * 32;
constexpr int kKmCons = 14;              // consumer warps (column groups per CTA at most)
constexpr int kKmDWarp = 14;             // the x1 row-sum warp
constexpr int kKmPWarp = 15;             // the producer warp
constexpr int kKmParts = 5;              // per-CTA partial sums a lane reads: grid <= 160
constexpr uint32_t kKmGbarOff = 128;     // header: grid counters (arrive, depart)
enum KmWhere : uint32_t { kKmWhereProducer = 21, kKmWhereRowSums = 22, kKmWhereConsumer = 23, kKmWhereGrid = 15 };

struct KmArgs {
  const uint8_t *w;
  const void *scale, *offset, *bias, *residual, *gamma;
  void *y, *normOut;
  uint32_t *status, *gbar;
  float *ss;            // 64 x G per-CTA sums of y^2, row-major by row
  int M, K, N, KS2, NCG, group, Ns, G;
  float eps;
  long long budget;
  uint32_t extra;
};

// Shared memory (dynamic, after alignment to 1024 bytes for the swizzled boxes).
template <int MT>
struct KmLayout {
  static constexpr int MP = 8 * MT;
  static constexpr int ST = MT == 2 ? 12 : (MT == 4 ? 8 : 6);  // x1 slice ring depth
  static constexpr uint32_t XBOX = MP * 128;          // one 64-k box of MP rows
  static constexpr uint32_t XSLOT = 2 * XBOX;         // one 128-k slice
  static constexpr uint32_t RING = ST * XSLOT;
  static constexpr uint32_t D_OFF = RING;             // [stages][MP] row sums
  static constexpr uint32_t P_OFF = D_OFF + ST * MP * 4;  // [cons][MP] row partials of y^2
  static constexpr uint32_t E_OFF = P_OFF + kKmCons * MP * 4;    // residual [M][ncols], bias, gamma
};

template <int MT>
uint64_t km_smem_t(const Problem &p, int G) {
  const int64_t ncg_max = (p.N / 16 + G - 1) / G;
  return 1024 + KmLayout<MT>::E_OFF + (uint64_t)(p.M + 2) * ncg_max * 16 * 2;
}
uint64_t km_smem(const Problem &p, int G, int MT) {
  return MT == 2 ? km_smem_t<2>(p, G) : (MT == 4 ? km_smem_t<4>(p, G) : km_smem_t<8>(p, G));
}

template <int DT, int MT, bool HAS_O, int TD>
__global__ void __launch_bounds__(KTHREADS, 1)
    decode_km_kernel(const __grid_constant__ CUtensorMap tm_x, const KmArgs a) {
  using L = KmLayout<MT>;
  using E = Elem<DT>;
  using T = typename E::T;
  constexpr bool BF = DT == WQ_BF16;
  constexpr int MP = L::MP;

  extern __shared__ uint8_t km_raw[];
  uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(km_raw) + 1023) &
                                            ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_u32(sm);
  float *dsl = reinterpret_cast<float *>(sm + L::D_OFF);
  float *rowp = reinterpret_cast<float *>(sm + L::P_OFF);
  constexpr int ST_ = L::ST;
  __shared__ __align__(8) uint64_t s_bar[3 * ST_];  // full, row sums ready, empty
  __shared__ float s_rstd[64];
  __shared__ int s_abort;
  auto FULL = [&](int s) { return smem_u32(&s_bar[s]); };
  auto DRDY = [&](int s) { return smem_u32(&s_bar[ST_ + s]); };
  auto EMPTY = [&](int s) { return smem_u32(&s_bar[2 * ST_ + s]); };
  volatile int *abort_flag = &s_abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int cta = blockIdx.x;
  const int cg0 = (int)((long long)cta * a.NCG / a.G);
  const int cg1 = (int)((long long)(cta + 1) * a.NCG / a.G);
  const int ncg = cg1 - cg0;  // <= kKmCons (host)
  const int ncols = 16 * ncg;
  T *eres = reinterpret_cast<T *>(sm + L::E_OFF);  // [M][ncols]
  T *ebias = eres + (size_t)a.M * ncols;           // [ncols]
  T *egam = ebias + ncols;                         // [ncols]

  if (threadIdx.x == 0) {
    for (int s = 0; s < ST_; ++s) {
      mbar_init(FULL(s), 1);
      mbar_init(DRDY(s), 1);
      mbar_init(EMPTY(s), (uint32_t)ncg + 1);  // the consumer warps and the row-sum warp
    }
    s_abort = 0;
    fence_mbar_init();
    prefetch_tmap(&tm_x);
  }
  __syncthreads();
  griddep_wait();  // the previous kernel on the stream has finished and flushed
  griddep_launch_dependents();
  {  // epilogue operands: 16-byte chunks, two per column group and row
    const int cpr = 2 * ncg;
    const T *bias = static_cast<const T *>(a.bias);
    for (int i = threadIdx.x; i < (a.M + 2) * cpr; i += KTHREADS) {
      const int r = i / cpr, q = i - r * cpr;
      const int col = 8 * q;
      if (r < a.M)
        cp_async16(smem_u32(eres + (size_t)r * ncols + col),
                   static_cast<const T *>(a.residual) + (size_t)r * a.N + 16 * cg0 + col);
      else if (r == a.M && bias)
        cp_async16(smem_u32(ebias + col), bias + 16 * cg0 + col);
      else if (r == a.M + 1)
        cp_async16(smem_u32(egam + col), static_cast<const T *>(a.gamma) + 16 * cg0 + col);
    }
    cp_async_commit();
  }

  // B column n of row block mt is x1 row 8 mt + xrow(n), xrow(n) = 4 (n & 1) + n / 2:
  // the lanes of one 8-lane phase of a 16-byte load (g = 2i, 2i + 1) then read
  // rows whose swizzle differs in bit 2, i.e. eight distinct 16-byte chunks.
  // Accumulator element e of lane (g, t) is x1 row 8 mt + 4 (e & 1) + t.
  const int xr = ((g & 1) << 2) | (g >> 1);
  // the lane's 16 bytes of x1 row 8 mt + xr, k-rows 32 h + 8 t .. of box q of a
  // stage (128-byte rows, 16-byte chunk c of row r at chunk c ^ (r & 7))
  // (half h of the lane's 32 k-rows, row blocks mt0 .. mt0 + NR - 1)
  auto load_xh = [&](uint32_t stage, int q, int h, int mt0, auto &xh) {
    constexpr int NR = sizeof(xh) / sizeof(uint4);
#pragma unroll
    for (int r = 0; r < NR; ++r) {
      const uint32_t row = (uint32_t)(8 * (mt0 + r) + xr);
      const uint32_t addr = stage + (uint32_t)q * L::XBOX + row * 128u +
                            ((uint32_t)((4 * h + t) ^ xr) << 4);
      asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                   : "=r"(xh[r].x), "=r"(xh[r].y), "=r"(xh[r].z), "=r"(xh[r].w)
                   : "r"(addr));
    }
  };

  // consumer warps: the folded sums of their 16 columns, then y (kept for normOut)
  float tot[MT][4];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int i = 0; i < 4; ++i) tot[mt][i] = 0.f;
  if (warp == kKmPWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int issued = 0;
      for (int j = 0; j < a.KS2; ++j) {
        const int s = j % ST_;
        const uint32_t ph = (uint32_t)((j / ST_) & 1);
        if (!wait_bar(EMPTY(s), ph ^ 1u, abort_flag, a.status, kKmWhereProducer)) break;
        mbar_arrive_expect_tx(FULL(s), L::XSLOT);
        tma_load_2d(sb + (uint32_t)s * L::XSLOT, &tm_x, 128 * j, 0, FULL(s));
        tma_load_2d(sb + (uint32_t)s * L::XSLOT + L::XBOX, &tm_x, 128 * j + 64, 0, FULL(s));
        ++issued;
      }
      // every copy issued has landed before the CTA may exit
      for (int j = issued - ST_ > 0 ? issued - ST_ : 0; j < issued; ++j)
        drain_bar(FULL(j % ST_), (uint32_t)((j / ST_) & 1));
    }
    __syncwarp();
  } else if (warp == kKmDWarp) {
    // ---------------------------------------- x1 row sums of every slice,
    // stored by B column (8 mt + n), the order in which the consumers read them
    constexpr uint32_t ONES = BF ? 0x3F803F80u : 0x3C003C00u;
    const uint32_t ONES4[4] = {ONES, ONES, ONES, ONES};
    for (int j = 0; j < a.KS2; ++j) {
      const int s = j % ST_;
      const uint32_t ph = (uint32_t)((j / ST_) & 1);
      if (!wait_bar_warp(FULL(s), ph, abort_flag, a.status, kKmWhereRowSums)) break;
      constexpr int DB = MT < 4 ? MT : 4;  // row blocks per pass (registers)
#pragma unroll
      for (int pp = 0; pp < MT / DB; ++pp) {
        float dd[DB][4];
#pragma unroll
        for (int r = 0; r < DB; ++r)
#pragma unroll
          for (int i = 0; i < 4; ++i) dd[r][i] = 0.f;
#pragma unroll
        for (int q = 0; q < 2; ++q)
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            uint4 xh[DB];
            load_xh(sb + (uint32_t)s * L::XSLOT, q, h, pp * DB, xh);
#pragma unroll
            for (int r = 0; r < DB; ++r) {
              mma_16816_f<BF>(dd[r], ONES4, xh[r].x, xh[r].y);
              mma_16816_f<BF>(dd[r], ONES4, xh[r].z, xh[r].w);
            }
          }
        if (g == 0) {
#pragma unroll
          for (int r = 0; r < DB; ++r)
            *reinterpret_cast<float2 *>(dsl + s * MP + 8 * (pp * DB + r) + 2 * t) =
                make_float2(dd[r][0], dd[r][1]);
        }
      }
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(DRDY(s));   // releases the row sums written above
        mbar_arrive(EMPTY(s));  // done reading the slice
      }
    }
  } else if (warp < ncg) {
    // ------------------------------------------------------------ consumers
    const int cg = cg0 + warp;  // this warp's column group
    const size_t slab = (size_t)a.NCG * 512;  // bytes of one 64-row slab of tiles
    const uint8_t *wbase = a.w + (size_t)cg * 512 + lane * 16;
    // per slot of the register ring (TD slices ahead): the two tiles of slice
    // j and the scale (offset) values of the lane's columns g and 8 + g for it
    // (group row 128 j / group, or row 0), kept as loaded (no register moves
    // of values in flight)
    const bool so = a.Ns != 1;
    const uint16_t *sbits = static_cast<const uint16_t *>(a.scale);
    const uint16_t *obits = static_cast<const uint16_t *>(a.offset);
    const int scol = 16 * cg + g;
    uint4 wb[TD][2];
    uint16_t sr[TD][2], orr[TD][2];
    auto fetch = [&](int j, uint4 (&b)[2], uint16_t (&sv)[2], uint16_t (&ov)[2]) {
      const uint8_t *p = wbase + (size_t)(2 * j) * slab;
      b[0] = ld_stream_u4(p);
      b[1] = ld_stream_u4(p + slab);
      if (so) {
        const size_t row = (size_t)(a.group ? (128 * j) / a.group : 0) * (size_t)a.N;
        sv[0] = __ldg(sbits + row + scol);
        sv[1] = __ldg(sbits + row + scol + 8);
        if constexpr (HAS_O) {
          ov[0] = __ldg(obits + row + scol);
          ov[1] = __ldg(obits + row + scol + 8);
        }
      }
    };
#pragma unroll
    for (int i = 0; i < TD; ++i)
      if (i < a.KS2) fetch(i, wb[i], sr[i], orr[i]);
    const float sscal = so ? 0.f : E::to_f(static_cast<const T *>(a.scale)[0]);
    const float oscal = (HAS_O && !so) ? E::to_f(static_cast<const T *>(a.offset)[0]) : 0.f;
    constexpr float C136 = BF ? 136.f : 1032.f;  // A = C136 + q
    auto to_f = [&](uint16_t u) {
      if constexpr (BF) return __uint_as_float((uint32_t)u << 16);
      else return __half2float(__ushort_as_half(u));
    };

    // one slice from ring slot i; refilled with slice j + TD after use
    auto slice = [&](int j, uint4 (&wbi)[2], uint16_t (&sri)[2], uint16_t (&ori)[2]) -> bool {
      const int s = j % ST_;
      const uint32_t ph = (uint32_t)((j / ST_) & 1);
      if (!wait_bar_warp(DRDY(s), ph, abort_flag, a.status, kKmWhereConsumer)) return false;
      if (!wait_bar_warp(FULL(s), ph, abort_flag, a.status, kKmWhereConsumer)) return false;
      const uint32_t stage = sb + (uint32_t)s * L::XSLOT;
      const float sl = so ? to_f(sri[0]) : sscal, shi = so ? to_f(sri[1]) : sscal;
      float ol = oscal, ohi = oscal;
      if constexpr (HAS_O) {
        if (so) {
          ol = to_f(ori[0]);
          ohi = to_f(ori[1]);
        }
      }
      const float c0 = fmaf(-C136, sl, ol), c1 = fmaf(-C136, shi, ohi);
      // passes of RB row blocks; with two row blocks one accumulator per k-step
      // of the slice (two chains of four MMAs instead of one of eight)
      constexpr int RB = MT < 4 ? MT : 4, NP = MT / RB;
      constexpr int NA = MT == 2 ? 2 : 1;
#pragma unroll
      for (int pp = 0; pp < NP; ++pp) {
        float acc[NA][RB][4];
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const int qa = NA == 2 ? q : 0;
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            uint4 xh[RB];
            load_xh(stage, q, h, pp * RB, xh);
#pragma unroll
            for (int jl = 0; jl < 2; ++jl) {
              const int jj = 2 * h + jl;
              uint32_t aa[4];
              word_to_a<DT>(jj == 0 ? wbi[q].x : jj == 1 ? wbi[q].y : jj == 2 ? wbi[q].z : wbi[q].w, aa);
#pragma unroll
              for (int r = 0; r < RB; ++r) {
                const uint32_t b0 = jl ? xh[r].z : xh[r].x;
                const uint32_t b1 = jl ? xh[r].w : xh[r].y;
                if (jj == 0 && (q == 0 || NA == 2))
                  mma_16816_z<BF>(acc[qa][r], aa, b0, b1);
                else
                  mma_16816_f<BF>(acc[qa][r], aa, b0, b1);
              }
            }
          }
        }
#pragma unroll
        for (int r = 0; r < RB; ++r) {
          const int mt = pp * RB + r;
          if constexpr (NA == 2) {
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[0][r][e] += acc[1][r][e];
          }
          const float2 dd = *reinterpret_cast<const float2 *>(dsl + s * MP + 8 * mt + 2 * t);
          tot[mt][0] = fmaf(c0, dd.x, fmaf(sl, acc[0][r][0], tot[mt][0]));
          tot[mt][1] = fmaf(c0, dd.y, fmaf(sl, acc[0][r][1], tot[mt][1]));
          tot[mt][2] = fmaf(c1, dd.x, fmaf(shi, acc[0][r][2], tot[mt][2]));
          tot[mt][3] = fmaf(c1, dd.y, fmaf(shi, acc[0][r][3], tot[mt][3]));
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(EMPTY(s));  // the slice and its row sums are read
      if (j + TD < a.KS2) fetch(j + TD, wbi, sri, ori);
      return true;
    };
    int j0 = 0;
    bool ok = true;
    for (; ok && j0 + TD <= a.KS2; j0 += TD) {
#pragma unroll
      for (int i = 0; i < TD; ++i)
        if (ok) ok = slice(j0 + i, wb[i], sr[i], orr[i]);
    }
#pragma unroll
    for (int i = 0; i < TD; ++i)
      if (ok && j0 + i < a.KS2) ok = slice(j0 + i, wb[i], sr[i], orr[i]);

  }
  cp_async_wait<0>();
  __syncthreads();  // the epilogue operands are in shared memory; every role is done

  // ---- y = tot + bias + residual for each consumer warp's 16 columns, written
  // out and kept in tot; per-row sums of y^2 of the warp into rowp[warp]
  T *yout = static_cast<T *>(a.y);
  T *nout = static_cast<T *>(a.normOut);
  const bool cons = warp < ncg && warp < kKmCons;
  if (cons) {
    const int cl = warp;
    const int c0 = 16 * cl + g, c1 = c0 + 8;  // this lane's columns within the CTA's range
    const float b0 = a.bias ? E::to_f(ebias[c0]) : 0.f, b1 = a.bias ? E::to_f(ebias[c1]) : 0.f;
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
      float sq[2];
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const int m = 8 * mt + 4 * r + t;
        float v0 = 0.f, v1 = 0.f;
        if (m < a.M) {
          v0 = tot[mt][r] + b0 + E::to_f(eres[(size_t)m * ncols + c0]);
          v1 = tot[mt][2 + r] + b1 + E::to_f(eres[(size_t)m * ncols + c1]);
          yout[(size_t)m * a.N + 16 * cg0 + c0] = E::from_f(v0);
          yout[(size_t)m * a.N + 16 * cg0 + c1] = E::from_f(v1);
        }
        tot[mt][r] = v0;
        tot[mt][2 + r] = v1;
        sq[r] = fmaf(v0, v0, v1 * v1);
      }
      // the warp's 16 columns of rows 8 mt + t (+4): a fixed tree over g
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        sq[0] += __shfl_xor_sync(0xffffffffu, sq[0], o);
        sq[1] += __shfl_xor_sync(0xffffffffu, sq[1], o);
      }
      if (g == 0) {
        rowp[warp * MP + 8 * mt + t] = sq[0];
        rowp[warp * MP + 8 * mt + 4 + t] = sq[1];
      }
    }
  }
  __syncthreads();
  // the CTA's partial of row m: its warps in order
  if (threadIdx.x < a.M) {
    float v = 0.f;
    for (int w = 0; w < ncg; ++w) v += rowp[w * MP + threadIdx.x];
    __stcg(a.ss + (size_t)threadIdx.x * a.G + cta, v);
  }
  __syncthreads();

  // ---- grid-wide counter: every CTA's row sums are published
  if (threadIdx.x == 0) {
    __threadfence();
    red_release_add(a.gbar, 1u);
    const long long t0 = clock64();
    while (ld_acquire_u32(a.gbar) < (uint32_t)a.G + a.extra) {
      if (clock64() - t0 > a.budget) {
        s_abort = 1;
        record_timeout(a.status, kKmWhereGrid);
        break;
      }
      __nanosleep(32);
    }
  }
  __syncthreads();
  // 1/RMS of row m (warp m % 16): the CTAs' partials, lane-strided loads first,
  // then the sum in CTA order and a fixed shuffle tree
  if (!s_abort) {
    for (int m = warp; m < a.M; m += KW) {
      float pv[kKmParts];
#pragma unroll
      for (int i = 0; i < kKmParts; ++i) {
        const int c = lane + 32 * i;
        pv[i] = c < a.G ? __ldcg(a.ss + (size_t)m * a.G + c) : 0.f;
      }
      float tot2 = 0.f;
#pragma unroll
      for (int i = 0; i < kKmParts; ++i) tot2 += pv[i];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) tot2 += __shfl_xor_sync(0xffffffffu, tot2, o);
      if (lane == 0) s_rstd[m] = rsqrtf(tot2 / (float)a.N + a.eps);
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    // the last CTA through clears the grid counters for the next call
    if (atomicAdd(a.gbar + 1, 1u) == (uint32_t)a.G - 1u) {
      atomicExch(a.gbar, 0u);
      atomicExch(a.gbar + 1, 0u);
    }
  }
  if (s_abort || !cons) return;  // a CTA whose wait gave up writes no normOut
  {
    const int c0 = 16 * warp + g, c1 = c0 + 8;
    const float g0 = E::to_f(egam[c0]), g1 = E::to_f(egam[c1]);
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const int m = 8 * mt + 4 * r + t;
        if (m < a.M) {
          const float rs = s_rstd[m];
          nout[(size_t)m * a.N + 16 * cg0 + c0] = E::from_f(tot[mt][r] * rs * g0);
          nout[(size_t)m * a.N + 16 * cg0 + c1] = E::from_f(tot[mt][2 + r] * rs * g1);
        }
      }
  }
}

}  // namespace
}  // namespace wq
// ------------------------------------------------------------------ host side
namespace wq {
namespace {

using EncodeTiledFnK = PFN_cuTensorMapEncodeTiled_v12000;

EncodeTiledFnK encode_fn_km() {
  static EncodeTiledFnK fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFnK>(p);
    else
      cudaGetLastError();
  });
  return fn;
}

int km_grid(const Problem &p) {
  int sms = device_info().sms > 0 ? device_info().sms : 148;
  if (sms > 32 * kKmParts) sms = 32 * kKmParts;  // the row sums' readers cover that many CTAs
  const int ncg = (int)(p.N / 16);
  return ncg < sms ? ncg : sms;
}

int km_mt(const Problem &p) { return p.M <= 16 ? 2 : (p.M <= 32 ? 4 : 8); }

bool km_a16(const void *q) { return q == nullptr || reinterpret_cast<uintptr_t>(q) % 16 == 0; }

template <int DT, int MT, bool HAS_O>
cudaError_t launch_km_t(const Problem &p, const Plan &plan, void *ws, cudaStream_t s) {
  constexpr int TD = MT == 2 ? 4 : (MT == 4 ? 2 : 1);  // weight slices in flight per warp (registers)
  const int G = plan.grid;
  const uint32_t smem = (uint32_t)km_smem(p, G, MT);
  static cudaError_t attr_err =
      cudaFuncSetAttribute(decode_km_kernel<DT, MT, HAS_O, TD>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)device_info().smem_optin - 2048);
  if (attr_err != cudaSuccess) return attr_err;
  EncodeTiledFnK enc = encode_fn_km();
  if (!enc) return cudaErrorNotSupported;
  CUtensorMap tm_x;
  {
    const cuuint64_t dims[2] = {(cuuint64_t)p.K, (cuuint64_t)p.M};
    const cuuint64_t strides[1] = {(cuuint64_t)p.K * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)(8 * MT)};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(&tm_x, DT == WQ_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
                     const_cast<void *>(p.x1), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  }
  char *wsb = static_cast<char *>(ws);
  KmArgs args = {};
  args.w = static_cast<const uint8_t *>(p.x2);
  args.scale = p.scale; args.offset = p.offset; args.bias = p.bias;
  args.residual = p.residual; args.gamma = p.gamma; args.y = p.y; args.normOut = p.normOut;
  args.status = reinterpret_cast<uint32_t *>(ws);
  args.gbar = reinterpret_cast<uint32_t *>(wsb + kKmGbarOff);
  args.ss = reinterpret_cast<float *>(wsb + kWsHeader);
  args.M = (int)p.M; args.K = (int)p.K; args.N = (int)p.N;
  args.KS2 = (int)(p.K / 128); args.NCG = (int)(p.N / 16);
  args.group = (int)p.group; args.Ns = (int)p.Ns; args.G = G;
  args.eps = p.eps;
  args.budget = wait_budget();
  args.extra = wait_extra_arrivals();
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)G, 1, 1);
  cfg.blockDim = dim3(KTHREADS, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, decode_km_kernel<DT, MT, HAS_O, TD>, tm_x, args);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

bool decode_km_applicable(const Problem &p) {
  if (!p.tiled || p.wbits != 4 || p.M < 9 || p.M > 64) return false;
  if (p.N < 16 || p.N % 16 != 0 || p.K < 128 || p.K % 128 != 0) return false;
  if (p.group != 0 && p.group % 128 != 0) return false;
  const void *v16[] = {p.x1, p.x2, p.bias, p.residual, p.gamma};
  for (const void *q : v16)
    if (!km_a16(q)) return false;
  const void *v2[] = {p.scale, p.offset, p.y, p.normOut};
  for (const void *q : v2)
    if (q && reinterpret_cast<uintptr_t>(q) % 2 != 0) return false;
  const int G = km_grid(p);
  const int64_t ncg_max = (p.N / 16 + G - 1) / G;
  if (ncg_max > kKmCons) return false;
  // with few column groups per CTA most warps idle: up to 16 rows the tiled
  // decode kernel is faster there
  if (p.M <= 16 && ncg_max < 8) return false;
  if (km_smem(p, G, km_mt(p)) + 2048 > (uint64_t)device_info().smem_optin) return false;
  return encode_fn_km() != nullptr;
}

bool plan_decode_km(const Problem &p, Plan &plan) {
  if (!decode_km_applicable(p)) return false;
  plan.kernel = WQ_KERNEL_DECODE;
  plan.mode = kPlanModeKm;
  plan.grid = km_grid(p);
  plan.ws_bytes = kWsHeader + (uint64_t)plan.grid * 64 * 4;
  return true;
}

cudaError_t launch_decode_km(const Problem &p, const Plan &plan, void *ws, cudaStream_t s) {
  const bool o = p.offset != nullptr;
  const int MT = km_mt(p);
  if (p.dtype == WQ_BF16) {
    if (MT == 2) return o ? launch_km_t<WQ_BF16, 2, true>(p, plan, ws, s)
                          : launch_km_t<WQ_BF16, 2, false>(p, plan, ws, s);
    if (MT == 4) return o ? launch_km_t<WQ_BF16, 4, true>(p, plan, ws, s)
                          : launch_km_t<WQ_BF16, 4, false>(p, plan, ws, s);
    return o ? launch_km_t<WQ_BF16, 8, true>(p, plan, ws, s) : launch_km_t<WQ_BF16, 8, false>(p, plan, ws, s);
  }
  if (MT == 2) return o ? launch_km_t<WQ_F16, 2, true>(p, plan, ws, s)
                        : launch_km_t<WQ_F16, 2, false>(p, plan, ws, s);
  if (MT == 4) return o ? launch_km_t<WQ_F16, 4, true>(p, plan, ws, s)
                        : launch_km_t<WQ_F16, 4, false>(p, plan, ws, s);
  return o ? launch_km_t<WQ_F16, 8, true>(p, plan, ws, s) : launch_km_t<WQ_F16, 8, false>(p, plan, ws, s);
}

}  // namespace wq
