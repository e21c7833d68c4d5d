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
// packed INT4 per k-row); K comes in 128-row stages. The nTiles x kst units
// (tile, stage), in tile-major order, are cut into G equal contiguous runs of
// `per` units, one per CTA, G <= SM count, one CTA per SM. A run covers the end
// of one tile and the start of the next (or more), so each CTA produces one
// partial sum per tile it touches (a "segment").
//
// Warp roles (8 consumer warps + 2 producer warps):
//   producers  the last two warps, one elected lane each, stream stages j = p, p+2, ... of
//              the run through a ring as deep as shared memory allows: the 128 x 128-byte box of packed
//              weights, two 64 x MP boxes of x1 (all 128-byte swizzled), and the
//              scale (and offset) rows of the groups the stage touches, all by
//              TMA, completion on the stage's full mbarrier.
//   consumers  column group c (of four) takes 64 columns and k-phase h (of
//              two) the stages with j % 2 == h; the ring depth is even, so a
//              slot always serves the same producer and the same k-phase.
//              Per stage a warp copies its operands to registers (the packed
//              weights of its 64 columns by transposed ldmatrix, so one register
//              pairs k-rows k, k+1 of four columns, and x1 by ldmatrix), hands
//              the slot back when the stage lies in one group, and feeds
//              m16n8k16 MMAs (A = W^T: 16 columns x 16 k; B = x1^T, 16 k x 8
//              rows; fp32 accumulation). One AND/XOR (and a shift) turns a
//              nibble pair into A's 16-bit floats 136 + q (1032 + q in fp16),
//              exact; one more MMA with an all-ones A gives the x1 row sums d of
//              the same rows, and when a group ends its sums are scaled in
//              fp32: tot += S * acc + (O - 136 S) * d. The dequantized weight is
//              never rounded; only fp32 accumulation rounds.
// Segment end. The k-phases add in shared memory (a fixed tree) and the CTA
// writes the segment's M x 256 fp32 partial to the workspace, then counts it on
// the tile's counter. The CTA that brings the counter to the number of
// segments of the tile finishes the tile: it sums the segments in CTA order,
// adds bias and residual, writes y (and y*gamma in fp32 to the workspace) and
// the tile's per-row sum of y^2, and clears the counter for the next call.
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
constexpr int DKB = 128;                    // k-rows per stage
constexpr uint32_t DW = DKB * DNT / 2;      // 16 KB of packed INT4 per stage
constexpr int kMaxSoRows = 4;               // group rows a 128-row stage can touch (group >= 32)
constexpr int kMaxStages = 16;              // ring depth bound (barrier storage)
constexpr int kProducers = 2;               // producer warps (alternate stages)
constexpr int kTileCounters = 256;          // N <= 65535 gives at most 256 tiles
constexpr uint32_t kGbarOff = 128;          // header: grid counters (arrive, depart)
constexpr uint32_t kTcntOff = 1024;         // header: per-tile segment counters
constexpr int kRingMultiple = 2;            // ring depth: a multiple of producers and k-phases

template <int MT>
struct DCfg {
  static constexpr int MP = 8 * MT;                // rows held (x1 box height)
  static constexpr int CPW = 64;                   // columns per consumer warp
  static constexpr int NCG = DNT / CPW;            // column groups
  static constexpr int CW = 8;                     // consumer warps
  static constexpr int KH = CW / NCG;              // k-phases
  static constexpr int CT = CW * 32;               // consumer threads
  static constexpr int THREADS = CT + 32 * kProducers;
  static constexpr uint32_t XB = MP * 128;         // one 64-k x1 box
  static_assert(KH * NCG == CW && KH == 2, "warp split");
  static_assert(kRingMultiple % KH == 0 && kRingMultiple % kProducers == 0,
                "a ring slot keeps one producer and one k-phase");
  static_assert((MP * DNT / 4) % 32 == 0 && CT % 32 == 0, "tile positions come in whole warps");
};

// Shared-memory layout of one call (the ring depth follows from the slot size).
struct DLayout {
  uint32_t slot, off_x, off_s, off_o, off_red, off_misc, off_bar, smem;
  int NS;
};

inline DLayout decode_layout(int MT, int so_rows, bool has_o, uint32_t budget) {
  DLayout L;
  const uint32_t MP = 8u * MT, XB = MP * 128u;
  L.off_x = DW;                              // slot: W | two x1 boxes | S rows | O rows
  L.off_s = DW + 2 * XB;
  L.off_o = L.off_s + (uint32_t)so_rows * DNT * 2u;
  const uint32_t end = L.off_o + (has_o ? (uint32_t)so_rows * DNT * 2u : 0u);
  L.slot = (end + 1023u) / 1024u * 1024u;    // keeps the 128-byte swizzle atoms aligned
  const uint32_t fixed = 2u * MP * DNT * 4u  // k-phase reduction buffer
                         + 2048u             // misc: 1/RMS, per-warp row sums, flags
                         + 8u * 2u * kMaxStages + 1024u;  // barriers, base alignment slack
  int ns = (int)((budget - fixed) / L.slot);
  // Each slot must belong to one producer and to one k-phase for good: stage j
  // goes to slot j % NS, producer j % 2 and k-phase j % KH. A k-phase that
  // waited on a slot last filled for another k-phase could run a whole phase
  // ahead of it, and a parity wait cannot tell phase p from phase p + 2.
  ns -= ns % kRingMultiple;
  if (ns > kMaxStages) ns = kMaxStages;
  L.NS = ns;
  L.off_red = (uint32_t)ns * L.slot;
  L.off_misc = L.off_red + 2u * MP * DNT * 4u;
  L.off_bar = L.off_misc + 2048u;
  L.smem = L.off_bar + 8u * 2u * kMaxStages + 1024u;
  return L;
}

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
  int M, K, N, group, Ns, so_rows;
  int nTiles, kst, U, per, G, SMAX, npf;
  float eps;
  long long budget;   // cycles the grid barrier waits before it gives up
  uint32_t extra;     // arrivals the grid barrier waits for beyond G (0; > 0 only in tests)
  int NS;                                      // ring depth
  uint32_t slot, off_x, off_s, off_o, off_red, off_misc, off_bar;  // shared-memory layout
};

// One A-fragment register from a transposed ldmatrix word r: r holds the 16-bit
// group of four columns (nibble c = column 4e + c) of k-rows k (low half) and
// k + 1 (high half); nibble c of both halves becomes the 16-bit float 136 + q
// (bf16) or 1032 + q (fp16): (nib ^ 8) | magic is exactly that float.
template <int DT>
__device__ __forceinline__ uint32_t nib_col(uint32_t r, int c) {
  constexpr uint32_t MAGIC = DT == WQ_BF16 ? 0x43084308u : 0x64086408u;
  return ((c ? r >> (4 * c) : r) & 0x000F000Fu) ^ MAGIC;
}

// Four consecutive 16-bit values at addr -> f[0..3].
template <int DT>
__device__ __forceinline__ void lds4f(uint32_t addr, float *f) {
  uint32_t v0, v1;
  asm volatile("ld.shared.v2.b32 {%0,%1}, [%2];" : "=r"(v0), "=r"(v1) : "r"(addr));
  const float2 p = unpack2<DT>(v0), q = unpack2<DT>(v1);
  f[0] = p.x; f[1] = p.y; f[2] = q.x; f[3] = q.y;
}

template <int DT, int MT, bool HAS_O>
__global__ void __launch_bounds__(DCfg<MT>::THREADS, 1)
    decode_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_x,
                  const __grid_constant__ CUtensorMap tm_s, const __grid_constant__ CUtensorMap tm_o,
                  const DecodeArgs a) {
  using C = DCfg<MT>;
  using E = Elem<DT>;
  using T = typename E::T;
  constexpr int MP = C::MP, KH = C::KH, CT = C::CT, CPW = C::CPW;
  constexpr int NB = DKB / 16;  // 16-k blocks per stage
  constexpr bool BF = DT == WQ_BF16;
  extern __shared__ uint8_t dsm_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(dsm_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_u32(smem);
  const int NS = a.NS;
  auto FULL = [&](int s) { return sb + a.off_bar + 8u * s; };
  auto EMPTY = [&](int s) { return sb + a.off_bar + 8u * (kMaxStages + s); };
  float *red = reinterpret_cast<float *>(smem + a.off_red);
  float *misc = reinterpret_cast<float *>(smem + a.off_misc);
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
      mbar_init(EMPTY(s), C::NCG);  // the column-group warps of the stage's k-phase
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
    int tile = u0 / a.kst, st = u0 - tile * a.kst;
    for (int j = 0; j < npf; ++j) {
      tma_prefetch_l2_2d(&tm_w, tile * (DNT / 2), st * DKB);
      if (++st == a.kst) { st = 0; ++tile; }
    }
  }
  __syncthreads();
  griddep_wait();  // the previous grid on the stream has finished and flushed
  griddep_launch_dependents();

  if (warp >= C::CW) {
    // ---------------------------------------------------------------- producers
    const int p = warp - C::CW;
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();  // each weight byte is used once per call
      const uint32_t so_bytes = a.Ns != 1 ? (uint32_t)a.so_rows * DNT * 2u : 0u;
      const uint32_t bytes = DW + 2u * C::XB + (HAS_O ? 2u : 1u) * so_bytes;
      int slot = p;
      uint32_t ph = 0;
      int issued = 0;
      int tile = (u0 + p) / a.kst, st = (u0 + p) - tile * a.kst;
      for (int u = u0 + p; u < u1; u += kProducers) {
        if (!wait_bar(EMPTY(slot), ph ^ 1u, abort_flag, a.status, kDWhereProducer)) break;
        const int row0 = st * DKB;
        const uint32_t dst = sb + (uint32_t)slot * a.slot;
        mbar_arrive_expect_tx(FULL(slot), bytes);
        tma_load_2d_hint(dst, &tm_w, tile * (DNT / 2), row0, FULL(slot), pol);
        tma_load_2d(dst + a.off_x, &tm_x, row0, 0, FULL(slot));
        tma_load_2d(dst + a.off_x + C::XB, &tm_x, row0 + 64, 0, FULL(slot));
        if (a.Ns != 1) {
          // the scale (and offset) rows of the groups this stage touches
          const int g0 = a.group ? row0 / a.group : 0;
          tma_load_2d(dst + a.off_s, &tm_s, tile * DNT, g0, FULL(slot));
          if (HAS_O) tma_load_2d(dst + a.off_o, &tm_o, tile * DNT, g0, FULL(slot));
        }
        ++issued;
        slot += kProducers;
        if (slot >= NS) { slot -= NS; ph ^= 1u; }
        st += kProducers;
        while (st >= a.kst) { st -= a.kst; ++tile; }
      }
      // every copy issued has landed before the CTA may exit
      int dslot = p;
      uint32_t dph = 0;
      for (int q = 0; q < issued; ++q) {
        if (q + NS / kProducers >= issued) drain_bar(FULL(dslot), dph);
        dslot += kProducers;
        if (dslot >= NS) { dslot -= NS; dph ^= 1u; }
      }
    }
    __syncwarp();
    return;
  }

  // ------------------------------------------------------------------ consumers
  const int ctid = threadIdx.x;
  const int cg = warp % C::NCG, kh = warp / C::NCG;  // column group, k-phase
  const int g = lane >> 2, t = lane & 3;
  const uint32_t ones = BF ? 0x3F803F80u : 0x3C003C00u;      // 1.0 in both halves
  const float bias136 = BF ? 136.f : 1032.f;                  // A = bias136 + q
  const T *bias = static_cast<const T *>(a.bias);
  const T *res = static_cast<const T *>(a.residual);
  const T *gam = static_cast<const T *>(a.gamma);
  T *yout = static_cast<T *>(a.y);
  T *nout = static_cast<T *>(a.normOut);

  // Columns of the warp: cb .. cb + 63, in 16-bit groups of four (element e =
  // columns 4e .. 4e+3). A transposed ldmatrix.x4 of 16 k-rows gives lane (g, t)
  // the elements 16cg + g (matrices 0, 2) and 16cg + 8 + g (matrices 1, 3) of
  // k-rows 2t, 2t+1 (matrices 0, 1) and 2t+8, 2t+9 (matrices 2, 3). MMA tile c
  // (of four) takes nibble c of each: its row g is column cb + 4g + c and its
  // row g + 8 is column cb + 32 + 4g + c.
  const int cb = cg * CPW;
  static_assert(CPW == 64, "four 16-column MMA tiles per warp");
  uint32_t wlane;  // this lane's row address offset within a 16-row block, swizzled
  {
    const int mi = lane >> 3, rr = lane & 7;
    const uint32_t chunk = 2u * cg + (uint32_t)(mi & 1);
    wlane = (uint32_t)(8 * (mi >> 1) + rr) * 128u + ((chunk ^ (uint32_t)rr) << 4);
  }
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
  // a stage whose rows lie in one group can be copied to registers and handed
  // back to the producer before any arithmetic
  const bool early = a.so_rows == 1;

  const int t0c = u0 / a.kst;                   // first tile of this CTA's run
  const int t1c = u1 > u0 ? (u1 - 1) / a.kst : t0c - 1;
  int fin_tiles[4];
  int nfin = 0;
  int j = 0, jph = 0, slot = 0;  // jph = j % KH
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
    // scale / offset of this thread's 8 columns in scale row `row` of a stage
    // copy: sf[c] is column cb + 4g + c, sf[4 + c] column cb + 32 + 4g + c
    auto load_so = [&](uint32_t base, int row, float (&sf)[8], float (&of)[8]) {
      if (a.Ns == 1) {
#pragma unroll
        for (int q = 0; q < 8; ++q) { sf[q] = sscal; of[q] = oscal; }
      } else {
        const uint32_t o = (uint32_t)(row * DNT + cb + 4 * g) * 2u;
        lds4f<DT>(base + a.off_s + o, sf);
        lds4f<DT>(base + a.off_s + o + 64u, sf + 4);
        if constexpr (HAS_O) {
          lds4f<DT>(base + a.off_o + o, of);
          lds4f<DT>(base + a.off_o + o + 64u, of + 4);
        } else {
#pragma unroll
          for (int q = 0; q < 8; ++q) of[q] = 0.f;
        }
      }
    };
    // fold the group's sums into tot. A holds 136 + q (1032 + q in fp16) and d
    // the x1 row sums of the same k-rows, so the group's exact sum is
    // S * (acc - 136 d) + O * d = S * acc + (O - 136 S) * d.
    auto flush = [&](const float (&sf)[8], const float (&of)[8]) {
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const float sl = sf[c], sh = sf[4 + c];  // rows g, g + 8 of MMA tile c
        const float cl = fmaf(-bias136, sl, of[c]);
        const float ch = fmaf(-bias136, sh, of[4 + c]);
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          tot[mt][c][0] = fmaf(cl, d1[mt][0], fmaf(sl, acc[mt][c][0], tot[mt][c][0]));
          tot[mt][c][1] = fmaf(cl, d1[mt][1], fmaf(sl, acc[mt][c][1], tot[mt][c][1]));
          tot[mt][c][2] = fmaf(ch, d1[mt][0], fmaf(sh, acc[mt][c][2], tot[mt][c][2]));
          tot[mt][c][3] = fmaf(ch, d1[mt][1], fmaf(sh, acc[mt][c][3], tot[mt][c][3]));
#pragma unroll
          for (int e = 0; e < 4; ++e) acc[mt][c][e] = 0.f;
        }
      }
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) d1[mt][0] = d1[mt][1] = 0.f;
    };

    for (int st = sbeg; st < send; ++st) {
      if (jph == kh) {
        const bool ok = wait_bar_warp(FULL(slot), ph, abort_flag, a.status, kDWhereConsumer);
        bool released = false;
        if (ok) {
          const uint32_t base = sb + (uint32_t)slot * a.slot;
          const int srow = st * DKB;
          // the stage's operands of this warp, all loaded before any arithmetic:
          // the packed weights by transposed ldmatrix (16 k-rows x 64 columns
          // per kb) and B = x1^T (box kb/4; row m at m*128, chunk c at c ^ (m & 7))
          uint32_t w[NB][4], b[NB][MT][2];
#pragma unroll
          for (int kb = 0; kb < NB; ++kb) {
            ldmatrix_x4_trans(base + (uint32_t)kb * 2048u + wlane, w[kb][0], w[kb][1], w[kb][2],
                              w[kb][3]);
            const int cidx = 2 * (kb & 3) + ldm_c;
            const uint32_t baddr = base + a.off_x + (uint32_t)(kb >> 2) * C::XB +
                                   (uint32_t)ldm_m * 128u + ((uint32_t)(cidx ^ (ldm_m & 7)) << 4);
            if constexpr (MT == 2)
              ldmatrix_x4(baddr, b[kb][0][0], b[kb][0][1], b[kb][1][0], b[kb][1][1]);
            else
              ldmatrix_x2(baddr, b[kb][0][0], b[kb][0][1]);
          }
          float sf[8], of[8];
          load_so(base, 0, sf, of);
          if (early) {
            __syncwarp();
            if (lane == 0) mbar_arrive(EMPTY(slot));  // the arrive orders the loads before it
            released = true;
          }
          const int gs = a.group ? srow / a.group : 0;  // group of the stage's first row
          int cur = gs;
          int gend = (!early && a.group) ? (gs + 1) * a.group : 0x7fffffff;
#pragma unroll
          for (int kb = 0; kb < NB; ++kb) {
            const int row0 = srow + 16 * kb;
            if (row0 >= gend) {  // group boundary inside a stage that is still held
              if (cur - gs < a.so_rows) flush(sf, of);
              ++cur;
              gend += a.group;
              if (cur - gs < a.so_rows) load_so(base, cur - gs, sf, of);
            }
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              const uint32_t a0 = nib_col<DT>(w[kb][0], c), a1 = nib_col<DT>(w[kb][1], c);
              const uint32_t a2 = nib_col<DT>(w[kb][2], c), a3 = nib_col<DT>(w[kb][3], c);
#pragma unroll
              for (int mt = 0; mt < MT; ++mt)
                mma_16816<BF>(acc[mt][c], a0, a1, a2, a3, b[kb][mt][0], b[kb][mt][1]);
            }
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {  // d: x1 row sums of the block (A = all ones)
              float dd[4] = {d1[mt][0], d1[mt][1], d1[mt][0], d1[mt][1]};
              mma_16816<BF>(dd, ones, ones, ones, ones, b[kb][mt][0], b[kb][mt][1]);
              d1[mt][0] = dd[0];
              d1[mt][1] = dd[1];
            }
          }
          // a group past the copied scale rows lies wholly beyond K: its sums are zero
          if (cur - gs < a.so_rows) flush(sf, of);
        }
        __syncwarp();
        if (!released && lane == 0) mbar_arrive(EMPTY(slot));
      }
      ++j;
      if (++jph == KH) jph = 0;
      if (++slot == NS) { slot = 0; ph ^= 1u; }
    }

    // ---- segment end: the k-phases add in shared memory, the partial goes out
    auto red_idx = [&](int mt, int c, int e) {  // MMA tile c, accumulator element e
      return (8 * mt + 2 * t + (e & 1)) * DNT + cb + 32 * (e >> 1) + 4 * g + c;
    };
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int c = 0; c < 4; ++c) red[kh * MP * DNT + red_idx(mt, i, c)] = tot[mt][i][c];
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
    // Every CTA fetches the residual, bias and gamma of the positions it would
    // finish now, so a finisher does not wait for them after the partial sums.
    // Position qq of this thread is float4 q = ctid + CT*qq: columns 4q' .. 4q'+3
    // of row m = q / 64 (N % 32 == 0: all four columns or none).
    constexpr int NQ = MP * DNT / 4;                 // float4 positions of a tile
    constexpr int QPT = (NQ + CT - 1) / CT;          // per thread (warp-uniform tail)
    uint2 rres[QPT], rbia[QPT], rgam[QPT];
#pragma unroll
    for (int qq = 0; qq < QPT; ++qq) {
      const int q = ctid + CT * qq;
      const int m = q / (DNT / 4), n = tile * DNT + 4 * (q - m * (DNT / 4));
      rres[qq] = rbia[qq] = rgam[qq] = make_uint2(0u, 0u);
      if (q < NQ && m < a.M && n < a.N) {
        rres[qq] = __ldg(reinterpret_cast<const uint2 *>(res + (int64_t)m * a.N + n));
        if (bias) rbia[qq] = __ldg(reinterpret_cast<const uint2 *>(bias + n));
        rgam[qq] = __ldg(reinterpret_cast<const uint2 *>(gam + n));
      }
    }
    // the CTA barrier orders every thread's partial stores before thread 0's
    // release; the finisher's acquire then orders them before its loads
    named_bar_sync(1, CT);
    if (ctid == 0) {
      const int c_first = (tile * a.kst) / a.per;
      const int c_last = ((tile + 1) * a.kst - 1) / a.per;
      const uint32_t old = atom_add_acq_rel(a.tcnt + tile, 1u);
      *s_fin = old == (uint32_t)(c_last - c_first);
    }
    named_bar_sync(1, CT);
    const bool finisher = *s_fin != 0;
    if (finisher) {
      // ---- finish the tile: segments in CTA order + bias + residual -> y, sum(y^2)
      const int c_first = (tile * a.kst) / a.per;
      const int c_last = ((tile + 1) * a.kst - 1) / a.per;
      const int nseg = c_last - c_first + 1;
      for (int q = ctid; q < C::CW * 16; q += CT) s_ssw[q] = 0.f;
      float4 v[QPT];
#pragma unroll
      for (int qq = 0; qq < QPT; ++qq) v[qq] = make_float4(0.f, 0.f, 0.f, 0.f);
      constexpr int EB = MT == 1 ? 8 : 4;  // segment loads per position in flight at once
      for (int e0 = 0; e0 < nseg; e0 += EB) {
        float4 pv[QPT][EB];
#pragma unroll
        for (int e = 0; e < EB; ++e) {
          const int cc = c_first + e0 + e;
          const bool live = e0 + e < nseg;
          const int seg = live ? tile - (cc * a.per) / a.kst : 0;
          const float4 *src = reinterpret_cast<const float4 *>(
              a.part + ((int64_t)(live ? cc : c_first) * a.SMAX + seg) * (MP * DNT));
#pragma unroll
          for (int qq = 0; qq < QPT; ++qq)
            pv[qq][e] = (live && ctid + CT * qq < NQ) ? __ldcg(src + ctid + CT * qq)
                                                      : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int qq = 0; qq < QPT; ++qq)
#pragma unroll
          for (int e = 0; e < EB; ++e) {  // added in CTA order
            v[qq].x += pv[qq][e].x; v[qq].y += pv[qq][e].y;
            v[qq].z += pv[qq][e].z; v[qq].w += pv[qq][e].w;
          }
      }
      named_bar_sync(1, CT);  // s_ssw cleared
#pragma unroll
      for (int qq = 0; qq < QPT; ++qq) {
        const int q = ctid + CT * qq;
        if (q >= NQ) break;  // whole warps (NQ and CT are multiples of 32)
        const int m = q / (DNT / 4), n = tile * DNT + 4 * (q - m * (DNT / 4));
        float yv[4] = {0.f, 0.f, 0.f, 0.f}, yg[4] = {0.f, 0.f, 0.f, 0.f};
        if (m < a.M && n < a.N) {
          const float2 r01 = unpack2<DT>(rres[qq].x), r23 = unpack2<DT>(rres[qq].y);
          const float2 b01 = unpack2<DT>(rbia[qq].x), b23 = unpack2<DT>(rbia[qq].y);
          const float2 g01 = unpack2<DT>(rgam[qq].x), g23 = unpack2<DT>(rgam[qq].y);
          yv[0] = v[qq].x + b01.x + r01.x;
          yv[1] = v[qq].y + b01.y + r01.y;
          yv[2] = v[qq].z + b23.x + r23.x;
          yv[3] = v[qq].w + b23.y + r23.y;
          yg[0] = yv[0] * g01.x; yg[1] = yv[1] * g01.y; yg[2] = yv[2] * g23.x; yg[3] = yv[3] * g23.y;
          *reinterpret_cast<uint2 *>(yout + (int64_t)m * a.N + n) =
              make_uint2(pack2<DT>(yv[0], yv[1]), pack2<DT>(yv[2], yv[3]));
        }
        // y * gamma in fp32: normOut needs only 1/RMS more
        __stcg(reinterpret_cast<float4 *>(a.y32 + (int64_t)tile * (MP * DNT)) + q,
               make_float4(yg[0], yg[1], yg[2], yg[3]));
        float sq = yv[0] * yv[0] + yv[1] * yv[1] + yv[2] * yv[2] + yv[3] * yv[3];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, o);
        if (lane == 0) s_ssw[warp * 16 + m] += sq;  // a warp shares one row m
      }
      named_bar_sync(1, CT);
      if (ctid < MP) {
        float sv = 0.f;
        for (int w = 0; w < C::CW; ++w) sv += s_ssw[w * 16 + ctid];
        __stcg(a.ss + tile * 16 + ctid, sv);
      }
      if (ctid == 0) a.tcnt[tile] = 0u;  // the last user of this counter in this call
      if (nfin < 4) fin_tiles[nfin] = tile;
      ++nfin;
    }
  }

  // ---- grid barrier, then 1/RMS per row and normOut of the tiles this CTA finished
  named_bar_sync(1, CT);
  if (ctid == 0) {
    red_release_add(a.gbar, 1u);
    const long long t0 = clock64();
    while (ld_acquire_u32(a.gbar) < (uint32_t)a.G + a.extra) {
      if (*abort_flag) break;
      if (clock64() - t0 > a.budget) {
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
  // a CTA whose wait gave up (or whose producers did) writes no normOut
  for (int f = 0; f < nfin && f < 4 && !*abort_flag; ++f) {
    const int tile = fin_tiles[f];
    for (int q = ctid; q < MP * DNT / 4; q += CT) {
      const int m = q / (DNT / 4), col = 4 * (q - m * (DNT / 4));
      const int n = tile * DNT + col;
      if (m < a.M && n < a.N) {
        const float4 yg = __ldcg(reinterpret_cast<const float4 *>(a.y32 + (int64_t)tile * (MP * DNT)) + q);
        const float rs = s_rstd[m];
        *reinterpret_cast<uint2 *>(nout + (int64_t)m * a.N + n) =
            make_uint2(pack2<DT>(yg.x * rs, yg.y * rs), pack2<DT>(yg.z * rs, yg.w * rs));
      }
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

// Scale rows one stage's TMA copies: the most group rows any 128-row stage
// touches (1 for per-channel scales).
int decode_so_rows(const Problem &p) {
  if (p.smode != kPerGroup) return 1;
  const int64_t kst = (p.K + DKB - 1) / DKB;
  int64_t most = 1;
  for (int64_t s = 0; s < kst; ++s) {
    const int64_t r0 = s * DKB, r1 = (s + 1) * DKB < p.K ? (s + 1) * DKB : p.K;
    const int64_t n = (r1 - 1) / p.group - r0 / p.group + 1;
    if (n > most) most = n;
  }
  return (int)(most < p.G ? most : p.G);
}

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
  // the epilogue moves four 16-bit values at a time
  const void *vecs[] = {p.bias, p.residual, p.gamma, p.y, p.normOut};
  for (const void *q : vecs)
    if (reinterpret_cast<uintptr_t>(q) % 8 != 0) return false;
  const int so_rows = decode_so_rows(p);
  if (so_rows > kMaxSoRows) return false;
  const uint32_t budget = device_info().smem_optin > 0 ? (uint32_t)device_info().smem_optin : 232448u;
  if (decode_layout(p.M <= 8 ? 1 : 2, so_rows, p.offset != nullptr && p.Ns != 1, budget).NS < 4)
    return false;
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
  const uint32_t budget = (uint32_t)device_info().smem_optin;
  static std::once_flag attr_once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(attr_once, [budget] {
    // the cap is the device's opt-in maximum; each call asks for its own layout's size
    attr_err = cudaFuncSetAttribute(decode_kernel<DT, MT, HAS_O>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, (int)budget);
  });
  if (attr_err != cudaSuccess) return attr_err;
  const DecodeGeom gm = decode_geom(p);
  if (gm.G > device_info().sms) return cudaErrorInvalidConfiguration;
  const int so_rows = decode_so_rows(p);
  const DLayout L = decode_layout(MT, so_rows, HAS_O && p.Ns != 1, budget);
  if (L.NS < 4 || L.smem > budget) return cudaErrorInvalidConfiguration;

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
    const cuuint32_t box[2] = {64, (cuuint32_t)C::MP};  // 128-byte rows: two boxes per stage
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
    const cuuint32_t box[2] = {DNT, (cuuint32_t)so_rows};
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
  args.so_rows = so_rows;
  args.nTiles = gm.nTiles; args.kst = gm.kst; args.U = gm.U; args.per = gm.per; args.G = gm.G;
  args.SMAX = gm.SMAX;
  args.npf = gm.per < 16 ? gm.per : 16;
  args.eps = p.eps;
  args.budget = wait_budget();
  args.extra = wait_extra_arrivals();
  args.NS = L.NS;
  args.slot = L.slot; args.off_x = L.off_x; args.off_s = L.off_s; args.off_o = L.off_o;
  args.off_red = L.off_red; args.off_misc = L.off_misc; args.off_bar = L.off_bar;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)gm.G, 1, 1);
  cfg.blockDim = dim3(C::THREADS, 1, 1);
  cfg.dynamicSmemBytes = L.smem;
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
