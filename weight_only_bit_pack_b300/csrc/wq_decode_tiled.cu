// Small-M (decode) kernel of the fused operator for weights in the kernel-native
// tiled INT4 layout (aclnnWeightQuantMatmulAllReduceAddRmsNorm, "Function
// description": mm_out = x1 @ (x2*antiquantScale + antiquantOffset) + bias;
// y = mm_out + residual; normOut = y / RMS(y) * gamma; the tiled weight is the
// pack's matrix-unit output, aclnnConvertWeightToINT4Pack).
//
// With M <= 16 the operator streams the weight once; everything here is built
// around keeping HBM busy with few instructions per weight byte.
//
// Work split. Column groups of 16 (one tile column) are dealt out to the CTAs
// in contiguous, balanced ranges, so every CTA owns whole output columns for the
// whole of K: no partial sums cross CTAs. Inside a CTA the units -- a pair of
// neighbouring column groups at one 64-row k-step -- are cut into 16 equal
// contiguous runs in (pair, k-step) order, one per warp; a run spans at most
// two pairs, and its partial sums are reduced in shared memory in warp order.
//
// Per unit a lane loads its 16 bytes of each of the two tiles (coalesced: a
// warp reads the 512-byte tiles whole) and its activations (two 16-byte runs per
// 8 rows of x1), turns each weight word into four A registers (one shift and one
// AND/XOR each build the 16-bit float 136 + q, or 1032 + q in fp16, exactly),
// and issues m16n8k16 MMAs with A = W^T and B = x1^T, fp32 accumulation; one
// all-ones MMA per 16 k-rows, shared by the pair's two tiles, gives the x1 row
// sums d of the same k-rows. Weights are loaded TD units ahead; the scale (and
// offset) values a unit needs come TD units ahead too, by cp.async into a small
// per-warp ring, so no group boundary waits on memory. A group's sums are
// scaled when the group ends: with A = 136 + q its exact sum is
// S * (acc - 136 d) + O * d = S * acc + (O - 136 S) * d.
//
// Epilogue: the CTA adds bias and residual, writes y, keeps y in fp32 in shared
// memory and publishes its per-row sum of y^2; after a grid-wide counter (all
// CTAs are resident: one per SM at most) every CTA sums those partials in CTA
// order, forms 1/RMS per row and writes normOut for its columns. All reductions
// run in a fixed order, so results are bitwise reproducible. Every wait is
// bounded; a wait that gives up records WQ_ERR_DEVICE_TIMEOUT and the kernel
// writes no normOut.
#include "wq_common.cuh"
#include "wq_internal.h"
#include "wq_sm100.cuh"
#include "wq_sync.cuh"
#include "wq_tiled_frag.cuh"

namespace wq {
namespace {

using namespace sm100;
using namespace tfrag;

constexpr int TW = 16;              // warps per CTA
constexpr int TTHREADS = TW * 32;
constexpr int TSL = 2;              // pairs a warp's run can touch
constexpr int TSLG = 3;             // group-structured loop: column groups a run can touch
constexpr uint32_t kTGbarOff = 128; // header: grid counters (arrive, depart)
enum TWhere : uint32_t { kTWhereGrid = 15 };
constexpr int kTParts = 5;          // per-CTA partial sums a lane reads: grid <= 160

struct DTArgs {
  const void *x1;
  const uint8_t *w;
  const void *scale, *offset, *bias, *residual, *gamma;
  void *y, *normOut;
  uint32_t *status, *gbar;
  float *ss;          // 16 x G per-CTA sums of y^2, row-major by row (a row's CTAs contiguous)
  int M, K, N, KS, NCG, group, Ns, G;
  int gu, GV;         // group-structured loop: k-steps per group, groups along K
  int G_rows;         // scale rows (ceil(K / group) per-group, else 1)
  float eps;
  long long budget;
  uint32_t extra;
};

// GRP: the group-structured main loop (K % 128 == 0 and scale groups of whole
// 128-row units, or one scale row cut into groups of one unit); UG1: one unit
// per group, so every unit starts its sums from zero and folds them. Otherwise
// the general loop: 32-row blocks, any group that is a multiple of 32, any K.
template <int DT, int MT, bool HAS_O, int TD, bool KFULL, bool XSMEM, bool GRP, bool UG1 = false>
__global__ void __launch_bounds__(TTHREADS, 1) decode_tiled_kernel(const DTArgs a) {
  static_assert(!GRP || KFULL, "the group-structured loop needs K % 64 == 0");
  constexpr int TRING = TD + 1;  // scale ring slots per warp
  using E = Elem<DT>;
  using T = typename E::T;
  constexpr bool BF = DT == WQ_BF16;
  constexpr int MP = 8 * MT;
  constexpr int SLOT_FLOATS = 2 * MP * 16;             // one pair's partial sums
  constexpr int RING_BYTES = (HAS_O ? 2 : 1) * 8 * 16;  // one unit's scale (offset) chunks

  extern __shared__ __align__(16) uint8_t tsm[];
  float *part = reinterpret_cast<float *>(tsm);                          // [TW][TSL][SLOT]
  uint8_t *ring = tsm + TW * TSL * SLOT_FLOATS * 4;                      // [TW][TRING][RING_BYTES]
  float *ysm = reinterpret_cast<float *>(ring + TW * TRING * RING_BYTES);  // [MP][ncols]
  // the CTA's residual rows, bias and gamma (16 columns per group), fetched at
  // the start so the epilogue does not wait on memory
  const int ncg_max = (a.NCG + a.G - 1) / a.G;  // the host sizes these for this many groups
  T *eres = reinterpret_cast<T *>(ysm + (size_t)MP * ncg_max * 16);  // [M][ncols]
  T *ebias = eres + (size_t)a.M * ncg_max * 16;                       // [ncols]
  T *egam = ebias + (size_t)ncg_max * 16;                             // [ncols]
  // per 32-row block of K: its scale row, and bit 15 = a group ends with it
  uint16_t *kblk = reinterpret_cast<uint16_t *>(egam + (size_t)ncg_max * 16);
  // XSMEM: the M rows of x1, row pitch 2K + 64 bytes (16-byte aligned, and the
  // 8 rows a warp reads at once fall in distinct bank groups)
  const uint32_t xpitch = 2u * (uint32_t)a.K + 64u;
  // GRP: the x1 row sums of every group, [GV][MP], and the CTA's scale (then
  // offset) rows, [G_rows][ncg_max * 16] each
  float *dsm = reinterpret_cast<float *>(
      (reinterpret_cast<uintptr_t>(kblk + (a.K + 31) / 32) + 15) & ~static_cast<uintptr_t>(15));
  T *ssm = reinterpret_cast<T *>(
      (reinterpret_cast<uintptr_t>(dsm + (GRP ? a.GV * MP : 0)) + 15) & ~static_cast<uintptr_t>(15));
  const size_t ssm_elems = GRP ? (size_t)(a.Ns == 1 ? 0 : a.G_rows) * ncg_max * 16 * (HAS_O ? 2 : 1) : 0;
  uint8_t *xsm = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(ssm + ssm_elems) + 15) & ~static_cast<uintptr_t>(15));
  __shared__ __align__(8) uint64_t s_xbar;
  __shared__ int s_tag[TW][TSLG];
  __shared__ float s_rstd[16];
  __shared__ int s_abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int cta = blockIdx.x;
  const int cg0 = (int)((long long)cta * a.NCG / a.G);
  const int cg1 = (int)((long long)(cta + 1) * a.NCG / a.G);
  const int ncols = 16 * (cg1 - cg0);
  const int ncp = (cg1 - cg0 + 1) / 2;
  const int U = ncp * a.KS;
  const int r0 = (int)((long long)U * warp / TW), r1 = (int)((long long)U * (warp + 1) / TW);
  const T *x1 = static_cast<const T *>(a.x1);
  const size_t slab = (size_t)a.NCG * 512;  // bytes of one 64-row slab of tiles

  if (threadIdx.x < TW * TSLG) s_tag[threadIdx.x / TSLG][threadIdx.x % TSLG] = -1;
  if (threadIdx.x == 0) s_abort = 0;
  for (int j = threadIdx.x; j < (a.K + 31) / 32; j += TTHREADS) {
    const int k0 = 32 * j;
    const int row = a.group ? k0 / a.group : 0;
    const bool ends = a.group && ((k0 + 32) % a.group == 0 || k0 + 32 >= a.K);
    kblk[j] = (uint16_t)(row | (ends ? 0x8000 : 0));
  }
  if (XSMEM && threadIdx.x == 0) {
    mbar_init(smem_u32(&s_xbar), 1);
    fence_mbar_init();
  }
  __syncthreads();  // tags cleared and the table built before any warp uses them

  griddep_wait();  // the previous kernel on the stream has finished and flushed
  griddep_launch_dependents();
  {  // epilogue operands: 16-byte chunks, two per column group and row
    const int cpr = 2 * (cg1 - cg0);  // chunks per row
    const T *bias = static_cast<const T *>(a.bias);
    for (int i = threadIdx.x; i < (a.M + 2) * cpr; i += TTHREADS) {
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
    cp_async_commit();  // the oldest group: complete before any ring wait returns
  }
  if (XSMEM && threadIdx.x == 0) {
    mbar_arrive_expect_tx(smem_u32(&s_xbar), (uint32_t)(a.M * 2 * a.K));
    for (int m = 0; m < a.M; ++m)
      bulk_copy_g2s(smem_u32(xsm + (size_t)m * xpitch), x1 + (size_t)m * a.K, 2u * (uint32_t)a.K,
                    smem_u32(&s_xbar));
  }

  if constexpr (!GRP) {
  // ---- unit (pair p, k-step s), fetched TD units ahead of its use: the lane's
  // 16 bytes of the pair's two tiles, an L1 prefetch of the activation lines
  // the unit will read (rows g and 8 + g, k-rows 64s..64s+63), and the scale
  // (offset) rows by cp.async into ring slot `slot`: chunk q of lanes 0..7
  // (8..15 for offsets) = (half h, column group c, 8-column half)
  const uint32_t ring_w = smem_u32(ring) + (uint32_t)(warp * TRING * RING_BYTES);
  // this lane's activation rows 8 mt + g at k-offset 8t; a row past M reads row
  // M - 1 instead (its outputs are never stored)
  const T *xrow[MT];
  uint32_t xsrow[MT];  // the same rows in the staged copy (XSMEM)
#pragma unroll
  for (int mt = 0; mt < MT; ++mt) {
    const int m = 8 * mt + g < a.M ? 8 * mt + g : a.M - 1;
    xrow[mt] = x1 + (size_t)m * a.K + 8 * t;
    xsrow[mt] = smem_u32(xsm) + (uint32_t)m * xpitch + 16u * (uint32_t)t;
  }
  const int sq = lane & 7, sh = sq >> 2, sc = (sq >> 1) & 1, shalf = sq & 1;  // ring chunk of the lane
  const bool s_lane = a.Ns != 1 && (lane < 8 || (HAS_O && lane < 16));
  const T *s_src = static_cast<const T *>(lane < 8 ? a.scale : a.offset);
  auto fetch_unit = [&](int p, int s, int slot, const uint8_t *wp, uint4 (&wb)[2]) {
    const bool two = cg0 + 2 * p + 1 < cg1;
    wb[0] = ld_stream_u4(wp);
    wb[1] = two ? ld_stream_u4(wp + 512) : make_uint4(0u, 0u, 0u, 0u);
    if (!XSMEM && t < 2) {
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)  // first and last byte of the row's 128: one or two lines
        asm volatile("prefetch.global.L1 [%0];" ::"l"(
            reinterpret_cast<const char *>(xrow[mt] - 8 * t + 64 * s) + 127 * t));
    }
    if (s_lane) {
      const int k0 = 64 * s + 32 * sh;
      const int col = 16 * (cg0 + 2 * p + sc) + 8 * shalf;
      if (k0 < a.K && (sc == 0 || two)) {
        const int row = kblk[2 * s + sh] & 0x7FFF;
        cp_async16(ring_w + (uint32_t)(slot * RING_BYTES + (lane >> 3) * 128 + sq * 16),
                   s_src + (size_t)row * a.N + col);
      }
    }
    cp_async_commit();
  };

  // acc: the MMA sums of the open group; dsum: its x1 row sums (elements 0, 1 =
  // rows 2t, 2t+1; 2, 3 duplicate them); tot: the folded sums of the pair
  float acc[2][MT][4], tot[2][MT][4], dsum[MT][4];
#pragma unroll
  for (int c = 0; c < 2; ++c)
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[c][mt][i] = tot[c][mt][i] = dsum[mt][i] = 0.f;

  const float sscal = a.Ns == 1 ? E::to_f(static_cast<const T *>(a.scale)[0]) : 0.f;
  const float oscal = (HAS_O && a.Ns == 1) ? E::to_f(static_cast<const T *>(a.offset)[0]) : 0.f;
  constexpr float C136 = BF ? 136.f : 1032.f;  // A = C136 + q

  // fold the pending group sums of half h of the unit in ring slot `slot`:
  // tot += S * acc + (O - 136 S) * d
  auto flush = [&](int slot, int h) {
    const T *sr = reinterpret_cast<const T *>(ring + (warp * TRING + slot) * RING_BYTES);
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      float sl = sscal, shi = sscal, ol = oscal, ohi = oscal;
      if (a.Ns != 1) {
        const int q0 = (h << 2) | (c << 1);  // chunks q0 (columns 0..7) and q0 + 1 (8..15)
        sl = E::to_f(sr[q0 * 8 + g]);
        shi = E::to_f(sr[(q0 + 1) * 8 + g]);
        if constexpr (HAS_O) {
          ol = E::to_f(sr[64 + q0 * 8 + g]);
          ohi = E::to_f(sr[64 + (q0 + 1) * 8 + g]);
        }
      }
      const float cl = fmaf(-C136, sl, ol), ch = fmaf(-C136, shi, ohi);
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        tot[c][mt][0] = fmaf(cl, dsum[mt][0], fmaf(sl, acc[c][mt][0], tot[c][mt][0]));
        tot[c][mt][1] = fmaf(cl, dsum[mt][1], fmaf(sl, acc[c][mt][1], tot[c][mt][1]));
        tot[c][mt][2] = fmaf(ch, dsum[mt][0], fmaf(shi, acc[c][mt][2], tot[c][mt][2]));
        tot[c][mt][3] = fmaf(ch, dsum[mt][1], fmaf(shi, acc[c][mt][3], tot[c][mt][3]));
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[c][mt][i] = 0.f;
      }
    }
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int i = 0; i < 4; ++i) dsum[mt][i] = 0.f;
  };

  // store the run's sums of pair p (slot sl of this warp) and clear them
  auto store_pair = [&](int p, int sl) {
    float *dst = part + (size_t)(warp * TSL + sl) * SLOT_FLOATS;
#pragma unroll
    for (int c = 0; c < 2; ++c)
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int m = 8 * mt + 2 * t + (i & 1), col = g + 8 * (i >> 1);
          dst[(c * MP + m) * 16 + col] = tot[c][mt][i];
          tot[c][mt][i] = 0.f;
        }
    if (lane == 0) s_tag[warp][sl] = p;
  };

  // ---- the run: (fp, fs, fslot, fwp) = the next unit to fetch, (p, s, slot) = the next to use
  uint4 wb[TD][2];
  int fp = r0 / a.KS, fs = r0 - fp * a.KS, fslot = 0;
  const uint8_t *fwp = a.w + (size_t)fs * slab + (size_t)(cg0 + 2 * fp) * 512 + lane * 16;
  auto advance_fetch = [&]() {
    fwp += slab;
    if (++fs == a.KS) {
      fs = 0;
      ++fp;
      fwp = a.w + (size_t)(cg0 + 2 * fp) * 512 + lane * 16;
    }
    if (++fslot == TRING) fslot = 0;
  };
#pragma unroll
  for (int i = 0; i < TD; ++i) {
    if (r0 + i < r1) {
      fetch_unit(fp, fs, fslot, fwp, wb[i]);
      advance_fetch();
    } else {
      cp_async_commit();
    }
  }
  if (XSMEM) {  // the staged x1 has landed (bounded wait; the copy always completes)
    const long long t0 = clock64();
    while (!mbar_try_wait(smem_u32(&s_xbar), 0u))
      if (clock64() - t0 > kWaitBudget) break;
  }
  int p = r0 / a.KS, s = r0 - p * a.KS, slot = 0;
  int cur_p = -1, slot_i = -1;
  // pending: the half whose group sums are not yet folded (per-channel: until the pair ends)
  int pend_slot = -1, pend_h = 0;
  constexpr uint32_t ONES = BF ? 0x3F803F80u : 0x3C003C00u;
  for (int u0 = r0; u0 < r1; u0 += TD) {
#pragma unroll
    for (int i = 0; i < TD; ++i) {
      const int u = u0 + i;
      if (u >= r1) break;
      const uint4 w0 = wb[i][0], w1 = wb[i][1];
      const bool two = cg0 + 2 * p + 1 < cg1;  // the pair's second column group exists
      if (p != cur_p) {
        if (pend_slot >= 0) {
          flush(pend_slot, pend_h);
          pend_slot = -1;
        }
        if (cur_p >= 0) store_pair(cur_p, slot_i);
        cur_p = p;
        ++slot_i;
      }
      // activations of this k-step: rows 8mt + g, k-rows 64s + 8t.. and 64s + 32 + 8t..
      // (past K: zeros -- the weight's padding nibbles are 136 + 0, not 0)
      const int krem = KFULL ? 64 : a.K - 64 * s - 8 * t;  // k-rows left from the lane's first
      uint4 xb[MT][2];
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          if (KFULL || 32 * h < krem) {
            if constexpr (XSMEM)
              asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                           : "=r"(xb[mt][h].x), "=r"(xb[mt][h].y), "=r"(xb[mt][h].z), "=r"(xb[mt][h].w)
                           : "r"(xsrow[mt] + (uint32_t)(128 * s + 64 * h)));
            else
              xb[mt][h] = __ldg(reinterpret_cast<const uint4 *>(xrow[mt] + 64 * s + 32 * h));
          } else {
            xb[mt][h] = make_uint4(0u, 0u, 0u, 0u);
          }
        }
      // this unit's scale chunks have landed (TD - 1 newer groups may still be in flight)
      cp_async_wait<TD - 1>();
      __syncwarp();
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        if (!KFULL && 64 * s + 32 * h >= a.K) break;
        const uint32_t info = kblk[2 * s + h];
#pragma unroll
        for (int jl = 0; jl < 2; ++jl) {
          const int j = 2 * h + jl;
          uint32_t aa[4], ab[4];
          word_to_a<DT>(j == 0 ? w0.x : j == 1 ? w0.y : j == 2 ? w0.z : w0.w, aa);
          if (two) word_to_a<DT>(j == 0 ? w1.x : j == 1 ? w1.y : j == 2 ? w1.z : w1.w, ab);
#pragma unroll
          for (int mt = 0; mt < MT; ++mt) {
            const uint32_t b0 = jl ? xb[mt][h].z : xb[mt][h].x;
            const uint32_t b1 = jl ? xb[mt][h].w : xb[mt][h].y;
            mma_16816<BF>(acc[0][mt], aa[0], aa[1], aa[2], aa[3], b0, b1);
            if (two) mma_16816<BF>(acc[1][mt], ab[0], ab[1], ab[2], ab[3], b0, b1);
            // x1 row sums of these k-rows (A = all ones), for both tiles
            mma_16816<BF>(dsum[mt], ONES, ONES, ONES, ONES, b0, b1);
          }
        }
        pend_slot = slot;
        pend_h = h;
        // fold at the end of a group or of K (per-channel / per-tensor: when the pair ends)
        if (info & 0x8000u) {
          flush(slot, h);
          pend_slot = -1;
        }
      }
      __syncwarp();  // every lane has read the slot before it is refilled
      if (u + TD < r1) {
        fetch_unit(fp, fs, fslot, fwp, wb[i]);
        advance_fetch();
      } else {
        cp_async_commit();
      }
      if (++s == a.KS) { s = 0; ++p; }
      if (++slot == TRING) slot = 0;
    }
  }
  if (pend_slot >= 0) flush(pend_slot, pend_h);
  if (cur_p >= 0) store_pair(cur_p, slot_i);
  } else {
  // ---- group-structured loop. A unit is one column group at two k-steps
  // (two 512-byte tiles, 128 k-rows); a group of scales is a whole number of
  // units (group % 128 == 0; per-channel and per-tensor scales are cut into
  // groups of one unit). Items (column group, group) in column-group-major
  // order are dealt to the warps in contiguous runs, at most three column
  // groups long (ncg <= 32), so no group's sums are split between warps and a
  // warp folds them at the group's last unit: tot += S (acc0 + acc1) +
  // (O - 136 S) d, with d the group's x1 row sums (computed once per CTA
  // below) and S, O from the CTA's scale block, staged in shared memory at the
  // start. Per unit: two 16-byte weight loads (TD units ahead), four 16-byte
  // activation loads from the staged x1, eight words into A registers and
  // eight MMAs (one chain per k-step).
  const int ncg = cg1 - cg0;
  const int KS2 = a.KS >> 1;
  const int ug = a.gu >> 1;  // units per group
  const int UG = ncg * a.GV;
  auto unit_of = [&](int item) {
    const int c = item / a.GV, q = item - c * a.GV;
    return c * KS2 + (q * ug < KS2 ? q * ug : KS2);
  };
  const int r0 = unit_of((int)((long long)UG * warp / TW));
  const int r1 = unit_of((int)((long long)UG * (warp + 1) / TW));
  // this lane's activation rows 8 mt + g at k-offset 8t (rows past M repeat
  // row M - 1; their outputs are never stored)
  const T *xrow[MT];
  uint32_t xsrow[MT];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt) {
    const int m = 8 * mt + g < a.M ? 8 * mt + g : a.M - 1;
    xrow[mt] = x1 + (size_t)m * a.K + 8 * t;
    xsrow[mt] = smem_u32(xsm) + (uint32_t)m * xpitch + 16u * (uint32_t)t;
  }
  // the lane's 16 bytes of k-step ks, k-rows 32h.. of the step
  auto load_x = [&](int ks, uint4 (&xb)[MT][2]) {
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        if constexpr (XSMEM)
          asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                       : "=r"(xb[mt][h].x), "=r"(xb[mt][h].y), "=r"(xb[mt][h].z), "=r"(xb[mt][h].w)
                       : "r"(xsrow[mt] + (uint32_t)(128 * ks + 64 * h)));
        else
          xb[mt][h] = __ldg(reinterpret_cast<const uint4 *>(xrow[mt] + 64 * ks + 32 * h));
      }
  };

  // the CTA's scale (offset) rows for its columns, [row][16 ncg] (rows: the
  // groups, or one per-channel row; none for a per-tensor scale)
  const int srows = a.Ns == 1 ? 0 : (a.group ? a.G_rows : 1);
  {
    const int cpr = 2 * ncg;  // 16-byte chunks per row
    const T *sg = static_cast<const T *>(a.scale), *og = static_cast<const T *>(a.offset);
    for (int i = threadIdx.x; i < srows * cpr; i += TTHREADS) {
      const int r = i / cpr, q = i - r * cpr;
      cp_async16(smem_u32(ssm + (size_t)r * ncols + 8 * q), sg + (size_t)r * a.N + 16 * cg0 + 8 * q);
      if constexpr (HAS_O)
        cp_async16(smem_u32(ssm + (size_t)(srows + r) * ncols + 8 * q),
                   og + (size_t)r * a.N + 16 * cg0 + 8 * q);
    }
    cp_async_commit();
  }

  // weights: the fetch walk over units (fcl, fj)
  int fcl = r0 / KS2, fj = r0 - fcl * KS2;
  const uint8_t *fwp = a.w + (size_t)(2 * fj) * slab + (size_t)(cg0 + fcl) * 512 + lane * 16;
  auto fetch = [&](uint4 (&wb)[2]) {
    wb[0] = ld_stream_u4(fwp);
    wb[1] = ld_stream_u4(fwp + slab);
    if (!XSMEM && t < 2) {
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)  // first and last byte of the row's 256: two to four lines
        asm volatile("prefetch.global.L1 [%0];" ::"l"(
            reinterpret_cast<const char *>(xrow[mt] - 8 * t + 128 * fj) + 255 * t));
    }
    fwp += 2 * slab;
    if (++fj == KS2) {
      fj = 0;
      ++fcl;
      fwp = a.w + (size_t)(cg0 + fcl) * 512 + lane * 16;
    }
  };
  uint4 wb[TD][2];
#pragma unroll
  for (int i = 0; i < TD; ++i)
    if (r0 + i < r1) fetch(wb[i]);

  if (XSMEM) {  // the staged x1 has landed (bounded wait; the copy always completes)
    const long long t0 = clock64();
    while (!mbar_try_wait(smem_u32(&s_xbar), 0u))
      if (clock64() - t0 > kWaitBudget) break;
  }
  constexpr uint32_t ONES = BF ? 0x3F803F80u : 0x3C003C00u;
  const uint32_t ONES4[4] = {ONES, ONES, ONES, ONES};
  // d[gq][m] = sum of x1[m, k] over group gq's k-rows, by MMAs with A = ones
  // (rows of D are equal; lanes 0..3 hold rows 2t and 2t + 1 of each block)
  for (int gq = warp; gq < a.GV; gq += TW) {
    float dd[MT][4];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int i = 0; i < 4; ++i) dd[mt][i] = 0.f;
    const int ks1 = (gq + 1) * a.gu < a.KS ? (gq + 1) * a.gu : a.KS;
    for (int ks = gq * a.gu; ks < ks1; ++ks) {
      uint4 xb[MT][2];
      load_x(ks, xb);
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          mma_16816_f<BF>(dd[mt], ONES4, xb[mt][h].x, xb[mt][h].y);
          mma_16816_f<BF>(dd[mt], ONES4, xb[mt][h].z, xb[mt][h].w);
        }
    }
    if (g == 0) {
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
        *reinterpret_cast<float2 *>(dsm + gq * MP + 8 * mt + 2 * t) = make_float2(dd[mt][0], dd[mt][1]);
    }
  }
  cp_async_wait<0>();
  __syncthreads();  // row sums and the scale block are in shared memory

  float acc[2][MT][4], tot[MT][4];
#pragma unroll
  for (int q = 0; q < 2; ++q)
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[q][mt][i] = tot[mt][i] = 0.f;
  const float sscal = a.Ns == 1 ? E::to_f(static_cast<const T *>(a.scale)[0]) : 0.f;
  const float oscal = (HAS_O && a.Ns == 1) ? E::to_f(static_cast<const T *>(a.offset)[0]) : 0.f;
  constexpr float C136 = BF ? 136.f : 1032.f;  // A = C136 + q

  // tot += S (acc0 + acc1) + (O - 136 S) d for group gq of column group cl
  auto fold = [&](int gq, int cl) {
    float2 dd[MT];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
      dd[mt] = *reinterpret_cast<const float2 *>(dsm + gq * MP + 8 * mt + 2 * t);
    float sl = sscal, shi = sscal, ol = oscal, ohi = oscal;
    if (srows) {
      const T *sr = ssm + (size_t)(a.group ? gq : 0) * ncols + 16 * cl + g;
      sl = E::to_f(sr[0]);
      shi = E::to_f(sr[8]);
      if constexpr (HAS_O) {
        ol = E::to_f(sr[(size_t)srows * ncols]);
        ohi = E::to_f(sr[(size_t)srows * ncols + 8]);
      }
    }
    const float cl0 = fmaf(-C136, sl, ol), ch0 = fmaf(-C136, shi, ohi);
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
      tot[mt][0] = fmaf(cl0, dd[mt].x, fmaf(sl, acc[0][mt][0] + acc[1][mt][0], tot[mt][0]));
      tot[mt][1] = fmaf(cl0, dd[mt].y, fmaf(sl, acc[0][mt][1] + acc[1][mt][1], tot[mt][1]));
      tot[mt][2] = fmaf(ch0, dd[mt].x, fmaf(shi, acc[0][mt][2] + acc[1][mt][2], tot[mt][2]));
      tot[mt][3] = fmaf(ch0, dd[mt].y, fmaf(shi, acc[0][mt][3] + acc[1][mt][3], tot[mt][3]));
      if constexpr (!UG1) {
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[0][mt][i] = acc[1][mt][i] = 0.f;
      }
    }
  };
  // the run's sums of column group cl into slot sl of this warp, then cleared
  auto store_cg = [&](int cl, int sl) {
    float *dst = part + (size_t)(warp * TSLG + sl) * (MP * 16);
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int m = 8 * mt + 2 * t + (i & 1), col = g + 8 * (i >> 1);
        dst[m * 16 + col] = tot[mt][i];
        tot[mt][i] = 0.f;
      }
    if (lane == 0) s_tag[warp][sl] = cl;
  };

  int cl = r0 / KS2, j = r0 - cl * KS2, slot_i = 0;
  int gq = j / ug;                           // the open group (runs start at a group's first unit)
  int ul = ug < KS2 - j ? ug : KS2 - j;      // its units left
  // one unit from wb[i]; its slot is refilled (TD units ahead) after use
  auto unit = [&](uint4 (&wbi)[2], bool refill) {
    uint4 xb[2][MT][2];
    load_x(2 * j, xb[0]);
    load_x(2 * j + 1, xb[1]);
#pragma unroll
    for (int q = 0; q < 2; ++q)
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) {
        const int h = jj >> 1, jl = jj & 1;
        uint32_t aa[4];
        word_to_a<DT>(jj == 0 ? wbi[q].x : jj == 1 ? wbi[q].y : jj == 2 ? wbi[q].z : wbi[q].w, aa);
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          const uint32_t b0 = jl ? xb[q][mt][h].z : xb[q][mt][h].x;
          const uint32_t b1 = jl ? xb[q][mt][h].w : xb[q][mt][h].y;
          if (UG1 && jj == 0)
            mma_16816_z<BF>(acc[q][mt], aa, b0, b1);
          else
            mma_16816_f<BF>(acc[q][mt], aa, b0, b1);
        }
      }
    if (refill) fetch(wbi);
    ++j;
    if (--ul == 0) {  // the group ends with this unit
      fold(gq, cl);
      ++gq;
      if (j == KS2) {  // and so does the column group
        store_cg(cl, slot_i);
        ++slot_i;
        ++cl;
        j = 0;
        gq = 0;
      }
      ul = ug < KS2 - j ? ug : KS2 - j;
    }
  };
  int u0 = r0;
  for (; u0 + 2 * TD <= r1; u0 += TD) {  // every refill in range
#pragma unroll
    for (int i = 0; i < TD; ++i) unit(wb[i], true);
  }
  for (; u0 < r1; u0 += TD) {
#pragma unroll
    for (int i = 0; i < TD; ++i)
      if (u0 + i < r1) unit(wb[i], u0 + i + TD < r1);
  }
  if (r0 < r1 && j != 0) store_cg(cl, slot_i);  // the run ended inside a column group
  }
  cp_async_wait<0>();
  __syncthreads();

  // ---- epilogue: partial sums in warp order + bias + residual -> y
  T *yout = static_cast<T *>(a.y);
  T *nout = static_cast<T *>(a.normOut);
  const int npair = ncols / 2;
  for (int e = threadIdx.x; e < a.M * npair; e += TTHREADS) {
    const int m = e / npair, col = 2 * (e - m * npair);
    const int cl = col >> 4, p = cl >> 1, c = cl & 1, cc = col & 15;
    float v0 = 0.f, v1 = 0.f;
    if constexpr (GRP) {  // slots of one column group, [MP][16]
      for (int w = 0; w < TW; ++w)
#pragma unroll
        for (int sl = 0; sl < TSLG; ++sl)
          if (s_tag[w][sl] == cl) {
            const float *src = part + (size_t)(w * TSLG + sl) * (MP * 16) + m * 16 + cc;
            v0 += src[0];
            v1 += src[1];
          }
    } else {  // slots of one pair, [2][MP][16]
      for (int w = 0; w < TW; ++w)
#pragma unroll
        for (int sl = 0; sl < TSL; ++sl)
          if (s_tag[w][sl] == p) {
            const float *src = part + (size_t)(w * TSL + sl) * SLOT_FLOATS + (c * MP + m) * 16 + cc;
            v0 += src[0];
            v1 += src[1];
          }
    }
    const int n = 16 * cg0 + col;
    const float2 bb = a.bias ? unpack2<DT>(*reinterpret_cast<const uint32_t *>(ebias + col))
                             : make_float2(0.f, 0.f);
    const float2 rr = unpack2<DT>(*reinterpret_cast<const uint32_t *>(eres + (size_t)m * ncols + col));
    v0 += bb.x + rr.x;
    v1 += bb.y + rr.y;
    *reinterpret_cast<uint32_t *>(yout + (size_t)m * a.N + n) = pack2<DT>(v0, v1);
    ysm[m * ncols + col] = v0;
    ysm[m * ncols + col + 1] = v1;
  }
  __syncthreads();
  // per-row sum of y^2 over this CTA's columns, in a fixed order
  for (int m = warp; m < a.M; m += TW) {
    float sq = 0.f;
    for (int col = lane; col < ncols; col += 32) sq = fmaf(ysm[m * ncols + col], ysm[m * ncols + col], sq);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, o);
    if (lane == 0) __stcg(a.ss + m * a.G + cta, sq);
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
        record_timeout(a.status, kTWhereGrid);
        break;
      }
      __nanosleep(32);
    }
  }
  __syncthreads();
  // 1/RMS of row m: warp m sums the CTAs' partials (lane-strided, then a fixed
  // shuffle tree: the same order in every CTA and every run)
  // the last CTA through clears the grid counters for the next call; with
  // fewer than TW rows the last warp has no row sum to form, so its atomic's
  // round trip overlaps the sums below (else thread 0 departs after them)
  auto depart = [&]() {
    if (atomicAdd(a.gbar + 1, 1u) == (uint32_t)a.G - 1u) {
      atomicExch(a.gbar, 0u);
      atomicExch(a.gbar + 1, 0u);
    }
  };
  const bool early = a.M < TW;
  if (early && threadIdx.x == TTHREADS - 32) depart();
  if (warp < a.M && !s_abort) {
    // all of the lane's loads first (the grid has at most 32 * kTParts CTAs),
    // then the sum in CTA order
    float pv[kTParts];
#pragma unroll
    for (int i = 0; i < kTParts; ++i) {
      const int c = lane + 32 * i;
      pv[i] = c < a.G ? __ldcg(a.ss + warp * a.G + c) : 0.f;
    }
    float tot2 = 0.f;
#pragma unroll
    for (int i = 0; i < kTParts; ++i) tot2 += pv[i];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) tot2 += __shfl_xor_sync(0xffffffffu, tot2, o);
    if (lane == 0) s_rstd[warp] = rsqrtf(tot2 / (float)a.N + a.eps);
  }
  __syncthreads();
  if (!early && threadIdx.x == 0) depart();
  if (s_abort) return;  // a CTA whose wait gave up writes no normOut
  for (int e = threadIdx.x; e < a.M * npair; e += TTHREADS) {
    const int m = e / npair, col = 2 * (e - m * npair);
    const int n = 16 * cg0 + col;
    const float2 gg = unpack2<DT>(*reinterpret_cast<const uint32_t *>(egam + col));
    const float rs = s_rstd[m];
    *reinterpret_cast<uint32_t *>(nout + (size_t)m * a.N + n) =
        pack2<DT>(ysm[m * ncols + col] * rs * gg.x, ysm[m * ncols + col + 1] * rs * gg.y);
  }
}

// ------------------------------------------------------------------ host side

int tiled_grid_size(const Problem &p) {
  int sms = device_info().sms > 0 ? device_info().sms : 148;
  if (sms > 32 * kTParts) sms = 32 * kTParts;  // the row sums' readers cover that many CTAs
  const int ncg = (int)(p.N / 16);
  return ncg < sms ? ncg : sms;
}

constexpr int kTD = 4;  // units in flight per warp

// The group-structured loop applies: whole 64-row k-steps, and scale groups of
// whole k-steps (or one scale row, cut into groups of two k-steps).
bool tiled_grp(const Problem &p) { return p.K % 128 == 0 && (p.group == 0 || p.group % 128 == 0); }
int tiled_gu(const Problem &p) { return tiled_grp(p) ? (p.group ? (int)(p.group / 64) : 2) : 0; }
int tiled_gv(const Problem &p) {
  if (!tiled_grp(p)) return 0;
  const int ks = (int)(p.K / 64), gu = tiled_gu(p);
  return (ks + gu - 1) / gu;
}

// Shared memory of one CTA; with `xsmem` the staged x1 rows too, with `grp`
// the group-structured loop's row sums and scale block.
uint64_t tiled_smem(const Problem &p, int G, bool xsmem, bool grp) {
  const int MT = p.M <= 8 ? 1 : 2;
  const int64_t ncg_max = (p.N / 16 + G - 1) / G;
  uint64_t b = (uint64_t)TW * TSL * 2 * (8 * MT) * 16 * 4 + (uint64_t)TW * (kTD + 1) * 256 +
               (uint64_t)(8 * MT) * ncg_max * 16 * 4 + (uint64_t)(p.M + 2) * ncg_max * 16 * 2 +
               (uint64_t)(p.K + 31) / 32 * 2;
  if (grp) {
    const uint64_t srows = p.Ns == 1 ? 0 : (uint64_t)p.G;  // G = 1 unless per-group
    b += 16 + (uint64_t)tiled_gv(p) * (8 * MT) * 4;
    b += 16 + srows * (uint64_t)ncg_max * 16 * 2 * (p.offset ? 2 : 1);
  }
  if (xsmem) b += 16 + (uint64_t)p.M * (2 * (uint64_t)p.K + 64);
  return b;
}

}  // namespace

bool decode_tiled_applicable(const Problem &p) {
  if (p.M < 1 || p.M > 16 || p.N < 16 || p.wbits != 4 || !p.tiled) return false;
  if (p.N % 16 != 0 || p.K % 8 != 0) return false;
  const void *v16[] = {p.x1, p.x2, p.scale, p.offset, p.bias, p.residual, p.gamma};
  for (const void *q : v16)
    if (q && reinterpret_cast<uintptr_t>(q) % 16 != 0) return false;
  const void *v4[] = {p.y, p.normOut};
  for (const void *q : v4)
    if (q && reinterpret_cast<uintptr_t>(q) % 4 != 0) return false;
  // a CTA's columns: at most 16 pairs of column groups (runs then touch <= 2 pairs)
  const int G = tiled_grid_size(p);
  const int64_t ncg_max = (p.N / 16 + G - 1) / G;
  if (ncg_max > 32) return false;
  return tiled_smem(p, G, false, false) + 2048 <= (uint64_t)device_info().smem_optin;
}

bool plan_decode_tiled(const Problem &p, Plan &plan) {
  if (plan_decode_km(p, plan)) return true;
  if (!decode_tiled_applicable(p)) return false;
  plan.kernel = WQ_KERNEL_DECODE;
  plan.grid = tiled_grid_size(p);
  plan.ws_bytes = kWsHeader + (uint64_t)plan.grid * 16 * 4;
  return true;
}

template <int DT, int MT, bool HAS_O, bool KFULL, bool XSMEM, bool GRP, bool UG1 = false>
static cudaError_t launch_decode_tiled_k(const Problem &p, const Plan &plan, void *ws,
                                         cudaStream_t s) {
  const int G = plan.grid;
  const uint32_t smem = (uint32_t)tiled_smem(p, G, XSMEM, GRP);
  // the cap leaves room for the kernel's few static shared variables
  static cudaError_t attr_err = cudaFuncSetAttribute(
      decode_tiled_kernel<DT, MT, HAS_O, kTD, KFULL, XSMEM, GRP, UG1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
      (int)device_info().smem_optin - 2048);
  if (attr_err != cudaSuccess) return attr_err;
  char *wsb = static_cast<char *>(ws);
  DTArgs args = {};
  args.x1 = p.x1; args.w = static_cast<const uint8_t *>(p.x2);
  args.scale = p.scale; args.offset = p.offset; args.bias = p.bias;
  args.residual = p.residual; args.gamma = p.gamma; args.y = p.y; args.normOut = p.normOut;
  args.status = reinterpret_cast<uint32_t *>(ws);
  args.gbar = reinterpret_cast<uint32_t *>(wsb + kTGbarOff);
  args.ss = reinterpret_cast<float *>(wsb + kWsHeader);
  args.M = (int)p.M; args.K = (int)p.K; args.N = (int)p.N;
  args.KS = (int)((p.K + 63) / 64); args.NCG = (int)(p.N / 16);
  args.group = (int)p.group; args.Ns = (int)p.Ns; args.G = G;
  args.gu = tiled_gu(p); args.GV = tiled_gv(p);
  args.G_rows = (int)p.G;
  args.eps = p.eps;
  args.budget = wait_budget();
  args.extra = wait_extra_arrivals();
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)G, 1, 1);
  cfg.blockDim = dim3(TTHREADS, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, decode_tiled_kernel<DT, MT, HAS_O, kTD, KFULL, XSMEM, GRP, UG1>, args);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <int DT, int MT, bool HAS_O>
static cudaError_t launch_decode_tiled_t(const Problem &p, const Plan &plan, void *ws,
                                         cudaStream_t s) {
  // x1 staged in shared memory when it fits beside the rest (2 KB of static
  // shared variables are kept free)
  const uint64_t cap = (uint64_t)device_info().smem_optin - 2048;
  // the group-structured loop (x1 staged; at least 8 units per warp: with
  // fewer, its per-CTA preparation outweighs the leaner loop)
  const int64_t ncg_max = (p.N / 16 + plan.grid - 1) / plan.grid;
  if (tiled_grp(p) && ncg_max * (p.K / 128) >= 8 * TW && tiled_smem(p, plan.grid, true, true) <= cap)
    return tiled_gu(p) == 2 ? launch_decode_tiled_k<DT, MT, HAS_O, true, true, true, true>(p, plan, ws, s)
                            : launch_decode_tiled_k<DT, MT, HAS_O, true, true, true, false>(p, plan, ws, s);
  const bool xs = tiled_smem(p, plan.grid, true, false) <= cap;
  if (p.K % 64 == 0)
    return xs ? launch_decode_tiled_k<DT, MT, HAS_O, true, true, false>(p, plan, ws, s)
              : launch_decode_tiled_k<DT, MT, HAS_O, true, false, false>(p, plan, ws, s);
  return xs ? launch_decode_tiled_k<DT, MT, HAS_O, false, true, false>(p, plan, ws, s)
            : launch_decode_tiled_k<DT, MT, HAS_O, false, false, false>(p, plan, ws, s);
}

cudaError_t launch_decode_tiled(const Problem &p, const Plan &plan, void *ws, cudaStream_t s) {
  if (plan.mode == kPlanModeKm) return launch_decode_km(p, plan, ws, s);
  const bool o = p.offset != nullptr;
  const int MT = p.M <= 8 ? 1 : 2;
  if (p.dtype == WQ_BF16) {
    if (MT == 1) return o ? launch_decode_tiled_t<WQ_BF16, 1, true>(p, plan, ws, s)
                          : launch_decode_tiled_t<WQ_BF16, 1, false>(p, plan, ws, s);
    return o ? launch_decode_tiled_t<WQ_BF16, 2, true>(p, plan, ws, s)
             : launch_decode_tiled_t<WQ_BF16, 2, false>(p, plan, ws, s);
  }
  if (MT == 1) return o ? launch_decode_tiled_t<WQ_F16, 1, true>(p, plan, ws, s)
                        : launch_decode_tiled_t<WQ_F16, 1, false>(p, plan, ws, s);
  return o ? launch_decode_tiled_t<WQ_F16, 2, true>(p, plan, ws, s)
           : launch_decode_tiled_t<WQ_F16, 2, false>(p, plan, ws, s);
}

}  // namespace wq
