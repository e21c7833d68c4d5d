// Internal declarations shared by the .cu files of libwq (not part of the ABI).
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "../../include/wq.h"

namespace wq {

// Scale layout after validation.
enum ScaleMode : int { kPerTensor = 0, kPerChannel = 1, kPerGroup = 2 };

// A validated problem: everything a launcher needs, in plain integers/pointers.
struct Problem {
  int64_t M = 0, K = 0, N = 0;
  int dtype = WQ_BF16;     // WQ_F16 or WQ_BF16 (x1, scale, offset, bias, residual, gamma, y, normOut)
  int wbits = 4;           // 4 (packed, two per byte along N) or 8
  bool tiled = false;      // INT4 in the kernel-native tiled layout (wq_tiled.cu)
  bool transposed = false; // x2 stored as its (N, K) transpose, K contiguous
  int smode = kPerTensor;  // ScaleMode
  int64_t group = 0;       // > 0 only for kPerGroup
  int64_t G = 1;           // scale rows: ceil(K/group) for kPerGroup, else 1
  int64_t Ns = 1;          // scale columns: 1 (per-tensor) or N
  float eps = 0.f;
  const void *x1 = nullptr, *x2 = nullptr, *scale = nullptr, *offset = nullptr,
             *bias = nullptr, *residual = nullptr, *gamma = nullptr;
  void *y = nullptr, *normOut = nullptr;
};

// Workspace header: the first kWsHeader bytes of every matmul workspace. The
// caller zeroes it once; every kernel leaves it zero after a call that ends
// without a device-side error (the prefill path clears it per call, the decode
// kernel resets its counters as it finishes, the generic path leaves it alone).
//   bytes    0..3     device status (0 = ok, else WQ_ERR_DEVICE_TIMEOUT | where << 8)
//   bytes  128..135   decode: grid barrier counters (arrive, depart)
//   bytes 1024..2047  decode: per-tile segment counters (at most 256 tiles)
constexpr uint64_t kWsHeader = 2048;

// Device properties cached per device (SM count, cluster support ...).
struct DeviceInfo {
  int device = -1;
  int sms = 148;
  int cc_major = 10, cc_minor = 3;
  size_t smem_optin = 227 * 1024;
};
const DeviceInfo &device_info();

// Launch plan of one call; computed on the host from the Problem alone, so the
// first and second phases agree on the workspace size.
struct Plan {
  int kernel = WQ_KERNEL_GENERIC;
  uint64_t ws_bytes = 0;
  // split-K partial sums: parts x M x N fp32, at ws + part_off
  int parts = 1;
  uint64_t part_off = kWsHeader;
  // generic kernel: k rows per split
  int64_t ksplit = 0;
  // epilogue: CTAs per row (a thread-block cluster), vectorised or not
  int epi_cluster = 1;
  bool epi_vec = false;
  // prefill: operand mode, counters, row partials and preparation buffers
  int mode = 0;
  uint64_t cnt_off = 0, rowpart_off = 0, rowsum_off = 0, erow_off = 0, ecol_off = 0, s16_off = 0,
           x16_off = 0, dext_off = 0, oext_off = 0;
  int ldx = 0;       // prefill F16EMU with offset: columns of the offset-term operands (2G up to 64)
  int64_t n_tiles = 0, m_tiles = 0;
  int grid = 0;
  int m_halves = 1;  // prefill: 128-row MMA halves per output tile (1 or 2)
};

// Launchers (return cudaError_t of the launch).
cudaError_t launch_pack_int4(const int32_t *in, uint8_t *out, int64_t K, int64_t N, cudaStream_t s);
// Kernel-native tiled INT4 layout: its byte count, the pack into it and the
// conversions between it and the dense layout (wq_tiled.cu).
uint64_t tiled_int4_bytes(int64_t K, int64_t N);
cudaError_t launch_pack_int4_tiled(const int32_t *in, uint8_t *out, int64_t K, int64_t N,
                                   cudaStream_t s);
cudaError_t launch_int4_nd_to_tiled(const uint8_t *in, uint8_t *out, int64_t K, int64_t N,
                                    cudaStream_t s);
cudaError_t launch_int4_tiled_to_nd(const uint8_t *in, uint8_t *out, int64_t K, int64_t N,
                                    cudaStream_t s);
// Any layout of a (K, N) INT4 weight (WQ_INT4, WQ_INT4_T, WQ_INT4_TILED) into another.
cudaError_t launch_int4_remap(const uint8_t *in, int in_layout, uint8_t *out, int out_layout,
                              int64_t K, int64_t N, cudaStream_t s);
cudaError_t launch_decode_tiled(const Problem &p, const Plan &plan, void *ws, cudaStream_t s);
// k-major decode for tiled INT4 weights with 9..64 rows (wq_decode_km.cu); its
// plans carry mode kPlanModeKm, and launch_decode_tiled hands them on.
constexpr int kPlanModeKm = 3;
bool decode_km_applicable(const Problem &p);
bool plan_decode_km(const Problem &p, Plan &plan);
cudaError_t launch_decode_km(const Problem &p, const Plan &plan, void *ws, cudaStream_t s);
// FP4 E2M1 pack and the mx block-scaled matmul (wq_fp4.cu).
cudaError_t launch_pack_fp4(const float *in, uint8_t *out, int64_t K, int64_t N, cudaStream_t s);
// x1t: x1 stored (K, M) packed along M and scale1 (ceil(K/32), M). The first
// form is exact (fp64 slice sums); the _tc form runs the slices on the tensor
// cores and adds them in fp32.
cudaError_t launch_mx_matmul_add_tc(const uint8_t *x1, const uint8_t *s1, bool x1t,
                                    const uint8_t *x2, const uint8_t *s2, float *y, int64_t M,
                                    int64_t K, int64_t N, cudaStream_t s);
cudaError_t launch_mx_matmul_add(const uint8_t *x1, const uint8_t *s1, bool x1t, const uint8_t *x2,
                                 const uint8_t *s2, float *y, int64_t M, int64_t K, int64_t N,
                                 cudaStream_t s);
// Large-M kernel for transposed INT4 weights with bf16 per-group scales and no
// offset (wq_prefill_t.cu), and its scale pre-pass (wq_prep.cu).
bool prefill_t_applicable(const Problem &p);
bool plan_prefill_t(const Problem &p, Plan &plan);
cudaError_t launch_prefill_t(const Problem &p, const Plan &plan, void *ws, cudaStream_t s);
cudaError_t launch_so_prep_t(const Problem &p, int16_t *e_col, uint32_t *S16T, cudaStream_t s);
// Per-token symmetric dynamic quantization (wq_dynquant.cu); bits 8 or 4.
cudaError_t launch_dynamic_quant(const void *x, const void *smooth, int dtype, int64_t M, int64_t K,
                                 int bits, void *y, float *scale, cudaStream_t s);
cudaError_t launch_generic(const Problem &p, const Plan &plan, void *ws, cudaStream_t s);
cudaError_t launch_prefill(const Problem &p, const Plan &plan, void *ws, cudaStream_t s);
cudaError_t launch_decode(const Problem &p, const Plan &plan, void *ws, cudaStream_t s);
cudaError_t launch_timeout_check(uint32_t *status, long long budget, cudaStream_t s);
// row_prep: row sums (RAWQ with offset) or the fp16 copy of x1 with its row
// exponents, plus (F16EMU with offset, dext != nullptr) the per-group row sums
// of that copy split into bf16 hi/lo, (M, ldx) row-major.
cudaError_t launch_row_prep(const Problem &p, float *rowsum, int16_t *e_row, __half *x16,
                            __nv_bfloat16 *dext, int ldx, cudaStream_t s);
// S16 rows are ld words long (ld >= N; INT4 rows are padded to whole
// 256-column tiles and stored in the dequant's interleaved column order);
// Oext (offset only) is the (N, ldx) bf16 operand of the offset term.
cudaError_t launch_so_prep(const Problem &p, int64_t ld, int16_t *e_col, uint32_t *S16,
                           __nv_bfloat16 *Oext, int ldx, cudaStream_t s);
cudaError_t launch_epilogue(const Problem &p, const Plan &plan, const void *ws, bool pdl,
                            cudaStream_t s);

// Budget (clock cycles) and extra target of the kernels' waits for other
// thread blocks: kWaitBudget and 0 unless wq_test_set_wait_limits changed them.
long long wait_budget();
uint32_t wait_extra_arrivals();

// Sets the thread-local message that wq_last_error() returns.
void set_last_error(int32_t code, const char *msg);

// Plan builders.
bool plan_generic(const Problem &p, Plan &plan);
bool prefill_applicable(const Problem &p);
bool plan_prefill(const Problem &p, Plan &plan);
bool decode_applicable(const Problem &p);
bool decode_tiled_applicable(const Problem &p);
bool plan_decode_tiled(const Problem &p, Plan &plan);
bool plan_decode(const Problem &p, Plan &plan);
void plan_epilogue(const Problem &p, Plan &plan);

}  // namespace wq
