/*
 * wq.h -- C ABI of the B300 (sm_103a) weight-only quantized matmul with a fused
 * residual-add + RMSNorm epilogue, and of the INT32 -> dense INT4 weight pack.
 *
 * Operations (Ascend CANN operator pages they restate):
 *   pack      aclnnConvertWeightToINT4Pack, "Function description": INT32 values
 *             that hold 4-bit integers are re-laid out from sparse storage (one
 *             per int32) to dense storage (two per byte), along the last
 *             dimension (aclnnDynamicQuant, "Constraints": INT4 needs the last
 *             dimension even, an INT32 view needs it divisible by 8).
 *   matmul    aclnnWeightQuantMatmulAllReduceAddRmsNorm, "Function description",
 *             formula:  mm_out  = x1 @ (x2 * antiquantScale + antiquantOffset) + bias
 *                       y       = mm_out + residual
 *                       normOut = y / sqrt(mean_n(y^2) + epsilon) * gamma
 *             The page's allReduce runs over one rank here, i.e. it is the
 *             identity. Shapes, dtypes and ranges follow that page's
 *             "Constraints" section.
 *
 * Call shape: both operations are two-phase like the pages' aclnn APIs
 * ("each operator has two calls"): *_get_workspace validates every argument and
 * returns the workspace size; the second call re-validates (cheaply), then
 * enqueues the work on `stream` and returns without waiting for it.
 *
 * Conventions for every function below:
 *   - Tensors are dense, row-major, on the current CUDA device. `data` is a
 *     device pointer; it may be NULL only when the tensor has zero elements.
 *     Strided or transposed tensors are not accepted.
 *   - The caller owns every buffer, the workspace and the stream. The library
 *     allocates no device memory and keeps no state between calls (apart from a
 *     thread-local error string for wq_last_error()).
 *   - `stream` is a cudaStream_t passed as void*; NULL is the legacy default
 *     stream. Work is asynchronous on it; errors found by the GPU while it runs
 *     are reported through the workspace status word (wq_read_device_status).
 *   - A function returns WQ_OK or a wq_status code and, on error, enqueues
 *     nothing. wq_last_error() then holds a one-line explanation.
 *   - Calls on the same stream are ordered; calls that share a workspace must
 *     not run concurrently on different streams.
 */
#ifndef WQ_H_
#define WQ_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Element types. WQ_INT4 is a logical type: a tensor of logical shape
 * (..., N) stores its elements two per byte along the last dimension, N/2 bytes
 * per row; the element in even column 2j sits in bits 3:0 of byte j and the
 * element in column 2j+1 in bits 7:4 (the pages do not fix this order; this is
 * the library's reading). Read as little-endian int32 words, element 8i+t of a
 * row sits in bits 4t+3:4t of word i.
 *
 * WQ_INT4_TILED is the same 4-bit values of a 2-D (K, N) weight, N % 16 == 0,
 * in the library's kernel-native tiled layout (the analogue of the pack page's
 * matrix-unit output format, aclnnConvertWeightToINT4Pack "Function
 * description"; the pages fix no layout for this GPU). The weight is cut into
 * tiles of 64 k-rows x 16 columns; tile (s, c) -- k-rows 64s.., columns 16c.. --
 * takes the 512 bytes at (s * N/16 + c) * 512, and K is padded with zero
 * nibbles to a multiple of 64 (ceil(K/64) * 64 * N / 2 bytes in all). Inside a
 * tile, element (kk, cc) = (k - 64s, n - 16c) takes nibble p of 32-bit word j of
 * 16-byte lane l: l = 4 (cc % 8) + (kk % 32) / 8, j = 2 (kk / 32) + (kk % 8) / 4,
 * p = (e < 2 ? 0 : 2) + cc / 8 + 4 (e % 2) with e = kk % 4, i.e. byte
 * l*16 + j*4 + p/2, bits 4(p%2)+3 : 4(p%2). Lane l's 16 bytes are then exactly
 * its A-operand registers (A = W^T) of four m16n8k16 MMAs. Tiled tensors must be
 * 16-byte aligned.
 *
 * WQ_INT8_T and WQ_INT4_T hold a weight transposed (aclnnWeightQuantMatmul-
 * AllReduceAddRmsNorm, "Constraints": x2 may be transposed): a (K, N) weight
 * stored as its (N, K) transpose, row-major with K contiguous; the descriptor
 * gives the stored shape (N, K). INT4_T packs two values per byte along K (k
 * even in bits 3:0), i.e. it is the WQ_INT4 packing of the (N, K) array.
 *
 * WQ_FP4_E2M1 is a logical 4-bit float (sign bit 3, 2-bit exponent, 1-bit
 * mantissa: magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6), stored two per byte along the
 * last dimension like WQ_INT4. WQ_E8M0 is one byte e per element, the power of
 * two 2^(e - 127), with e = 255 standing for NaN (the OCP MX encoding).
 * WQ_FP4_E2M1_T is the same element type for an operand given transposed: like
 * WQ_INT4_T the descriptor gives the stored shape, (K, M) for an x1 whose
 * logical shape is (M, K), packed two per byte along M. */
typedef enum wq_dtype {
    WQ_F16 = 1,
    WQ_BF16 = 2,
    WQ_INT8 = 3,
    WQ_INT4 = 4,
    WQ_INT32 = 5,
    WQ_INT4_TILED = 6,
    WQ_F32 = 7,
    WQ_INT8_T = 8,
    WQ_INT4_T = 9,
    WQ_FP4_E2M1 = 10,
    WQ_E8M0 = 11,
    WQ_FP4_E2M1_T = 12
} wq_dtype;

/* Tensor descriptor (the analogue of aclTensor): pointer, element type, rank
 * (1..3) and logical shape. Unused trailing shape entries are ignored. */
typedef struct wq_tensor {
    void *data;
    int32_t dtype;      /* a wq_dtype value */
    int32_t ndim;       /* 1, 2 or 3 */
    int64_t shape[3];
} wq_tensor;

typedef enum wq_status {
    WQ_OK = 0,
    WQ_ERR_NULL = 1,           /* a required pointer is NULL */
    WQ_ERR_DTYPE = 2,          /* an element type is not allowed */
    WQ_ERR_SHAPE = 3,          /* ranks, dimensions or ranges disagree */
    WQ_ERR_GROUP = 4,          /* group size not allowed for the scale shape */
    WQ_ERR_WORKSPACE = 5,      /* workspace NULL or smaller than required */
    WQ_ERR_UNSUPPORTED = 6,    /* a forced kernel cannot run this problem */
    WQ_ERR_CUDA = 7,           /* a CUDA runtime call or kernel launch failed */
    WQ_ERR_DEVICE_TIMEOUT = 8, /* a bounded device-side wait gave up (see below) */
    WQ_ERR_ALIAS = 9           /* an output overlaps an input it must not overlap */
} wq_status;

/* Kernel selection for the *_ex entry points. WQ_KERNEL_AUTO is what the plain
 * entry points use: DECODE for M <= 16, PREFILL for larger M, each when the
 * shapes meet its alignment rules, GENERIC otherwise. */
typedef enum wq_kernel {
    WQ_KERNEL_AUTO = 0,
    WQ_KERNEL_GENERIC = 1,     /* predicated CUDA-core kernel, any shape */
    WQ_KERNEL_DECODE = 2,      /* weight-streaming TMA + mma.sync kernel, M <= 16, INT4 */
    WQ_KERNEL_PREFILL = 3      /* TMA + tcgen05/TMEM kernel, large M */
} wq_kernel;

/* ------------------------------------------------------------------ pack */

/* First phase of the pack (aclnnConvertWeightToINT4Pack).
 *   weight       WQ_INT32, 2-D (K, N), N even, K >= 0, N >= 0. Values should lie
 *                in [-8, 7]; any other value keeps its low four bits (two's
 *                complement truncation). Or WQ_F32 (K, N) with a WQ_FP4_E2M1
 *                output (the page's FLOAT -> FLOAT4_E2M1 pack): each float becomes
 *                the nearest E2M1 value, ties to the even code, saturating at +-6
 *                (the page fixes neither; a NaN input is outside the domain).
 *   weight_int4  WQ_INT4, 2-D, logical shape (K, N), i.e. K*N/2 bytes; or
 *                WQ_INT4_TILED (N % 16 == 0, 16-byte aligned), the tiled layout;
 *                or WQ_INT4_T: the same bytes as WQ_INT4, for a `weight` that is
 *                already the transposed (N, K) array.
 *   ws_bytes     out: workspace bytes the second phase needs (always 0).
 * Errors: WQ_ERR_NULL, WQ_ERR_DTYPE, WQ_ERR_SHAPE. Touches no device memory. */
int32_t wq_pack_int4_get_workspace(const wq_tensor *weight, const wq_tensor *weight_int4,
                                   uint64_t *ws_bytes);

/* Second phase: enqueue the pack on `stream`. The output must not overlap the
 * input (WQ_ERR_ALIAS). K*N == 0 enqueues nothing. The result is bit-exact and
 * deterministic. `ws` may be NULL when ws_bytes is 0. */
int32_t wq_pack_int4(const wq_tensor *weight, const wq_tensor *weight_int4,
                     void *ws, uint64_t ws_bytes, void *stream);

/* Converts a (K, N) INT4 weight between any two of its layouts: dense
 * (WQ_INT4, shape (K, N)), tiled (WQ_INT4_TILED, shape (K, N), N % 16 == 0,
 * 16-byte aligned) and transposed (WQ_INT4_T, shape (N, K), K even), in the
 * direction the two dtypes give. The padding nibbles of a tiled output are zero.
 * Bit-exact, asynchronous on `stream`, no workspace. Errors: WQ_ERR_NULL,
 * WQ_ERR_DTYPE, WQ_ERR_SHAPE, WQ_ERR_UNSUPPORTED (alignment), WQ_ERR_ALIAS,
 * WQ_ERR_CUDA.
 * (aclnnConvertWeightToINT4Pack, "Function description": the ND to tiled
 * conversion of the pack's output format; the tiled to ND direction serves
 * checking and re-use of the weight elsewhere.) */
int32_t wq_convert_int4_layout(const wq_tensor *src, const wq_tensor *dst, void *stream);

/* ------------------------------------------------------------------ matmul */

/* First phase of the fused operator (aclnnWeightQuantMatmulAllReduceAddRmsNorm).
 *   x1        WQ_F16 or WQ_BF16, (M, K) or (b, s, K) with M = b*s; 0 <= M < 2^31,
 *             1 <= K <= 65535. Not transposed.
 *   x2        WQ_INT8 (K, N) or WQ_INT4 (K, N) packed as described above (N even),
 *             WQ_INT4_TILED (K, N) (N % 16 == 0, 16-byte aligned), or transposed:
 *             WQ_INT8_T / WQ_INT4_T given as (N, K) (K even for INT4_T);
 *             0 <= N <= 65535. A tiled weight runs on the tiled decode kernels
 *             for M <= 16, and for M <= 64 when K % 128 == 0 and the scales are
 *             per-tensor, per-channel or in groups of a multiple of 128 rows,
 *             else on the generic kernel. A transposed INT4 weight with bf16
 *             per-group scales and no offset runs on the transposed-weight
 *             prefill kernel for M > 16 (K % 64 == 0, N % 32 == 0); any other
 *             transposed weight runs on the generic kernel
 *             (wq_convert_int4_layout turns an INT4_T weight into the dense or
 *             tiled layout once, for the other fast kernels).
 *   scale     antiquantScale, x1's dtype: (1) per-tensor, (N) or (1, N)
 *             per-channel, (ceil(K/group), N) per-group.
 *   offset    antiquantOffset or NULL; if given, the scale's shape and dtype.
 *             The dequantized weight is W[k][n] = x2[k][n] * S + O, where S and O
 *             are taken at row floor(k/group) (per-group) or 0, column n or 0.
 *   bias      NULL or (N), x1's dtype.
 *   residual  (M, N) or (b, s, N) with b*s = M, x1's dtype.
 *   gamma     (N), x1's dtype.
 *   eps       epsilon inside the square root, >= 0.
 *   group     0 for per-tensor / per-channel scales; otherwise the group size:
 *             a multiple of 32 with 32 <= group <= K - 1, and then the scale
 *             must be (ceil(K/group), N).
 *   y         out, residual's shape and dtype. It MAY be the residual buffer
 *             itself (the page's in-place variant writes y into residual); any
 *             other overlap with an input is rejected.
 *   normOut   out, residual's shape and dtype; must not overlap any input or y.
 *   ws_bytes  out: bytes of device workspace the second phase needs.
 * Errors: WQ_ERR_NULL, WQ_ERR_DTYPE, WQ_ERR_SHAPE (K = 0 included), WQ_ERR_GROUP,
 * WQ_ERR_ALIAS. M = 0 or N = 0 is valid and the second phase enqueues nothing.
 * Touches no device memory. */
int32_t wq_matmul_add_rmsnorm_get_workspace(
    const wq_tensor *x1, const wq_tensor *x2, const wq_tensor *scale,
    const wq_tensor *offset, const wq_tensor *bias, const wq_tensor *residual,
    const wq_tensor *gamma, double eps, int64_t group,
    const wq_tensor *y, const wq_tensor *normOut, uint64_t *ws_bytes);

/* Second phase: enqueue the fused operator on `stream`.
 *   ws / ws_bytes  device workspace of at least the size the first phase
 *                  returned for the same arguments (WQ_ERR_WORKSPACE otherwise),
 *                  256-byte aligned. Its first 2048 bytes (the header: the device
 *                  status word and the counters of the decode kernel) must
 *                  be zero before the workspace is used for the first time, e.g.
 *                  one cudaMemsetAsync after allocating it; every call that ends
 *                  without a device-side error leaves the header zero again, so
 *                  no per-call clearing is needed. After a device-side error
 *                  (see wq_read_device_status) zero the header again. The rest
 *                  of the workspace may hold anything on entry.
 * Accumulation is fp32; the RMS is taken over the unrounded y, and y and normOut
 * are rounded once to x1's dtype (the large-M kernel scales the y it stored, so
 * its normOut carries one more rounding of y: at most 2^-9 relative in bf16,
 * 2^-11 in fp16). Results are bitwise identical from run to run for the same
 * arguments (no floating-point atomics; fixed reduction order). */
int32_t wq_matmul_add_rmsnorm(
    const wq_tensor *x1, const wq_tensor *x2, const wq_tensor *scale,
    const wq_tensor *offset, const wq_tensor *bias, const wq_tensor *residual,
    const wq_tensor *gamma, double eps, int64_t group,
    const wq_tensor *y, const wq_tensor *normOut,
    void *ws, uint64_t ws_bytes, void *stream);

/* Same two phases with an explicit kernel choice (a wq_kernel value). A forced
 * kernel that cannot run the given shapes returns WQ_ERR_UNSUPPORTED. The
 * workspace size depends on the kernel, so pass the same `kernel` to both. */
int32_t wq_matmul_add_rmsnorm_get_workspace_ex(
    const wq_tensor *x1, const wq_tensor *x2, const wq_tensor *scale,
    const wq_tensor *offset, const wq_tensor *bias, const wq_tensor *residual,
    const wq_tensor *gamma, double eps, int64_t group,
    const wq_tensor *y, const wq_tensor *normOut, int32_t kernel, uint64_t *ws_bytes);

int32_t wq_matmul_add_rmsnorm_ex(
    const wq_tensor *x1, const wq_tensor *x2, const wq_tensor *scale,
    const wq_tensor *offset, const wq_tensor *bias, const wq_tensor *residual,
    const wq_tensor *gamma, double eps, int64_t group,
    const wq_tensor *y, const wq_tensor *normOut, int32_t kernel,
    void *ws, uint64_t ws_bytes, void *stream);

/* Which kernel WQ_KERNEL_AUTO picks for these arguments (a wq_kernel value),
 * or a negative wq_status if the arguments are invalid. Host only. */
int32_t wq_matmul_add_rmsnorm_select_kernel(
    const wq_tensor *x1, const wq_tensor *x2, const wq_tensor *scale,
    const wq_tensor *offset, const wq_tensor *bias, const wq_tensor *residual,
    const wq_tensor *gamma, double eps, int64_t group,
    const wq_tensor *y, const wq_tensor *normOut);

/* ------------------------------------------------------------------ mx block-scaled matmul */

/* First phase of the mx block-scaled matmul with in-place add
 * (aclnnQuantBatchMatmulInplaceAdd, "Function description", mx quantization):
 *     y[m,n] += sum_j (sum_{k in slice j} x1[m,k] * x2[k,n]) * scale1[m,j] * scale2[j,n]
 * over slices of gsK = 32 along K (kLoops = ceil(K/32), the last slice may be
 * short).
 *   x1      WQ_FP4_E2M1 (M, K), K even, packed along K; or WQ_FP4_E2M1_T,
 *           stored (K, M) packed along M, M even (the page's transposeX1 =
 *           true, the form its constraints list as supported).
 *   scale1  WQ_E8M0 (M, ceil(K/32)); with a transposed x1, stored (ceil(K/32), M)
 *           (the scales follow x1's storage order: a reading, the page's table
 *           of scale shapes is not legible).
 *   x2      WQ_FP4_E2M1 (K, N), N even, packed along N.
 *   scale2  WQ_E8M0 (ceil(K/32), N).
 *   y       WQ_F32 (M, N), read and written (it must not overlap the inputs).
 *   ws_bytes out: 0.
 * Each slice's sum of products is exact (a multiple of 1/4 below 2^11). With
 * the default kernel (tensor cores, WQ_MX_KERNEL_TENSOR) the scaled slices are
 * added in fp32, one rounding per slice: |error| <= (kLoops + 3) * 2^-24 *
 * (|y| + sum_j |slice_j * scale1 * scale2|) plus subnormal rounding. With
 * WQ_MX_KERNEL_EXACT (CUDA cores) they are added in fp64 and the sum is added
 * to y and rounded once to fp32: the exactly rounded result unless the fp64
 * sum itself rounds. Errors: WQ_ERR_NULL, WQ_ERR_DTYPE, WQ_ERR_SHAPE,
 * WQ_ERR_ALIAS. Touches no device memory. */
int32_t wq_mx_matmul_add_get_workspace(const wq_tensor *x1, const wq_tensor *scale1,
                                       const wq_tensor *x2, const wq_tensor *scale2,
                                       const wq_tensor *y, uint64_t *ws_bytes);

/* Second phase: enqueue the product on `stream` (the tensor-core kernel). */
int32_t wq_mx_matmul_add(const wq_tensor *x1, const wq_tensor *scale1, const wq_tensor *x2,
                         const wq_tensor *scale2, const wq_tensor *y, void *ws, uint64_t ws_bytes,
                         void *stream);

enum { WQ_MX_KERNEL_TENSOR = 0, WQ_MX_KERNEL_EXACT = 1 };

/* The same with a choice of kernel (WQ_MX_KERNEL_*; anything else is
 * WQ_ERR_UNSUPPORTED). */
int32_t wq_mx_matmul_add_ex(const wq_tensor *x1, const wq_tensor *scale1, const wq_tensor *x2,
                            const wq_tensor *scale2, const wq_tensor *y, int32_t kernel, void *ws,
                            uint64_t ws_bytes, void *stream);

/* ------------------------------------------------------------------ dynamic quantization */

/* First phase of the per-token symmetric dynamic quantization
 * (aclnnDynamicQuant, "Function description": scaleOut = row_max(|input|) /
 * dtypeMax, yOut = round(input / scaleOut), input = x or x * smoothScales).
 *   x              WQ_F16 or WQ_BF16, 1-D (K), 2-D (M, K) or 3-D (b, s, K);
 *                  1 <= K <= 65535. Rows are the leading dimensions.
 *   smooth_scales  NULL or (K), x's dtype: multiplies column k before the
 *                  maximum is taken.
 *   y              out: WQ_INT8 with x's shape (dtypeMax 127), or WQ_INT4 with
 *                  x's logical shape, K even, packed two per byte along the row
 *                  like the weight pack (dtypeMax 7); read as little-endian int32
 *                  words it is the page's INT32 output (8 codes per word).
 *   scale          out: WQ_F32 with x's leading shape ((1) for a 1-D x).
 *   ws_bytes       out: 0.
 * Every step is one IEEE fp32 operation (x * smooth, the maximum, max /
 * dtypeMax, x / scale), round() is round half to even, a code is clamped to
 * [-dtypeMax, dtypeMax] and a NaN quotient gives 0, and a row whose maximum is
 * 0 gets scale 0 and codes 0 (readings where the page is silent). Errors:
 * WQ_ERR_NULL, WQ_ERR_DTYPE, WQ_ERR_SHAPE, WQ_ERR_ALIAS. Touches no device memory. */
int32_t wq_dynamic_quant_get_workspace(const wq_tensor *x, const wq_tensor *smooth_scales,
                                       const wq_tensor *y, const wq_tensor *scale,
                                       uint64_t *ws_bytes);

/* Second phase: enqueue the quantization on `stream`. Bit-exact and
 * deterministic (the maximum is order-independent); M = 0 enqueues nothing. */
int32_t wq_dynamic_quant(const wq_tensor *x, const wq_tensor *smooth_scales, const wq_tensor *y,
                         const wq_tensor *scale, void *ws, uint64_t ws_bytes, void *stream);

/* ------------------------------------------------------------------ no-alloc variant */

/* The operator pages have no counterpart to this entry point.
 *
 * For callers that cannot allocate device memory or hand over a workspace --
 * a host framework whose custom-operator interface passes only inputs and
 * outputs, or a runtime that fixes its device memory at start-up and forbids
 * later allocations (cudaMalloc may synchronize the device, fail under memory
 * pressure or fragment a planned heap mid-run). It computes exactly what
 * wq_matmul_add_rmsnorm computes, with the same kernels, but takes no workspace:
 * its scratch memory is a fixed array of WQ_NOALLOC_SCRATCH_BYTES inside the
 * library, which every GPU that loads the library holds until the process
 * exits. It calls no cudaMalloc, cudaFree or other allocating routine.
 *   - Arguments, validation and errors are those of wq_matmul_add_rmsnorm.
 *   - A problem whose workspace (as wq_matmul_add_rmsnorm_get_workspace
 *     reports it) exceeds WQ_NOALLOC_SCRATCH_BYTES is rejected with
 *     WQ_ERR_WORKSPACE before anything is enqueued.
 *   - The first call in each CUDA context (in practice: on each device) looks
 *     up that context's address of the array (cudaGetSymbolAddress with the
 *     device current); make that first call before any stream capture.
 *   - All calls share the one array per device and it keeps the last call's
 *     contents (each call clears the part that must start at zero). Calls whose
 *     work overlaps on the GPU -- on different streams or from different host
 *     threads without ordering -- race on it and give wrong results. */
#define WQ_NOALLOC_SCRATCH_BYTES (8ull << 20)

int32_t wq_matmul_add_rmsnorm_noalloc(
    const wq_tensor *x1, const wq_tensor *x2, const wq_tensor *scale,
    const wq_tensor *offset, const wq_tensor *bias, const wq_tensor *residual,
    const wq_tensor *gamma, double eps, int64_t group,
    const wq_tensor *y, const wq_tensor *normOut, void *stream);

/* Device status word of the no-alloc scratch of the current device, as
 * wq_read_device_status gives it for a workspace: synchronizes `stream`, copies
 * the word to the host and stores it in *device_status (0 = no device-side
 * error). Read it after a wq_matmul_add_rmsnorm_noalloc call and before the
 * next one, which clears it. Returns WQ_ERR_NULL or WQ_ERR_CUDA on failure.
 * (No counterpart on the pages, like the entry point it serves.) */
int32_t wq_noalloc_read_device_status(void *stream, int32_t *device_status);

/* ------------------------------------------------------------------ status */

/* Device status word of a workspace after the work enqueued on `stream` has
 * finished: synchronizes `stream`, copies the word to the host and stores it in
 * *device_status (0 = no device-side error; otherwise WQ_ERR_DEVICE_TIMEOUT in
 * the low 8 bits and the place that gave up in the upper bits). A kernel whose
 * bounded wait for other thread blocks runs out stops waiting, sets this word,
 * skips the dependent writes and exits, so the CUDA context stays usable.
 * Returns WQ_ERR_NULL, WQ_ERR_WORKSPACE (ws_bytes < 16) or WQ_ERR_CUDA on
 * failure. */
int32_t wq_read_device_status(const void *ws, uint64_t ws_bytes, void *stream,
                              int32_t *device_status);

/* Self-check of the device error channel (no counterpart on the pages): one
 * thread waits, with the library's bounded wait, for an mbarrier phase that
 * nothing completes; after `budget_cycles` SM clock cycles (clamped to
 * [1000, 4e9]) the wait gives up and records WQ_ERR_DEVICE_TIMEOUT with place
 * WQ_WHERE_SELF_CHECK in the status word of `ws`, exactly as an operator kernel
 * whose wait ran out would, and the kernel exits. Nothing faults and the CUDA
 * context stays usable; read the word with wq_read_device_status, then zero the
 * workspace header before the workspace serves an operator call again.
 * Asynchronous on `stream`. Returns WQ_ERR_NULL, WQ_ERR_WORKSPACE
 * (ws_bytes < 2048) or WQ_ERR_CUDA. */
#define WQ_WHERE_SELF_CHECK 31
int32_t wq_check_device_timeout(void *ws, uint64_t ws_bytes, uint64_t budget_cycles, void *stream);

/* Test hook of the device error channel (no counterpart on the pages). For
 * every later launch in this process, the operator kernels' waits for other
 * thread blocks -- the decode kernel's grid-wide counter (place
 * WQ_WHERE_DECODE_GRID) and the prefill kernel's row-block counters (place
 * WQ_WHERE_PREFILL_ROW_BLOCK) -- give up after `budget_cycles` SM clock cycles
 * (in [1000, 4e9]) and wait for `extra_arrivals` (<= 2^20) more arrivals than
 * the kernel makes. With extra_arrivals > 0 every such wait runs out: the
 * kernel records WQ_ERR_DEVICE_TIMEOUT | place << 8 in the status word, writes
 * no normOut, drains its copies and MMAs, frees its tensor memory and exits; the
 * call itself returns WQ_OK. (0, 0) restores the defaults (about 2 s, no extra
 * arrivals). Process-wide and not thread-safe with respect to calls in flight:
 * for tests only. Returns WQ_ERR_SHAPE for values out of range. */
#define WQ_WHERE_PREFILL_ROW_BLOCK 5
#define WQ_WHERE_DECODE_GRID 15
int32_t wq_test_set_wait_limits(uint64_t budget_cycles, uint32_t extra_arrivals);

/* Static description of a status code ("WQ_OK", "WQ_ERR_SHAPE", ...). */
const char *wq_status_string(int32_t status);

/* Thread-local detail of the last error returned on this thread ("" if none). */
const char *wq_last_error(void);

/* Library version as major*10000 + minor*100 + patch. */
int32_t wq_version(void);

#ifdef __cplusplus
}
#endif

#endif /* WQ_H_ */
