/*
 * Plain fp64 CPU oracle for the weight-only quantized matmul with fused
 * residual-add + RMSNorm, and for the INT32 -> dense INT4 weight pack.
 *
 * TEST INFRASTRUCTURE ONLY. This file is the independent checker for the CUDA
 * library in weight_only_bit_pack_b300/. It shares no code, header, table or
 * helper with it and must never be linked into, or called from, the product
 * path. Only tests/, __graft_entry__.smoke() and bench.py's cpu_baseline /
 * --impl reference leg may load it.
 *
 * What it follows (page titles and sections of the Ascend CANN operator docs):
 *   - aclnnConvertWeightToINT4Pack, "Function description": INT32 values that
 *     hold 4-bit integers are re-laid out from sparse storage (one per int32)
 *     to dense storage (two per byte).
 *   - aclnnDynamicQuant, "Constraints": an INT4 output needs its last
 *     dimension divisible by 2 and an INT32-packed output needs it divisible by
 *     8, i.e. packing runs along the LAST dimension.
 *   - aclnnWeightQuantMatmulAllReduceAddRmsNorm, "Function description",
 *     formula: mm_out = allReduce(x1 @ (x2*antiquantScale + antiquantOffset)
 *     + bias); y = mm_out + residual; normOut = y / RMS(y) * gamma with
 *     RMS(y) = sqrt((1/d) * sum_i y_i^2 + epsilon).
 *   - same page, "Constraints": antiquantScale is (1) per-tensor, (n)/(1,n)
 *     per-channel, (ceil(k/groupSize), n) per-group; antiquantOffset has the
 *     scale's shape.
 *
 * Readings where the pages are silent (each one is listed with its reason in
 * the repository's design notes):
 *   - nibble order: the element in even column 2j goes to bits 3:0 of byte j,
 *     the element in column 2j+1 to bits 7:4.
 *   - an INT32 outside [-8, 7] keeps its low four bits (two's complement
 *     truncation), so the pack is defined for every input.
 *   - the offset is added after scaling: W = q*S + O.
 *   - per-group row r(k) = floor(k / g); the last group may be short.
 *   - d in RMS is n, the last dimension of y; epsilon sits inside the sqrt.
 *   - allReduce over one rank is the identity, so bias is added once.
 *
 * Everything is fp64 with no intermediate rounding. Each output element of the
 * matmul is summed over k in ascending order. Rows are independent, so the
 * caller may pass any subset of rows of x1/residual (row sampling).
 *
 * Parity status: every function here is pinned by tests/test_oracle.py
 * (closed forms, library matmul, exhaustive nibble round trip, hand-worked
 * cases). Nothing is "parity unpinned".
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <math.h>

#define WQO_OK 0
#define WQO_EINVAL 1
#define WQO_ENOMEM 2

/* Pack: v is (K, N) int32, row-major; out is (K, N/2) bytes. N must be even. */
int wqo_pack_int4(const int32_t *v, int64_t K, int64_t N, uint8_t *out)
{
    if (K < 0 || N < 0 || (N % 2) != 0) return WQO_EINVAL;
    for (int64_t k = 0; k < K; ++k) {
        for (int64_t j = 0; j < N / 2; ++j) {
            uint32_t lo = (uint32_t)v[k * N + 2 * j] & 0xFu;      /* even column */
            uint32_t hi = (uint32_t)v[k * N + 2 * j + 1] & 0xFu;  /* odd column  */
            out[k * (N / 2) + j] = (uint8_t)(lo | (hi << 4));
        }
    }
    return WQO_OK;
}

/* Unpack: inverse of the pack for values in [-8, 7]. A nibble is read as a
 * 4-bit two's complement integer. */
int wqo_unpack_int4(const uint8_t *b, int64_t K, int64_t N, int32_t *out)
{
    if (K < 0 || N < 0 || (N % 2) != 0) return WQO_EINVAL;
    for (int64_t k = 0; k < K; ++k) {
        for (int64_t n = 0; n < N; ++n) {
            uint8_t byte = b[k * (N / 2) + n / 2];
            int32_t nib = (n % 2 == 0) ? (byte & 0xF) : (byte >> 4);
            out[k * N + n] = nib >= 8 ? nib - 16 : nib;
        }
    }
    return WQO_OK;
}

/* Scale/offset element for weight (k, n).
 * S and O are (Gs, Ns) row-major: Gs = 1 unless per-group; Ns = 1 for
 * per-tensor, N otherwise. g = 0 means no grouping. */
static double so_at(const double *T, int64_t Gs, int64_t Ns, int64_t g,
                    int64_t k, int64_t n)
{
    int64_t r = (g > 0) ? k / g : 0;
    int64_t c = (Ns == 1) ? 0 : n;
    (void)Gs;
    return T[r * Ns + c];
}

/* Antiquant: W = q * S + O (O absent -> 0). q and W are (K, N). */
int wqo_dequant(const int32_t *q, int64_t K, int64_t N,
                const double *S, const double *O, int64_t Gs, int64_t Ns,
                int64_t g, double *W)
{
    if (K < 0 || N < 0 || Gs < 1 || Ns < 1) return WQO_EINVAL;
    if (g > 0 && Gs != (K + g - 1) / g) return WQO_EINVAL;
    if (g == 0 && Gs != 1) return WQO_EINVAL;
    if (Ns != 1 && Ns != N) return WQO_EINVAL;
    for (int64_t k = 0; k < K; ++k)
        for (int64_t n = 0; n < N; ++n) {
            double w = (double)q[k * N + n] * so_at(S, Gs, Ns, g, k, n);
            if (O) w += so_at(O, Gs, Ns, g, k, n);
            W[k * N + n] = w;
        }
    return WQO_OK;
}

/* The fused operator on M rows.
 *   x1 (M, K), q (K, N) integer weights (unpacked values), S/O (Gs, Ns),
 *   bias (N) or NULL, residual (M, N), gamma (N).
 * Outputs (any may be NULL): mm (M, N) = x1 @ W + bias, y (M, N), normOut (M, N).
 *
 * The k-sum of every (m, n) runs in ascending k. W[k, :] is formed once per k
 * and applied to every row (a loop order that leaves each sum's order as is).
 * OpenMP threads split the n range; every element is still summed by one
 * thread in ascending k. */
int wqo_matmul_add_rmsnorm(const double *x1, int64_t M, int64_t K,
                           const int32_t *q, int64_t N,
                           const double *S, const double *O, int64_t Gs,
                           int64_t Ns, int64_t g,
                           const double *bias, const double *residual,
                           const double *gamma, double eps,
                           double *mm, double *y, double *normOut)
{
    if (M < 0 || K < 1 || N < 0 || Gs < 1 || Ns < 1 || g < 0) return WQO_EINVAL;
    if (g > 0 && Gs != (K + g - 1) / g) return WQO_EINVAL;
    if (g == 0 && Gs != 1) return WQO_EINVAL;
    if (Ns != 1 && Ns != N) return WQO_EINVAL;
    if (M == 0 || N == 0) return WQO_OK;

    double *acc = (double *)calloc((size_t)(M * N), sizeof(double));
    if (!acc) return WQO_ENOMEM;

    const int64_t NB = 256; /* n-chunk handled by one thread at a time */
    int64_t nchunks = (N + NB - 1) / NB;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t c = 0; c < nchunks; ++c) {
        int64_t n0 = c * NB, n1 = n0 + NB < N ? n0 + NB : N;
        double w[256];
        for (int64_t k = 0; k < K; ++k) {
            for (int64_t n = n0; n < n1; ++n) {
                double wk = (double)q[k * N + n] * so_at(S, Gs, Ns, g, k, n);
                if (O) wk += so_at(O, Gs, Ns, g, k, n);
                w[n - n0] = wk;
            }
            for (int64_t m = 0; m < M; ++m) {
                double xk = x1[m * K + k];
                double *a = acc + m * N;
                for (int64_t n = n0; n < n1; ++n) a[n] += xk * w[n - n0];
            }
        }
    }

    for (int64_t m = 0; m < M; ++m) {
        double ss = 0.0;
        for (int64_t n = 0; n < N; ++n) {
            double v = acc[m * N + n] + (bias ? bias[n] : 0.0);
            if (mm) mm[m * N + n] = v;
            double yv = v + residual[m * N + n];
            acc[m * N + n] = yv;
            ss += yv * yv;
        }
        double rms = sqrt(ss / (double)N + eps);
        for (int64_t n = 0; n < N; ++n) {
            double yv = acc[m * N + n];
            if (y) y[m * N + n] = yv;
            if (normOut) normOut[m * N + n] = yv / rms * gamma[n];
        }
    }
    free(acc);
    return WQO_OK;
}

/* Kernel-native tiled INT4 layout (the library's analogue of the pack page's
 * FRACTAL_NZ output option, aclnnConvertWeightToINT4Pack "Function
 * description": the same pack, re-tiled for the matrix unit; the pages do not
 * fix a tiled layout, so this is the library's own definition).
 *
 * A (K, N) weight, N % 16 == 0, is cut into tiles of 64 k-rows x 16 columns;
 * tile (s, c) (k-rows 64s.., columns 16c..) takes the 512 bytes at
 * (s * N/16 + c) * 512, tiles of one 64-row slab in column order. K is padded
 * with zero nibbles up to a multiple of 64. Inside a tile, element (kk, cc) =
 * (k - 64s, n - 16c) goes to
 *     h = kk / 32, t = (kk % 32) / 8, jl = (kk % 8) / 4, e = kk % 4,
 *     g = cc % 8, upper = cc / 8,
 *     lane = 4g + t, word j = 2h + jl,
 *     nibble p = (e < 2 ? 0 : 2) + upper + 4 * (e % 2),
 *     byte lane*16 + j*4 + p/2, bits 4*(p%2)+3 : 4*(p%2)
 * and holds the low four bits of the value (reading c3), like the ND pack. */
static int64_t tiled_offset(int64_t k, int64_t n, int64_t N, int *shift)
{
    int64_t s = k / 64, c = n / 16, kk = k % 64, cc = n % 16;
    int64_t h = kk / 32, t = (kk % 32) / 8, jl = (kk % 8) / 4, e = kk % 4;
    int64_t g = cc % 8, upper = cc / 8;
    int64_t lane = 4 * g + t, j = 2 * h + jl;
    int64_t p = (e < 2 ? 0 : 2) + upper + 4 * (e % 2);
    *shift = (int)(4 * (p % 2));
    return (s * (N / 16) + c) * 512 + lane * 16 + j * 4 + p / 2;
}

/* Bytes of the tiled layout of a (K, N) weight: ceil(K/64) * 64 * N / 2. */
int64_t wqo_tiled_bytes(int64_t K, int64_t N)
{
    return (K + 63) / 64 * 64 * N / 2;
}

/* Pack v (K, N) int32 into the tiled layout; out holds wqo_tiled_bytes bytes. */
int wqo_pack_int4_tiled(const int32_t *v, int64_t K, int64_t N, uint8_t *out)
{
    if (K < 0 || N < 0 || (N % 16) != 0) return WQO_EINVAL;
    memset(out, 0, (size_t)wqo_tiled_bytes(K, N));
    for (int64_t k = 0; k < K; ++k)
        for (int64_t n = 0; n < N; ++n) {
            int shift;
            int64_t b = tiled_offset(k, n, N, &shift);
            out[b] |= (uint8_t)(((uint32_t)v[k * N + n] & 0xFu) << shift);
        }
    return WQO_OK;
}

/* Inverse: tiled bytes -> (K, N) int32 values in [-8, 7]. */
int wqo_unpack_int4_tiled(const uint8_t *b, int64_t K, int64_t N, int32_t *out)
{
    if (K < 0 || N < 0 || (N % 16) != 0) return WQO_EINVAL;
    for (int64_t k = 0; k < K; ++k)
        for (int64_t n = 0; n < N; ++n) {
            int shift;
            int64_t o = tiled_offset(k, n, N, &shift);
            int32_t u = (b[o] >> shift) & 0xF;
            out[k * N + n] = u < 8 ? u : u - 16;
        }
    return WQO_OK;
}

/* Per-token symmetric dynamic quantization (aclnnDynamicQuant, "Function
 * description", formula): for each row of x (M rows of K),
 *     input    = x                      (or x * smoothScales, per column)
 *     scaleOut = row_max(|input|) / dtypeMax
 *     yOut     = round(input / scaleOut)
 * with dtypeMax = 127 (INT8) or 7 (INT4). Readings where the page is silent:
 * the arithmetic is fp32 (x * smooth, the maximum, the division by dtypeMax
 * and the division by scaleOut are each one IEEE fp32 operation, as the GPU
 * does them, because the rounding decides an integer); round() is round half
 * to even; a row whose maximum is 0 gets scaleOut = 0 and codes 0; a NaN code
 * becomes 0 and codes are clamped to [-dtypeMax, dtypeMax]. x and smooth hold
 * fp16/bf16 values (exact in fp32). q receives int8 codes (M, K). */
int wqo_dynamic_quant(const float *x, int64_t M, int64_t K, const float *smooth,
                      int qmax, int8_t *q, float *scale)
{
    if (M < 0 || K < 1 || (qmax != 127 && qmax != 7)) return WQO_EINVAL;
    float *row = (float *)malloc((size_t)K * sizeof(float));
    if (!row) return WQO_ENOMEM;
    for (int64_t m = 0; m < M; ++m) {
        float amax = 0.0f;
        for (int64_t k = 0; k < K; ++k) {
            volatile float v = x[m * K + k];
            if (smooth) v = v * smooth[k];
            row[k] = v;
            float a = fabsf(v);
            if (a > amax) amax = a;   /* a NaN element never wins the comparison */
        }
        volatile float s = amax / (float)qmax;
        scale[m] = s;
        for (int64_t k = 0; k < K; ++k) {
            int32_t c = 0;
            if (s != 0.0f) {
                volatile float r = row[k] / s;
                float rr = rintf(r);      /* current rounding mode: to nearest, ties to even */
                if (rr != rr) c = 0;
                else if (rr > (float)qmax) c = qmax;
                else if (rr < (float)-qmax) c = -qmax;
                else c = (int32_t)rr;
            }
            q[m * K + k] = (int8_t)c;
        }
    }
    free(row);
    return WQO_OK;
}

/* FP4 E2M1 pack (aclnnConvertWeightToINT4Pack, "Function description": FLOAT
 * weights are packed into dense FLOAT4_E2M1). An E2M1 code is sign (bit 3),
 * a 2-bit exponent and a 1-bit mantissa: magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6
 * for codes 0..7. A float becomes the nearest magnitude, ties to the even code,
 * saturating at 6 (readings: the page fixes neither rounding nor overflow; a
 * NaN input is outside the operator's domain). Codes pack two per byte along
 * the last dimension, even column in bits 3:0, like the INT4 pack. */
static const double kE2M1[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

static int e2m1_code(double v)
{
    int sign = v < 0 || (v == 0 && signbit(v)) ? 8 : 0;
    double a = fabs(v);
    int best = 0;
    for (int c = 1; c < 8; ++c) {
        double dc = fabs(a - kE2M1[c]), db = fabs(a - kE2M1[best]);
        if (dc < db || (dc == db && (c % 2 == 0))) best = c;  /* tie: the even code */
    }
    if (a >= 6.0) best = 7;
    return sign | best;
}

int wqo_pack_fp4(const float *v, int64_t K, int64_t N, uint8_t *out)
{
    if (K < 0 || N < 0 || (N % 2) != 0) return WQO_EINVAL;
    for (int64_t k = 0; k < K; ++k)
        for (int64_t j = 0; j < N / 2; ++j)
            out[k * (N / 2) + j] = (uint8_t)(e2m1_code(v[k * N + 2 * j]) |
                                             (e2m1_code(v[k * N + 2 * j + 1]) << 4));
    return WQO_OK;
}

static double e2m1_value(int code)
{
    double m = kE2M1[code & 7];
    return (code & 8) ? -m : m;
}

/* mx block-scaled matmul with in-place add (aclnnQuantBatchMatmulInplaceAdd,
 * "Function description", mx quantization formula):
 *   y[m,n] = sum_{j<kLoops} (sum_{k in slice j} x1[m,k] * x2[k,n]) * (scale1[m,j] * scale2[j,n]) + y[m,n]
 * with gsK = 32, kLoops = ceil(K/32) (a short last slice), x1 (M, K) and x2
 * (K, N) FP4 E2M1 codes packed two per byte along their last dimension, and
 * E8M0 scales: byte e stands for 2^(e - 127), and 255 for NaN (the OCP MX
 * encoding; the page does not say). fp64, slices in ascending j. */
int wqo_mx_matmul_add(const uint8_t *x1, const uint8_t *s1, const uint8_t *x2, const uint8_t *s2,
                      int64_t M, int64_t K, int64_t N, double *y)
{
    if (M < 0 || K < 1 || N < 0 || (K % 2) || (N % 2)) return WQO_EINVAL;
    int64_t J = (K + 31) / 32;
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n) {
            double acc = 0.0;
            for (int64_t j = 0; j < J; ++j) {
                double slice = 0.0;
                for (int64_t k = 32 * j; k < K && k < 32 * (j + 1); ++k) {
                    uint8_t a = x1[m * (K / 2) + k / 2], b = x2[k * (N / 2) + n / 2];
                    int ca = (k % 2) ? (a >> 4) : (a & 15), cb = (n % 2) ? (b >> 4) : (b & 15);
                    slice += e2m1_value(ca) * e2m1_value(cb);
                }
                if (s1[m * J + j] == 255 || s2[j * N + n] == 255) acc += NAN;
                else acc += slice * ldexp(1.0, (int)s1[m * J + j] - 127) * ldexp(1.0, (int)s2[j * N + n] - 127);
            }
            y[m * N + n] += acc;
        }
    return WQO_OK;
}
