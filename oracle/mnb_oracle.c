/*
 * mnb_oracle.c -- the CPU oracle for the block-quantized MatMulNBits product
 * with an optional rank-r LoRA term.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or calls
 * this file: only the tests, the package smoke check and the benchmark's
 * CPU-baseline leg do.  It shares no code, header, table or helper with the
 * CUDA library.
 *
 * What it computes is the plain definition, written out step by step, in
 * IEEE binary64 ("fp64") so that every intermediate that is exact in the
 * definition is exact here too:
 *
 *   w[n,k] = (q[n,k] - zp[n, k/bs]) * scale[n, k/bs]                  (dequant)
 *   t[m,r] = sum_k x[m,k] * A[k,r]                                     (LoRA down)
 *   y[m,n] = sum_k x[m,k] * w[n,k]  +  sum_r t[m,r] * B[n,r]           (base + LoRA up)
 *            (+ bias[n] when a bias is given)
 *   Y[m,n] = fp16_round_to_nearest_even(y[m,n])
 *
 * Sources, cited by page title and section:
 *  - "[WebGPU] Fuse rank-32 quantized LoRA with MatMulNBits" (onnxruntime pull
 *    request 33370), commit message that adds the opt-in MatMulNBitsLoRA
 *    operator: INT4 / block-32 base weights, FP16 rank-32 adapters, the output
 *    is base + T * Bt^T with T = X * A, an empty adapter runs the base
 *    projection only, B is read in its transposed [N, r] layout.
 *  - Same page, "Description": the fused operator covers the base projection,
 *    the LoRA down and up projections and the residual addition.
 *  - "Fuse DQ->MatMulNBits for shared initializers and skip outer-scope
 *    weights" (onnxruntime pull request 33800), "Description" and the repro
 *    under "Motivation and Context": DequantizeLinear(w_q, w_scale, w_zp)
 *    followed by MatMul is the computation MatMulNBits replaces, i.e. the
 *    dequant map is (q - zp) * scale and the weight is used transposed.
 *
 * Readings where the pages leave a step open:
 *  - INT4 packing: two 4-bit codes per byte along K; element k = 2j sits in
 *    the low nibble (bits 0..3) of byte j of the block, k = 2j + 1 in the
 *    high nibble.  INT8: one code per byte.  INT2 (the 2-bit weights of the
 *    empty-packed-weights commit's tests): four codes per byte, the same
 *    low-bits-first order, element k = 4j + i in bits 2i..2i+1 of byte j.
 *  - Zero points: one unsigned byte per (row, block), used as given; when no
 *    array is passed the default is 2^(bits-1) (2 for INT2, 8 for INT4, 128
 *    for INT8).
 *  - T is kept exact (fp64) here; the fused GPU path rounds T to FP16 as the
 *    pages do.  mnb_ref_run can also round T first (round_t = 1).
 *  - Bias: "[WebGPU] Fuse rank-32 quantized LoRA with MatMulNBits", the
 *    referenced commit "Support empty packed weights in CPU and WebGPU
 *    MatMulNBits", Description: with empty weights the output holds zeros or
 *    the broadcast bias.  Read as: an optional FP16 vector over N added to
 *    every output row before the one rounding (mnb_ref_run_bias).
 *
 *  - INT8 adapters (mnb_ref_run_qlora): each adapter projection is an 8-bit
 *    block-32 MatMulNBits weight, the down one [rank rows x K], the up one
 *    [N rows x rank]; dequantized exactly, then the same product.
 *
 * Everything is plain loops; OpenMP only splits independent output rows.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ---------------------------------------------------------------------------
 * IEEE 754 binary16 <-> binary64, written from the format's definition:
 * 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits; exponent field 0
 * holds the subnormals m * 2^-24, field 31 holds inf / NaN.
 * ------------------------------------------------------------------------- */

double mnb_ref_f16_to_f64(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0) {
        v = ldexp((double)f, -24);
    } else if (e == 31) {
        v = (f == 0) ? INFINITY : NAN;
    } else {
        v = ldexp((double)(1024 + f), e - 15 - 10);
    }
    return sign ? -v : v;
}

/* Round a non-negative real m to the nearest integer, ties to the even one. */
static double round_half_even(double m)
{
    double fl = floor(m);
    double d = m - fl; /* exact: m and fl share the exponent range used here */
    if (d > 0.5) return fl + 1.0;
    if (d < 0.5) return fl;
    return (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;
}

uint16_t mnb_ref_f64_to_f16(double v)
{
    uint16_t sign = signbit(v) ? 0x8000u : 0u;
    double a = fabs(v);
    if (isnan(v)) return (uint16_t)(sign | 0x7e00u);
    /* 65520 is the midpoint between the largest finite value 65504 (odd
     * fraction 0x3ff) and 2^16; the tie goes to the even neighbour, i.e. to
     * infinity. */
    if (a >= 65520.0) return (uint16_t)(sign | 0x7c00u);
    if (a < ldexp(1.0, -14)) {
        /* subnormal range: a = m * 2^-24 with m real in [0, 1024) */
        double m = round_half_even(ldexp(a, 24));
        return (uint16_t)(sign | (uint16_t)m); /* m == 1024 is the smallest normal */
    }
    int e2;
    (void)frexp(a, &e2);          /* a = f * 2^e2, f in [0.5, 1) */
    int E = e2 - 1;               /* 2^E <= a < 2^(E+1), E in [-14, 15] */
    double m = round_half_even(ldexp(a, 10 - E)); /* significand in [1024, 2048] */
    if (m == 2048.0) { m = 1024.0; E += 1; }
    if (E > 15) return (uint16_t)(sign | 0x7c00u);
    return (uint16_t)(sign | (uint16_t)((E + 15) << 10) | (uint16_t)((int)m - 1024));
}

/* ---------------------------------------------------------------------------
 * Packing of the quantized codes.  Wq is [N, K/bs, bs*bits/8] bytes, i.e.
 * each output row n holds its K codes in order along K.
 * ------------------------------------------------------------------------- */

static int check_shape(int64_t N, int64_t K, int bits, int bs)
{
    if (N < 0 || K < 0) return -1;
    if (bits != 2 && bits != 4 && bits != 8) return -2;
    if (bs <= 0 || (bs * bits) % 8 != 0) return -2;
    if (K % bs != 0) return -2;
    return 0;
}

/* code q[n,k] read from the packed weight bytes: row n is K * bits / 8 bytes,
 * code k is in byte k / per_byte at bit bits * (k % per_byte) */
static int code_at(const uint8_t* Wq, int64_t K, int bits, int64_t n, int64_t k)
{
    int per_byte = 8 / bits;
    uint8_t byte = Wq[n * (K / per_byte) + k / per_byte];
    return (byte >> (bits * (int)(k % per_byte))) & ((1 << bits) - 1);
}

int mnb_ref_unpack(const uint8_t* Wq, int64_t N, int64_t K, int bits, int bs, uint8_t* q)
{
    int rc = check_shape(N, K, bits, bs);
    if (rc) return rc;
    for (int64_t n = 0; n < N; ++n)
        for (int64_t k = 0; k < K; ++k) q[n * K + k] = (uint8_t)code_at(Wq, K, bits, n, k);
    return 0;
}

int mnb_ref_pack(const uint8_t* q, int64_t N, int64_t K, int bits, int bs, uint8_t* Wq)
{
    int rc = check_shape(N, K, bits, bs);
    if (rc) return rc;
    int per_byte = 8 / bits, mask = (1 << bits) - 1;
    for (int64_t n = 0; n < N; ++n)
        for (int64_t j = 0; j < K / per_byte; ++j) {
            int byte = 0;
            for (int i = 0; i < per_byte; ++i) byte |= (q[n * K + j * per_byte + i] & mask) << (bits * i);
            Wq[n * (K / per_byte) + j] = (uint8_t)byte;
        }
    return 0;
}

/* ---------------------------------------------------------------------------
 * Dequantization: w = (q - zp) * scale, one (scale, zp) per row and block.
 * The product of an integer of at most 9 bits and an 11-bit significand is
 * exact in binary64.
 * ------------------------------------------------------------------------- */

static double dequant_at(const uint8_t* Wq, const uint16_t* scales, const uint8_t* zp,
                         int64_t K, int bits, int bs, int64_t n, int64_t k)
{
    int64_t nb = K / bs, b = k / bs;
    int q = code_at(Wq, K, bits, n, k);
    int z = zp ? (int)zp[n * nb + b] : (1 << (bits - 1));
    double s = mnb_ref_f16_to_f64(scales[n * nb + b]);
    return (double)(q - z) * s;
}

int mnb_ref_dequant(const uint8_t* Wq, const uint16_t* scales, const uint8_t* zp,
                    int64_t N, int64_t K, int bits, int bs, double* W)
{
    int rc = check_shape(N, K, bits, bs);
    if (rc) return rc;
    for (int64_t n = 0; n < N; ++n)
        for (int64_t k = 0; k < K; ++k) W[n * K + k] = dequant_at(Wq, scales, zp, K, bits, bs, n, k);
    return 0;
}

/* The dequantized weight rounded once to binary16 (what a kernel that stages
 * FP16 weights for a tensor-core product must hold, bit for bit). */
int mnb_ref_dequant_f16(const uint8_t* Wq, const uint16_t* scales, const uint8_t* zp,
                        int64_t N, int64_t K, int bits, int bs, uint16_t* W16)
{
    int rc = check_shape(N, K, bits, bs);
    if (rc) return rc;
    for (int64_t n = 0; n < N; ++n)
        for (int64_t k = 0; k < K; ++k)
            W16[n * K + k] = mnb_ref_f64_to_f16(dequant_at(Wq, scales, zp, K, bits, bs, n, k));
    return 0;
}

/* ---------------------------------------------------------------------------
 * LoRA down projection T = X * A, X [Mt, K] fp16, A [K, r] fp16, T fp64.
 * ------------------------------------------------------------------------- */

int mnb_ref_lora_down(const uint16_t* X, const uint16_t* A, int64_t Mt, int64_t K, int r, double* T)
{
    if (Mt < 0 || K < 0 || r < 0) return -1;
    for (int64_t m = 0; m < Mt; ++m)
        for (int j = 0; j < r; ++j) {
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k)
                acc += mnb_ref_f16_to_f64(X[m * K + k]) * mnb_ref_f16_to_f64(A[k * r + j]);
            T[m * r + j] = acc;
        }
    return 0;
}

/* ---------------------------------------------------------------------------
 * The whole operation.  X [Mt, K] fp16 (Mt = batch * M rows, every row is an
 * independent product), Wq / scales / zp as above, A [K, rank] and B [N, rank]
 * fp16 or NULL (rank 0 = empty adapter = base only).
 * Outputs (any may be NULL):
 *   Y16   [Mt, N]  fp16 bits of round-to-nearest-even(y)
 *   Y64   [Mt, N]  y in binary64
 *   bound [Mt, N]  sum_k |x w| + sum_r |t B|, the scale of the FP16
 *                  tolerance |y_gpu - y| <= 1e-3 * bound + 1e-3
 * round_t = 1 rounds each t[m,r] to fp16 before the up projection (the
 * pages' FP16 intermediate); 0 keeps it exact.
 * ------------------------------------------------------------------------- */

/* The product with the adapter given as exact values: A64 [K, rank],
 * B64 [N, rank] (either adapter format is turned into these first). */
static int run_core(const uint16_t* X, const uint8_t* Wq, const uint16_t* scales, const uint8_t* zp,
                    const double* A64, const double* B64, int rank, const uint16_t* bias,
                    int64_t Mt, int64_t N, int64_t K, int bits, int bs, int round_t,
                    uint16_t* Y16, double* Y64, double* bound)
{
    double* T = NULL;
    if (rank > 0) {
        T = (double*)malloc(sizeof(double) * (size_t)(Mt > 0 ? Mt : 1) * (size_t)rank);
        if (!T) return -3;
        for (int64_t m = 0; m < Mt; ++m)
            for (int j = 0; j < rank; ++j) {
                double t = 0.0;
                for (int64_t k = 0; k < K; ++k) t += mnb_ref_f16_to_f64(X[m * K + k]) * A64[k * rank + j];
                T[m * rank + j] = round_t ? mnb_ref_f16_to_f64(mnb_ref_f64_to_f16(t)) : t;
            }
    }

    int64_t total = Mt * N;
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < total; ++i) {
        int64_t m = i / N, n = i % N;
        double acc = 0.0, mag = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            double p = mnb_ref_f16_to_f64(X[m * K + k]) * dequant_at(Wq, scales, zp, K, bits, bs, n, k);
            acc += p;
            mag += fabs(p);
        }
        for (int j = 0; j < rank; ++j) {
            double p = T[m * rank + j] * B64[n * rank + j];
            acc += p;
            mag += fabs(p);
        }
        if (bias) {
            double b = mnb_ref_f16_to_f64(bias[n]);
            acc += b;
            mag += fabs(b);
        }
        if (Y64) Y64[i] = acc;
        if (bound) bound[i] = mag;
        if (Y16) Y16[i] = mnb_ref_f64_to_f16(acc);
    }
    free(T);
    return 0;
}

int mnb_ref_run_bias(const uint16_t* X, const uint8_t* Wq, const uint16_t* scales, const uint8_t* zp,
                     const uint16_t* A, const uint16_t* B, int rank, const uint16_t* bias,
                     int64_t Mt, int64_t N, int64_t K, int bits, int bs, int round_t,
                     uint16_t* Y16, double* Y64, double* bound)
{
    int rc = check_shape(N, K, bits, bs);
    if (rc) return rc;
    if (Mt < 0 || rank < 0) return -1;
    if (rank > 0 && (!A || !B)) return -1;
    double *A64 = NULL, *B64 = NULL;
    if (rank > 0) {
        A64 = (double*)malloc(sizeof(double) * (size_t)(K > 0 ? K : 1) * (size_t)rank);
        B64 = (double*)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1) * (size_t)rank);
        if (!A64 || !B64) {
            free(A64);
            free(B64);
            return -3;
        }
        for (int64_t i = 0; i < K * rank; ++i) A64[i] = mnb_ref_f16_to_f64(A[i]);
        for (int64_t i = 0; i < N * rank; ++i) B64[i] = mnb_ref_f16_to_f64(B[i]);
    }
    rc = run_core(X, Wq, scales, zp, A64, B64, rank, bias, Mt, N, K, bits, bs, round_t, Y16, Y64, bound);
    free(A64);
    free(B64);
    return rc;
}

/* ---------------------------------------------------------------------------
 * INT8 block-32 adapters ("[WebGPU] Fuse rank-32 quantized LoRA with
 * MatMulNBits", commit message adding the INT8-adapter kernels and the later
 * MatMulNBitsQLoRA commit: INT4 base weights with block-32 INT8 rank-32
 * adapters, the adapters' original INT8 arithmetic kept).  Reading: each
 * adapter projection is itself an 8-bit MatMulNBits weight --
 *   down: Aq [rank, K/bs, bs] with A_scales / A_zp [rank, K/bs]
 *         (rank output rows along K), a[k, r] = dequant of row r, column k;
 *   up:   Bq [N, rank/bs, bs] with B_scales / B_zp [N, rank/bs]
 *         (N output rows along the rank), b[n, r] = dequant of row n, column r;
 * zero points NULL = the 8-bit default 128.  The dequantized values are exact
 * here; the rest is the product above.
 * ------------------------------------------------------------------------- */

int mnb_ref_run_qlora(const uint16_t* X, const uint8_t* Wq, const uint16_t* scales, const uint8_t* zp,
                      const uint8_t* Aq, const uint16_t* A_scales, const uint8_t* A_zp,
                      const uint8_t* Bq, const uint16_t* B_scales, const uint8_t* B_zp, int rank,
                      const uint16_t* bias, int64_t Mt, int64_t N, int64_t K, int bits, int bs, int round_t,
                      uint16_t* Y16, double* Y64, double* bound)
{
    int rc = check_shape(N, K, bits, bs);
    if (rc) return rc;
    if (Mt < 0 || rank < 0) return -1;
    if (rank > 0 && (!Aq || !A_scales || !Bq || !B_scales)) return -1;
    if (rank > 0 && (check_shape(rank, K, 8, bs) || check_shape(N, rank, 8, bs))) return -2;
    double *A64 = NULL, *B64 = NULL;
    if (rank > 0) {
        A64 = (double*)malloc(sizeof(double) * (size_t)(K > 0 ? K : 1) * (size_t)rank);
        B64 = (double*)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1) * (size_t)rank);
        if (!A64 || !B64) {
            free(A64);
            free(B64);
            return -3;
        }
        for (int r = 0; r < rank; ++r)
            for (int64_t k = 0; k < K; ++k) A64[k * rank + r] = dequant_at(Aq, A_scales, A_zp, K, 8, bs, r, k);
        for (int64_t n = 0; n < N; ++n)
            for (int r = 0; r < rank; ++r) B64[n * rank + r] = dequant_at(Bq, B_scales, B_zp, rank, 8, bs, n, r);
    }
    rc = run_core(X, Wq, scales, zp, A64, B64, rank, bias, Mt, N, K, bits, bs, round_t, Y16, Y64, bound);
    free(A64);
    free(B64);
    return rc;
}

/* ---------------------------------------------------------------------------
 * The int8-activation base ("accuracy level 4" in "[WebGPU] Fuse rank-32
 * quantized LoRA with MatMulNBits", Performance, and in "Fuse DQ->MatMulNBits
 * for shared initializers and skip outer-scope weights", Motivation and
 * Context; the MatMulNBitsLoRA commit keeps "DP4A activation quantization for
 * the base, with original FP16 X for T").  The pages name the method, not its
 * steps; the reading written out here:
 *   per row m and block b of 32 along K, in binary32:
 *     amax = max_k |x[m,k]|                      (exact)
 *     amax == 0:  xq = 0, xs = 0
 *     else:       inv = 127 / amax,  xq = clamp(rint(x * inv), -127, 127),
 *                 xs = amax / 127                 (each op rounded to nearest)
 *   base[m,n] = sum_b xs[m,b] * s[n,b] * sum_{k in b} xq[m,k] (q[n,k] - zp[n,b])
 * the inner sum an exact integer (the DP4A / integer-MMA product).  T, the
 * adapter term and the bias as in the plain product (T from the FP16 X).
 * ------------------------------------------------------------------------- */

int mnb_ref_quantize_x(const uint16_t* X, int64_t Mt, int64_t K, int bs, int8_t* Xq, float* Xs)
{
    if (Mt < 0 || K < 0 || bs <= 0 || K % bs != 0) return -2;
    int64_t nb = K / bs;
    for (int64_t m = 0; m < Mt; ++m)
        for (int64_t b = 0; b < nb; ++b) {
            const uint16_t* x = X + m * K + b * bs;
            float amax = 0.0f;
            for (int k = 0; k < bs; ++k) {
                float a = fabsf((float)mnb_ref_f16_to_f64(x[k]));
                if (a > amax) amax = a;
            }
            int8_t* q = Xq + m * K + b * bs;
            if (amax == 0.0f) {
                for (int k = 0; k < bs; ++k) q[k] = 0;
                Xs[m * nb + b] = 0.0f;
                continue;
            }
            float inv = 127.0f / amax;
            for (int k = 0; k < bs; ++k) {
                float r = rintf((float)mnb_ref_f16_to_f64(x[k]) * inv);
                if (r > 127.0f) r = 127.0f;
                if (r < -127.0f) r = -127.0f;
                q[k] = (int8_t)r;
            }
            Xs[m * nb + b] = amax / 127.0f;
        }
    return 0;
}

int mnb_ref_run_q8x(const uint16_t* X, const uint8_t* Wq, const uint16_t* scales, const uint8_t* zp,
                    const uint16_t* A, const uint16_t* B, int rank, const uint16_t* bias,
                    int64_t Mt, int64_t N, int64_t K, int bits, int bs, int round_t,
                    uint16_t* Y16, double* Y64, double* bound)
{
    int rc = check_shape(N, K, bits, bs);
    if (rc) return rc;
    if (Mt < 0 || rank < 0) return -1;
    if (rank > 0 && (!A || !B)) return -1;
    int64_t nb = K / bs;
    int8_t* Xq = (int8_t*)malloc((size_t)(Mt * K > 0 ? Mt * K : 1));
    float* Xs = (float*)malloc(sizeof(float) * (size_t)(Mt * nb > 0 ? Mt * nb : 1));
    double* T = (double*)malloc(sizeof(double) * (size_t)(Mt > 0 ? Mt : 1) * (size_t)(rank > 0 ? rank : 1));
    if (!Xq || !Xs || !T) {
        free(Xq);
        free(Xs);
        free(T);
        return -3;
    }
    mnb_ref_quantize_x(X, Mt, K, bs, Xq, Xs);
    if (rank > 0) {
        mnb_ref_lora_down(X, A, Mt, K, rank, T);
        if (round_t)
            for (int64_t i = 0; i < Mt * rank; ++i) T[i] = mnb_ref_f16_to_f64(mnb_ref_f64_to_f16(T[i]));
    }
    int64_t total = Mt * N;
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < total; ++i) {
        int64_t m = i / N, n = i % N;
        double acc = 0.0, mag = 0.0;
        for (int64_t b = 0; b < nb; ++b) {
            int64_t dot = 0, adot = 0;
            int z = zp ? (int)zp[n * nb + b] : (1 << (bits - 1));
            for (int64_t k = b * bs; k < (b + 1) * bs; ++k) {
                int64_t p = (int64_t)Xq[m * K + k] * (code_at(Wq, K, bits, n, k) - z);
                dot += p;
                adot += p < 0 ? -p : p;
            }
            double sc = (double)Xs[m * nb + b] * mnb_ref_f16_to_f64(scales[n * nb + b]);
            acc += sc * (double)dot;
            mag += fabs(sc) * (double)adot;
        }
        for (int j = 0; j < rank; ++j) {
            double p = T[m * rank + j] * mnb_ref_f16_to_f64(B[n * rank + j]);
            acc += p;
            mag += fabs(p);
        }
        if (bias) {
            double bv = mnb_ref_f16_to_f64(bias[n]);
            acc += bv;
            mag += fabs(bv);
        }
        if (Y64) Y64[i] = acc;
        if (bound) bound[i] = mag;
        if (Y16) Y16[i] = mnb_ref_f64_to_f16(acc);
    }
    free(Xq);
    free(Xs);
    free(T);
    return 0;
}

/* mnb_ref_run_bias without a bias. */
int mnb_ref_run(const uint16_t* X, const uint8_t* Wq, const uint16_t* scales, const uint8_t* zp,
                const uint16_t* A, const uint16_t* B, int rank,
                int64_t Mt, int64_t N, int64_t K, int bits, int bs, int round_t,
                uint16_t* Y16, double* Y64, double* bound)
{
    return mnb_ref_run_bias(X, Wq, scales, zp, A, B, rank, NULL, Mt, N, K, bits, bs, round_t, Y16, Y64, bound);
}

/* Threads the parallel loop above will use. */
int mnb_ref_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
