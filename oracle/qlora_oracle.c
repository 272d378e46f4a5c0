/*
 * qlora_oracle.c -- the plain, slow CPU oracle for the NF4 + double-quantized
 * LoRA linear layer.
 *
 * THIS IS TEST INFRASTRUCTURE. Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg load it. The GPU library shares no code, no
 * header and no constant with this file, and must never call it.
 *
 * Sources (web pages on QLoRA; cited by page title and section):
 *  [QL-note]  inquiringlines.com, "Can we finetune huge language models on a
 *             single GPU?" -- the paragraph on the mechanism (NF4 bins hold an
 *             equal share of a zero-centred normal; double quantization
 *             quantizes the quantization constants; gradients flow through the
 *             frozen 4-bit weights into LoRA adapters).
 *  [QL-70B]   ashishsrivastav.com, "QLoRA: Fine-Tuning a 70B on One GPU" --
 *             sections "NF4 Quantization: Beyond Standard INT4" (16 levels from
 *             the normal CDF, each weight mapped to the closest level, done once
 *             before training) and "Double Quantization: Squeezing the
 *             Constants" (constants stored as INT8; dequantization on the fly
 *             to the compute type).
 *  [QL-host]  serverroom.net, "Fine-tuning an LLM on a GPU: memory requirements
 *             for LoRA and QLoRA" -- section "What LoRA and QLoRA change in
 *             memory" (nf4, double quant, bf16 compute; dropout 0, no bias in
 *             the adapter setup listing).
 *  [QL-mem]   xingyuzhitong.com, "Fine-Tuning Memory Requirements: Full
 *             Training vs LoRA vs QLoRA" -- sections "LoRA: freeze the base,
 *             train small adapters" (r x (d_in + d_out) adapter parameters) and
 *             "QLoRA: quantize the frozen base to 4 bits" (dequantize on the fly).
 *
 * Precision: the codec takes every decision that yields an integer (a 4-bit
 * code, an int8 absmax code) in fp32, the precision the GPU kernels use, and
 * spells out each fp32 rounding. The linear algebra accumulates in fp64.
 * Compile with -ffp-contract=off: no fused multiply-add anywhere.
 *
 * Layout conventions shared with the library's C-ABI (a data format, not code):
 * W is [rows=N out, cols=K in] row-major bf16; blocks of 64 run along the
 * flattened row-major order; byte i of the packed codes holds element 2i in
 * its high nibble and element 2i+1 in its low nibble; absmax codes are int8,
 * one per block; one fp32 scale per group of 256 blocks; one fp32 mean.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define NF4_BLOCK 64
#define DQ_GROUP 256

/* ------------------------------------------------------------------------ */
/* bf16 <-> fp32 (bit-level; bf16 is the upper half of an IEEE binary32).    */
/* ------------------------------------------------------------------------ */
static float bf16_to_f32(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* Round-to-nearest-even from binary32 to bfloat16, for finite inputs. */
static uint16_t f32_to_bf16_rne(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7FFFu + lsb;
    return (uint16_t)(u >> 16);
}

uint16_t oracle_f32_to_bf16(float f) { return f32_to_bf16_rne(f); }

/* Thread count of the OpenMP loops below (for timing the oracle on a given
 * number of host cores; no effect on any result). */
#ifdef _OPENMP
#include <omp.h>
void oracle_set_threads(int n) { if (n > 0) omp_set_num_threads(n); }
int oracle_max_threads(void) { return omp_get_max_threads(); }
#else
void oracle_set_threads(int n) { (void)n; }
int oracle_max_threads(void) { return 1; }
#endif
float oracle_bf16_to_f32(uint16_t h) { return bf16_to_f32(h); }

/* ------------------------------------------------------------------------ */
/* NF4 code table [QL-note mechanism; QL-70B "NF4 Quantization"].            */
/* ------------------------------------------------------------------------ */

/* Standard normal CDF through the complementary error function. */
static double std_normal_cdf(double x) { return 0.5 * erfc(-x / sqrt(2.0)); }

/* Inverse standard normal CDF by bisection until the bracket cannot shrink
 * further in double precision. Slow and obviously monotone. */
double oracle_norm_ppf(double p) {
    double lo = -40.0, hi = 40.0;
    for (int it = 0; it < 4000; ++it) {
        double mid = 0.5 * (lo + hi);
        if (mid <= lo || mid >= hi) break;
        if (std_normal_cdf(mid) < p) lo = mid; else hi = mid;
    }
    /* return the bracket end whose CDF is closer to p */
    return (fabs(std_normal_cdf(lo) - p) <= fabs(std_normal_cdf(hi) - p)) ? lo : hi;
}

double oracle_norm_cdf(double x) { return std_normal_cdf(x); }

/* Outermost probability used for the table. With 16 equal-mass bins the
 * centre of the outermost bin sits at 1 - 1/32; with 15 bins at 1 - 1/30.
 * The table is built from an 8-level half and a 7-level half, so the reading
 * taken here is the average of the two. */
double oracle_nf4_delta(void) { return 0.5 * (31.0 / 32.0 + 29.0 / 30.0); }

/* Probability of level j on a half with n levels: equal steps from 1/2 to
 * delta (j = 1..n). */
double oracle_nf4_prob(int j, int n) {
    double d = oracle_nf4_delta();
    return 0.5 + (d - 0.5) * ((double)j / (double)n);
}

/* Fills L[0..15]: 7 negative levels, an exact zero at code 7, 8 positive
 * levels; each half is divided by its own outermost quantile so that
 * L[0] = -1 and L[15] = +1 exactly. Rounded once from double to fp32. */
void oracle_nf4_table(float L[16]) {
    double pos[9], neg[8];
    for (int j = 1; j <= 8; ++j) pos[j] = oracle_norm_ppf(oracle_nf4_prob(j, 8));
    for (int j = 1; j <= 7; ++j) neg[j] = -oracle_norm_ppf(oracle_nf4_prob(j, 7));
    for (int j = 1; j <= 7; ++j) L[7 - j] = (float)(neg[j] / fabs(neg[7]));
    L[7] = 0.0f;
    for (int j = 1; j <= 8; ++j) L[7 + j] = (float)(pos[j] / pos[8]);
}

/* Nearest level to x (fp32). Distances are compared in double; ties go to
 * the lower code because only a strictly smaller distance moves the choice. */
int oracle_nf4_nearest(float x, const float L[16]) {
    int best = 0;
    double bd = fabs((double)x - (double)L[0]);
    for (int i = 1; i < 16; ++i) {
        double d = fabs((double)x - (double)L[i]);
        if (d < bd) { bd = d; best = i; }
    }
    return best;
}

/* ------------------------------------------------------------------------ */
/* Blockwise absmax + NF4 encode + packing [QL-70B "NF4 Quantization"].     */
/* ------------------------------------------------------------------------ */

/* INT4 baseline table [QL-70B "NF4 Quantization: Beyond Standard INT4": the
 * standard 4-bit integer format has 16 evenly spaced levels]. Reading:
 * symmetric absmax INT4, L[i] = (i - 7) / 7, so code 7 is the exact zero,
 * codes 0 and 14 are -1 and +1, and code 15 (8/7) is never the nearest level
 * of an x in [-1, 1]. Rounded once from double to fp32. */
void oracle_int4_table(float L[16]) {
    for (int i = 0; i < 16; ++i) L[i] = (float)((double)(i - 7) / 7.0);
}

/* Encodes n = rows*cols bf16 weights (n % 64 == 0) with the 16-level table L
 * (NF4 or INT4). Writes the packed codes (n/2 bytes) and the exact per-block
 * absmax (n/64 floats). The codes use the exact absmax: the weights are
 * quantized first, then the constants. */
void oracle_q4_encode(const uint16_t *W, int64_t n, const float L[16], uint8_t *codes, float *absmax) {
    int64_t nb = n / NF4_BLOCK;
#pragma omp parallel for schedule(static)
    for (int64_t b = 0; b < nb; ++b) {
        const uint16_t *w = W + b * NF4_BLOCK;
        float a = 0.0f;
        for (int i = 0; i < NF4_BLOCK; ++i) {
            float v = fabsf(bf16_to_f32(w[i]));
            if (v > a) a = v;
        }
        absmax[b] = a;
        int c[NF4_BLOCK];
        for (int i = 0; i < NF4_BLOCK; ++i) {
            if (a == 0.0f) {
                c[i] = 7; /* the exact-zero level */
            } else {
                float x = bf16_to_f32(w[i]) / a; /* fp32, round to nearest */
                c[i] = oracle_nf4_nearest(x, L);
            }
        }
        for (int i = 0; i < NF4_BLOCK / 2; ++i)
            codes[b * (NF4_BLOCK / 2) + i] = (uint8_t)((c[2 * i] << 4) | c[2 * i + 1]);
    }
}

/* NF4 encode: oracle_q4_encode with the NF4 table. */
void oracle_nf4_encode(const uint16_t *W, int64_t n, uint8_t *codes, float *absmax) {
    float L[16];
    oracle_nf4_table(L);
    oracle_q4_encode(W, n, L, codes, absmax);
}

/* ------------------------------------------------------------------------ */
/* Double quantization of the absmax [QL-note; QL-70B "Double Quantization"] */
/* ------------------------------------------------------------------------ */

/* Pairwise (balanced binary tree) sum in double: the leaves, in order, padded
 * with zeros to a power of two; each level adds neighbours (2i, 2i+1). */
double oracle_pairwise_sum(const float *v, int64_t n) {
    if (n <= 0) return 0.0;
    int64_t p = 1;
    while (p < n) p <<= 1;
    double *t = (double *)calloc((size_t)p, sizeof(double));
    for (int64_t i = 0; i < n; ++i) t[i] = (double)v[i];
    while (p > 1) {
        for (int64_t i = 0; i < p / 2; ++i) t[i] = t[2 * i] + t[2 * i + 1];
        p /= 2;
    }
    double s = t[0];
    free(t);
    return s;
}

/* Second-level quantization of the nb block absmax values:
 *   mean  = fp32( S / nb ),  S the pairwise double sum above;
 *   per group g of 256 blocks (the last may be partial):
 *     c_b = fp32(a_b - mean)
 *     s2_g = fp32( max_b |c_b| / 127 )
 *     q_b  = 0 if s2_g == 0, else clamp(rint(fp32(c_b / s2_g)), -127, 127)
 *   with rint rounding half to even. */
void oracle_dq_encode(const float *absmax, int64_t nb, int8_t *q, float *scale, float *mean_out) {
    double S = oracle_pairwise_sum(absmax, nb);
    float mean = (float)(S / (double)nb);
    *mean_out = mean;
    int64_t ng = (nb + DQ_GROUP - 1) / DQ_GROUP;
    for (int64_t g = 0; g < ng; ++g) {
        int64_t b0 = g * DQ_GROUP, b1 = b0 + DQ_GROUP;
        if (b1 > nb) b1 = nb;
        float m = 0.0f;
        for (int64_t b = b0; b < b1; ++b) {
            float c = absmax[b] - mean;
            if (fabsf(c) > m) m = fabsf(c);
        }
        float s2 = m / 127.0f;
        scale[g] = s2;
        for (int64_t b = b0; b < b1; ++b) {
            float c = absmax[b] - mean;
            if (s2 == 0.0f) {
                q[b] = 0;
            } else {
                float r = rintf(c / s2);
                if (r > 127.0f) r = 127.0f;
                if (r < -127.0f) r = -127.0f;
                q[b] = (int8_t)r;
            }
        }
    }
}

/* Whole quantizer: encode, then double-quantize the absmax. absmax_exact may
 * be NULL; when given it receives the first-level absmax (n/64 floats). */
void oracle_nf4_quantize(const uint16_t *W, int64_t rows, int64_t cols, uint8_t *codes,
                         int8_t *q, float *scale, float *mean, float *absmax_exact) {
    int64_t n = rows * cols, nb = n / NF4_BLOCK;
    float *a = absmax_exact ? absmax_exact : (float *)malloc((size_t)nb * sizeof(float));
    oracle_nf4_encode(W, n, codes, a);
    oracle_dq_encode(a, nb, q, scale, mean);
    if (!absmax_exact) free(a);
}

/* ------------------------------------------------------------------------ */
/* Decode [QL-70B "Double Quantization": dequantize on the fly to the        */
/* compute type; QL-host: the compute type is bf16].                         */
/* ------------------------------------------------------------------------ */

/* Reconstructed absmax of block b: fp32(q) * s2 rounded, then + mean rounded
 * (two separate fp32 operations, never fused). */
float oracle_dq_decode(int8_t qb, float s2, float mean) {
    float t = (float)qb * s2;
    return t + mean;
}

/* W'[i] = bf16_rne( fp32( L[code_i] * a'_b ) ) for all n elements, with
 * the table L and the double-quantized absmax a'_b. */
void oracle_q4_dequantize_dq(const uint8_t *codes, const int8_t *q, const float *scale, float mean,
                             int64_t rows, int64_t cols, const float L[16], uint16_t *out) {
    int64_t n = rows * cols, nb = n / NF4_BLOCK;
#pragma omp parallel for schedule(static)
    for (int64_t b = 0; b < nb; ++b) {
        float a = oracle_dq_decode(q[b], scale[b / DQ_GROUP], mean);
        for (int i = 0; i < NF4_BLOCK; ++i) {
            uint8_t byte = codes[b * (NF4_BLOCK / 2) + i / 2];
            int c = (i % 2 == 0) ? (byte >> 4) : (byte & 15);
            float v = L[c] * a;
            out[b * NF4_BLOCK + i] = f32_to_bf16_rne(v);
        }
    }
}

/* The same with the absmax kept as fp32 per block (no double quantization;
 * the 4.5 bits per weight of xingyuzhitong.com, section "QLoRA: quantize the
 * frozen base to 4 bits"): a_b is used as stored. */
void oracle_q4_dequantize_f32(const uint8_t *codes, const float *absmax, int64_t rows, int64_t cols,
                              const float L[16], uint16_t *out) {
    int64_t n = rows * cols, nb = n / NF4_BLOCK;
#pragma omp parallel for schedule(static)
    for (int64_t b = 0; b < nb; ++b) {
        float a = absmax[b];
        for (int i = 0; i < NF4_BLOCK; ++i) {
            uint8_t byte = codes[b * (NF4_BLOCK / 2) + i / 2];
            int c = (i % 2 == 0) ? (byte >> 4) : (byte & 15);
            float v = L[c] * a;
            out[b * NF4_BLOCK + i] = f32_to_bf16_rne(v);
        }
    }
}

/* NF4 dequantize: oracle_q4_dequantize_dq with the NF4 table. */
void oracle_nf4_dequantize(const uint8_t *codes, const int8_t *q, const float *scale, float mean,
                           int64_t rows, int64_t cols, uint16_t *out) {
    float L[16];
    oracle_nf4_table(L);
    oracle_q4_dequantize_dq(codes, q, scale, mean, rows, cols, L, out);
}

/* ------------------------------------------------------------------------ */
/* Linear layer with LoRA, forward and backward, in fp64 on the dequantized  */
/* bf16 weights [QL-note: gradients flow through the frozen 4-bit weights    */
/* into the adapters; QL-mem "LoRA": A is r x d_in, B is d_out x r].         */
/* s is the LoRA scale (alpha / r); adapter dropout is 0 and there is no     */
/* bias [QL-host adapter setup].                                             */
/* ------------------------------------------------------------------------ */

/* U[m, j] = sum_k X[m,k] A[j,k]   for all m (U: M x r, double). */
void oracle_lora_down(const uint16_t *X, int64_t M, int64_t K, const uint16_t *A, int r, double *U) {
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m)
        for (int j = 0; j < r; ++j) {
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k)
                acc += (double)bf16_to_f32(X[m * K + k]) * (double)bf16_to_f32(A[(int64_t)j * K + k]);
            U[m * r + j] = acc;
        }
}

/* V[m, j] = sum_n dY[m,n] B[n,j]   for all m (V: M x r, double). */
void oracle_lora_up_t(const uint16_t *dY, int64_t M, int64_t N, const uint16_t *B, int r, double *V) {
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m)
        for (int j = 0; j < r; ++j) {
            double acc = 0.0;
            for (int64_t n = 0; n < N; ++n)
                acc += (double)bf16_to_f32(dY[m * N + n]) * (double)bf16_to_f32(B[n * r + j]);
            V[m * r + j] = acc;
        }
}

/* Forward: Y[m, n] = sum_k X[m,k] W'[n,k] + s * sum_j U[m,j] B[n,j].
 * rows: the nr row indices m to compute (NULL: all M rows, nr = M);
 * Y is nr x N in the order of rows. U is the full M x r down-projection. */
void oracle_linear_fwd(const uint16_t *X, int64_t M, const uint16_t *Wdq, int64_t N, int64_t K,
                       const uint16_t *A, const uint16_t *B, int r, float scale,
                       const int64_t *rows, int64_t nr, double *Y, double *U) {
    oracle_lora_down(X, M, K, A, r, U);
    if (!rows) nr = M;
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < nr; ++i) {
        int64_t m = rows ? rows[i] : i;
        for (int64_t n = 0; n < N; ++n) {
            double base = 0.0;
            for (int64_t k = 0; k < K; ++k)
                base += (double)bf16_to_f32(X[m * K + k]) * (double)bf16_to_f32(Wdq[n * K + k]);
            double lora = 0.0;
            for (int j = 0; j < r; ++j) lora += U[m * r + j] * (double)bf16_to_f32(B[n * r + j]);
            Y[i * N + n] = base + (double)scale * lora;
        }
    }
}

/* Backward, with V = dY B and U = X A^T recomputed in fp64:
 *   dX[m, k] = sum_n dY[m,n] W'[n,k] + s * sum_j V[m,j] A[j,k]   (rows m listed)
 *   dB[n, j] = s * sum_m dY[m,n] U[m,j]                          (rows n listed)
 *   dA[j, k] = s * sum_m V[m,j] X[m,k]                           (columns k listed)
 * No gradient for the frozen W. A NULL list means every index (and its count
 * is then M, N or K); outputs are packed in list order: dX is nr x K, dB is
 * nn x r, dA is r x nk.
 * Every sum runs over its contraction index in increasing order (n for dX, m
 * for dB and dA). The loops keep a row of running sums per output row (or a
 * chunk of outputs) so that W', dY and X are read along their rows; this does
 * not change the order in which any single sum is formed. */
#define ORACLE_CHUNK 256
void oracle_linear_bwd(const uint16_t *dY, const uint16_t *X, int64_t M, const uint16_t *Wdq,
                       int64_t N, int64_t K, const uint16_t *A, const uint16_t *B, int r,
                       float scale, const int64_t *rows, int64_t nr, const int64_t *ncols,
                       int64_t nn, const int64_t *kcols, int64_t nk, double *dX, double *dA,
                       double *dB) {
    double *U = (double *)malloc((size_t)(M * r) * sizeof(double));
    double *V = (double *)malloc((size_t)(M * r) * sizeof(double));
    oracle_lora_down(X, M, K, A, r, U);
    oracle_lora_up_t(dY, M, N, B, r, V);
    if (!rows) nr = M;
    if (!ncols) nn = N;
    if (!kcols) nk = K;
    /* dX: for row m, base[k] = sum over n = 0..N-1 of dY[m,n] W'[n,k] */
#pragma omp parallel
    {
        double *base = (double *)malloc((size_t)K * sizeof(double));
#pragma omp for schedule(static)
        for (int64_t i = 0; i < nr; ++i) {
            int64_t m = rows ? rows[i] : i;
            for (int64_t k = 0; k < K; ++k) base[k] = 0.0;
            for (int64_t n = 0; n < N; ++n) {
                double g = (double)bf16_to_f32(dY[m * N + n]);
                const uint16_t *w = Wdq + n * K;
                for (int64_t k = 0; k < K; ++k) base[k] += g * (double)bf16_to_f32(w[k]);
            }
            for (int64_t k = 0; k < K; ++k) {
                double lora = 0.0;
                for (int j = 0; j < r; ++j) lora += V[m * r + j] * (double)bf16_to_f32(A[(int64_t)j * K + k]);
                dX[i * K + k] = base[k] + (double)scale * lora;
            }
        }
        free(base);
    }
    /* dB[n, j] = s * sum over m = 0..M-1 of dY[m,n] U[m,j], ORACLE_CHUNK listed n at a time */
    int64_t nchunks = (nn + ORACLE_CHUNK - 1) / ORACLE_CHUNK;
#pragma omp parallel
    {
        double *acc = (double *)malloc((size_t)ORACLE_CHUNK * (size_t)r * sizeof(double));
#pragma omp for schedule(static)
        for (int64_t c = 0; c < nchunks; ++c) {
            int64_t i0 = c * ORACLE_CHUNK, i1 = i0 + ORACLE_CHUNK < nn ? i0 + ORACLE_CHUNK : nn;
            for (int64_t t = 0; t < (i1 - i0) * r; ++t) acc[t] = 0.0;
            for (int64_t m = 0; m < M; ++m)
                for (int64_t i = i0; i < i1; ++i) {
                    int64_t n = ncols ? ncols[i] : i;
                    double g = (double)bf16_to_f32(dY[m * N + n]);
                    for (int j = 0; j < r; ++j) acc[(i - i0) * r + j] += g * U[m * r + j];
                }
            for (int64_t i = i0; i < i1; ++i)
                for (int j = 0; j < r; ++j) dB[i * r + j] = (double)scale * acc[(i - i0) * r + j];
        }
        free(acc);
    }
    /* dA[j, k] = s * sum over m = 0..M-1 of V[m,j] X[m,k], ORACLE_CHUNK listed k at a time */
    nchunks = (nk + ORACLE_CHUNK - 1) / ORACLE_CHUNK;
#pragma omp parallel
    {
        double *acc = (double *)malloc((size_t)ORACLE_CHUNK * (size_t)r * sizeof(double));
#pragma omp for schedule(static)
        for (int64_t c = 0; c < nchunks; ++c) {
            int64_t i0 = c * ORACLE_CHUNK, i1 = i0 + ORACLE_CHUNK < nk ? i0 + ORACLE_CHUNK : nk;
            for (int64_t t = 0; t < (i1 - i0) * r; ++t) acc[t] = 0.0;
            for (int64_t m = 0; m < M; ++m)
                for (int64_t i = i0; i < i1; ++i) {
                    int64_t k = kcols ? kcols[i] : i;
                    double x = (double)bf16_to_f32(X[m * K + k]);
                    for (int j = 0; j < r; ++j) acc[(i - i0) * r + j] += V[m * r + j] * x;
                }
            for (int64_t i = i0; i < i1; ++i)
                for (int j = 0; j < r; ++j) dA[(int64_t)j * nk + i] = (double)scale * acc[(i - i0) * r + j];
        }
        free(acc);
    }
    free(U);
    free(V);
}

/* ------------------------------------------------------------------------ */
/* Merge the adapter into the base and quantize again [QL-mem "Choosing a   */
/* method": for deployment the adapters are merged into the base weights].  */
/* ------------------------------------------------------------------------ */

/* merged[n,k] = bf16_rne( w'[n,k] + s * t[n,k] ),  t[n,k] = sum_j B[n,j] A[j,k]
 * with every operation a separately rounded fp32 operation: t starts at 0
 * and adds the products for j = 0 .. r-1 in that order (a product of two
 * bf16 numbers is exact in fp32), then s * t, then the add to w'. The
 * merged weight is then quantized with oracle_nf4_quantize like any other
 * bf16 weight. */
void oracle_lora_merge(const uint16_t *Wdq, int64_t N, int64_t K, const uint16_t *A, const uint16_t *B, int r,
                       float s, uint16_t *merged) {
#pragma omp parallel for schedule(static)
    for (int64_t n = 0; n < N; ++n)
        for (int64_t k = 0; k < K; ++k) {
            float t = 0.0f;
            for (int j = 0; j < r; ++j) {
                float prod = bf16_to_f32(B[n * r + j]) * bf16_to_f32(A[(int64_t)j * K + k]);
                t = t + prod;
            }
            float st = s * t;
            float m = bf16_to_f32(Wdq[n * K + k]) + st;
            merged[n * K + k] = f32_to_bf16_rne(m);
        }
}

/* ------------------------------------------------------------------------ */
/* AdamW step for the adapters [QL-note: paged optimizers; QL-70B "Paged    */
/* Optimizers": optimizer state that can live in host memory; the addaly    */
/* lesson's paged_adamw]. The update rule is not on the pages; the reading  */
/* is AdamW with decoupled weight decay (Loshchilov & Hutter), in the order */
/* torch.optim.AdamW applies it, in fp64:                                   */
/*   p = p * (1 - lr * wd)                                                  */
/*   m = b1 m + (1 - b1) g ;  v = b2 v + (1 - b2) g^2                       */
/*   p = p - (lr / (1 - b1^t)) * m / (sqrt(v) / sqrt(1 - b2^t) + eps)       */
/* ------------------------------------------------------------------------ */
void oracle_adamw_step(double *p, const double *g, double *m, double *v, int64_t n, double lr, double b1,
                       double b2, double eps, double wd, int64_t t) {
    double bias1 = 1.0 - pow(b1, (double)t), bias2 = 1.0 - pow(b2, (double)t);
    double step_size = lr / bias1, bias2_sqrt = sqrt(bias2);
    for (int64_t i = 0; i < n; ++i) {
        p[i] = p[i] * (1.0 - lr * wd);
        m[i] = b1 * m[i] + (1.0 - b1) * g[i];
        v[i] = b2 * v[i] + (1.0 - b2) * g[i] * g[i];
        double denom = sqrt(v[i]) / bias2_sqrt + eps;
        p[i] = p[i] - step_size * m[i] / denom;
    }
}
