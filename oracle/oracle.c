/*
 * oracle.c -- TEST INFRASTRUCTURE, not part of the product.
 *
 * A plain, slow, obviously correct CPU statement of what the tensor-core
 * path computes:  C = epilogue(A . B)  with A (M x K) and B (K x N) row-major
 * 16-bit floating-point operands, a sum taken in fp64, an optional fp32
 * per-column bias and ReLU, and one final round-to-nearest-even into the
 * output's storage type.
 *
 * Only the test suite, the smoke check and the benchmark's CPU-baseline leg
 * may load this library.  It shares no code, header or constant with the
 * CUDA path: it has its own decoders and encoders, written from the IEEE 754
 * binary16/binary32 and bfloat16 bit layouts, and its own type codes.
 *
 * What each piece follows:
 *   - Operand types: gizml:tile, "F16", "BF16" and "FP8" ("FP8 E4M3
 *     floats") are the storage types of the matrix-core operands.
 *   - The product itself: gizml:tile, "Tile.dot" -- the matrix product
 *     [M,K][K,N] -> [M,N] kept in F32; here it is kept in fp64 so that the
 *     GPU's F32 accumulation is graded against the (almost) exact sum.
 *   - Edges: gizml:tile, "In.at" -- elements past a tensor's edge read 0, and
 *     "Out.put" -- elements past the edge are not written.  The loops below
 *     run over the logical M x N x K box only, so an out-of-range element is
 *     never read (the same as reading 0) and nothing outside M x N (including
 *     the ldc padding) is written.
 *   - Epilogue: gizml:tile, the fused example under "Tile.run" (put of
 *     acc.relu()), "Tile.relu" = max(x, 0), "Tile.add" (broadcast add of a
 *     per-column bias row).  The bias is added before the ReLU, in the sum's
 *     precision, as the per-column seed of the accumulator in the Swin-layer
 *     epilogue notes (d4r, rrswin_enc2_epilogues.md, bias as the MMA's C).
 *   - Output rounding: gizml:tile, "Tile.to" -- rounded to the storage type
 *     "as a store and a load of it give them": IEEE round-to-nearest-even,
 *     overflow to +-infinity, NaN stays NaN.
 *   - Empty K: gizml:tile, "Program.fold" -- a fold with no trips returns its
 *     init, so K = 0 gives C = epilogue(0 [+ bias]).
 *   - Residual: the Swin-layer MLP band (d4r, rrswin_enc2_epilogues.md,
 *     "Shape of the whole MLP band") ends with a back-projection whose MMA
 *     takes the previous accumulator as its C input, D = A . B + C.  With a
 *     residual R (M x N, in a storage type) the sum becomes
 *     s_ij = R_ij + sum_k a_ik b_kj, before the bias and the ReLU: the
 *     fold starts from R instead of zeros (gizml:tile, "Program.fold",
 *     init), so K = 0 gives C = epilogue(R [+ bias]).
 *   - Integer-coded B (orc_gemm_qb): Tolk.Stage, "Decoded panels on the
 *     host" -- an operand decoded from integer codes, as a quantised
 *     matrix's is; read here as int8 codes times one fp32 scale per column.
 *   - Staging never changes values (Tolk.Stage, module overview): the oracle
 *     has no staging at all; the GPU path's results at every stage count are
 *     graded against this one definition.
 *
 * Loop order is i-k-j with an fp64 accumulator row per output row (the plain
 * definition: s_ij = sum over ascending k of a_ik * b_kj).  Products of two
 * 16-bit floats are exact in fp64.  Rows are split over POSIX threads; each
 * row is computed by exactly one thread, so the result does not depend on
 * the thread count.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* The oracle's own storage-type codes (ASCII letters; unrelated to the
 * product's enumeration). */
#define ORC_FP32 'S' /* IEEE 754 binary32 */
#define ORC_FP16 'H' /* IEEE 754 binary16 */
#define ORC_BF16 'B' /* bfloat16: binary32's sign and exponent, 7 fraction bits */
#define ORC_E4M3 'E' /* OCP FP8 E4M3: 4 exponent bits (bias 7), 3 fraction bits, no
                        infinities, NaN only at S.1111.111, largest finite 448 */

#define ORC_EPI_NONE 'n'
#define ORC_EPI_RELU 'r'
#define ORC_EPI_BIAS_RELU 'b'

/* ---------------------------------------------------------------- formats */

/* Field widths of a storage type: exponent bits, stored fraction bits. */
static int fmt_fields(int dtype, int *ebits, int *fbits) {
    switch (dtype) {
    case ORC_FP32: *ebits = 8; *fbits = 23; return 0;
    case ORC_FP16: *ebits = 5; *fbits = 10; return 0;
    case ORC_BF16: *ebits = 8; *fbits = 7; return 0;
    case ORC_E4M3: *ebits = 4; *fbits = 3; return 0;
    default: return -1;
    }
}

/* Decode the bit pattern of a binary floating-point number with the given
 * field widths: value = (-1)^s * 2^(e - bias) * (1 + f / 2^fbits) for a
 * normal number, (-1)^s * 2^(1 - bias) * (f / 2^fbits) for a subnormal one,
 * infinity or NaN for the all-ones exponent. */
double orc_decode(int dtype, uint32_t bits) {
    int ebits, fbits;
    if (fmt_fields(dtype, &ebits, &fbits) != 0) return NAN;
    const uint32_t emask = (1u << ebits) - 1u;
    const uint32_t fmask = (1u << fbits) - 1u;
    const int bias = (int)(emask >> 1);
    const uint32_t s = (bits >> (ebits + fbits)) & 1u;
    const uint32_t e = (bits >> fbits) & emask;
    const uint32_t f = bits & fmask;
    double mag;
    if (dtype == ORC_E4M3 && e == emask) {
        /* E4M3 keeps the all-ones exponent for finite values; only f = 7 is NaN */
        mag = (f == fmask) ? NAN : ldexp((double)((1u << fbits) | f), (int)e - bias - fbits);
    } else if (e == emask) {
        mag = (f == 0) ? INFINITY : NAN;
    } else if (e == 0) {
        mag = ldexp((double)f, 1 - bias - fbits);
    } else {
        mag = ldexp((double)((1u << fbits) | f), (int)e - bias - fbits);
    }
    return s ? -mag : mag;
}

/* Encode x into the storage type, rounding to nearest with ties to even.
 * Values whose magnitude rounds above the largest finite number become
 * infinity; NaN becomes the quiet NaN with x's sign. */
uint32_t orc_encode(int dtype, double x) {
    int ebits, fbits;
    if (dtype == ORC_E4M3) return 0; /* E4M3 is an operand type only: never encoded */
    if (fmt_fields(dtype, &ebits, &fbits) != 0) return 0;
    const uint32_t emask = (1u << ebits) - 1u;
    const int bias = (int)(emask >> 1);
    const int emin = 1 - bias;       /* smallest normal exponent */
    const int emax = bias;           /* largest finite exponent */
    const uint32_t sbit = (signbit(x) ? 1u : 0u) << (ebits + fbits);
    const uint32_t inf = emask << fbits;
    if (isnan(x)) return sbit | inf | (1u << (fbits - 1));
    double a = fabs(x);
    if (isinf(a)) return sbit | inf;
    if (a == 0.0) return sbit;

    int ex;
    (void)frexp(a, &ex);      /* a = m * 2^ex, m in [0.5, 1) */
    int e = ex - 1;           /* a in [2^e, 2^(e+1)) */
    if (e < emin) e = emin;   /* subnormal range: fixed quantum */
    /* quantum of the target at this exponent; a / q is exact (power of 2) */
    const double m = ldexp(a, fbits - e);
    double r = floor(m);
    const double rem = m - r;
    if (rem > 0.5 || (rem == 0.5 && fmod(r, 2.0) != 0.0)) r += 1.0;
    const double one = ldexp(1.0, fbits); /* implicit leading bit */
    if (r >= 2.0 * one) {  /* rounding carried into the next binade */
        r = one;
        e += 1;
    }
    if (e > emax) return sbit | inf;
    if (r < one) {         /* subnormal (only possible when e == emin) */
        return sbit | (uint32_t)r;
    }
    return sbit | ((uint32_t)(e + bias) << fbits) | ((uint32_t)(r - one));
}

static uint32_t load_bits(int dtype, const void *p, int64_t idx) {
    if (dtype == ORC_E4M3) return ((const unsigned char *)p)[idx];
    if (dtype == ORC_FP32) {
        uint32_t v;
        memcpy(&v, (const unsigned char *)p + 4 * idx, 4);
        return v;
    }
    uint16_t v;
    memcpy(&v, (const unsigned char *)p + 2 * idx, 2);
    return v;
}

static void store_bits(int dtype, void *p, int64_t idx, uint32_t v) {
    if (dtype == ORC_FP32) {
        memcpy((unsigned char *)p + 4 * idx, &v, 4);
    } else {
        uint16_t h = (uint16_t)v;
        memcpy((unsigned char *)p + 2 * idx, &h, 2);
    }
}

/* The epilogue on one fp64 sum: + bias[j] (bias_relu), then ReLU.
 * ReLU is max(s, 0) with -0 -> +0 and NaN passed through. */
static double epilogue(int epi, double s, const float *bias, int64_t j) {
    if (epi == ORC_EPI_BIAS_RELU) s += orc_decode(ORC_FP32, load_bits(ORC_FP32, bias, j));
    if (epi == ORC_EPI_RELU || epi == ORC_EPI_BIAS_RELU) s = (s <= 0.0) ? 0.0 : s;
    return s;
}

/* ------------------------------------------------------------- full GEMM */

typedef struct {
    int64_t M, N, K;
    const void *R;   /* M x N residual (r_dtype, pitch ldr), or NULL */
    int r_dtype;
    int64_t ldr;
    const double *Ad; /* M x K decoded A, row-major, dense */
    const double *Bd; /* K x N decoded B, row-major, dense */
    int epi;
    const float *bias;
    int out_dtype;
    void *C;
    int64_t ldc;
    double *C_exact; /* M x N, may be NULL */
    double *S;       /* M x N sum of |a_ik * b_kj|, may be NULL */
    int64_t row_begin, row_end;
} gemm_job;

static void *gemm_rows(void *arg) {
    gemm_job *jb = (gemm_job *)arg;
    const int64_t N = jb->N, K = jb->K;
    double *acc = (double *)calloc((size_t)(N > 0 ? N : 1), sizeof(double));
    double *sab = (double *)calloc((size_t)(N > 0 ? N : 1), sizeof(double));
    if (!acc || !sab) {
        free(acc);
        free(sab);
        return (void *)1;
    }
    for (int64_t i = jb->row_begin; i < jb->row_end; ++i) {
        for (int64_t j = 0; j < N; ++j) {
            acc[j] = 0.0;
            sab[j] = 0.0;
        }
        for (int64_t k = 0; k < K; ++k) {
            const double a = jb->Ad[i * K + k];
            const double *brow = jb->Bd + k * N;
            for (int64_t j = 0; j < N; ++j) {
                const double p = a * brow[j];
                acc[j] += p;
                sab[j] += fabs(p);
            }
        }
        for (int64_t j = 0; j < N; ++j) {
            double s = acc[j];
            if (jb->R) s += orc_decode(jb->r_dtype, load_bits(jb->r_dtype, jb->R, i * jb->ldr + j));
            const double v = epilogue(jb->epi, s, jb->bias, j);
            if (jb->C_exact) jb->C_exact[i * N + j] = v;
            if (jb->S) jb->S[i * N + j] = sab[j];
            if (jb->C) store_bits(jb->out_dtype, jb->C, i * jb->ldc + j, orc_encode(jb->out_dtype, v));
        }
    }
    free(acc);
    free(sab);
    return NULL;
}

static int valid_in(int d) { return d == ORC_FP16 || d == ORC_BF16 || d == ORC_E4M3; }
static int valid_out(int d) { return d == ORC_FP32 || d == ORC_FP16 || d == ORC_BF16; }
static int valid_epi(int e) { return e == ORC_EPI_NONE || e == ORC_EPI_RELU || e == ORC_EPI_BIAS_RELU; }

/* Decode the logical K-column (or N-column) box of a strided operand into a
 * dense fp64 matrix.  Elements beyond the logical box (ld padding) are never
 * read. */
static double *decode_matrix(int dtype, const void *X, int64_t rows, int64_t cols, int64_t ld) {
    size_t n = (size_t)(rows * cols);
    double *out = (double *)malloc((n ? n : 1) * sizeof(double));
    if (!out) return NULL;
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t c = 0; c < cols; ++c) out[r * cols + c] = orc_decode(dtype, load_bits(dtype, X, r * ld + c));
    return out;
}

static int run_decoded(int64_t M, int64_t N, int64_t K, const double *Ad, const double *Bd, const void *R,
                       int r_dtype, int64_t ldr, int epi, const float *bias, int out_dtype, void *C, int64_t ldc,
                       double *C_exact, double *S, int threads);

/* C[i*ldc + j] = encode(out_dtype, epilogue(R_ij + sum_k a_ik b_kj)) for
 * i < M, j < N, with R_ij = 0 when R is NULL.  C_exact and S, when given,
 * receive the fp64 value before rounding and the sum of |a_ik b_kj| (dense
 * M x N).  Returns 0, or -1 on a bad argument, -2 when memory runs out. */
int orc_gemm_residual(int64_t M, int64_t N, int64_t K, const void *A, int64_t lda, const void *B, int64_t ldb,
                      const void *R, int r_dtype, int64_t ldr, int in_dtype, int epi, const float *bias,
                      int out_dtype, void *C, int64_t ldc, double *C_exact, double *S, int threads) {
    if (M < 0 || N < 0 || K < 0) return -1;
    if (R && (!valid_out(r_dtype) || ldr < N)) return -1;
    if (!valid_in(in_dtype) || !valid_out(out_dtype) || !valid_epi(epi)) return -1;
    if ((epi == ORC_EPI_BIAS_RELU) != (bias != NULL)) return -1;
    if (lda < K || ldb < N || ldc < N) return -1;
    if (M == 0 || N == 0) return 0;
    double *Ad = decode_matrix(in_dtype, A, M, K, lda);
    double *Bd = decode_matrix(in_dtype, B, K, N, ldb);
    if (!Ad || !Bd) {
        free(Ad);
        free(Bd);
        return -2;
    }
    const int rc = run_decoded(M, N, K, Ad, Bd, R, r_dtype, ldr, epi, bias, out_dtype, C, ldc, C_exact, S, threads);
    free(Ad);
    free(Bd);
    return rc;
}

/* The row loop of the GEMM on decoded (fp64, dense) operands, split over
 * POSIX threads by whole rows. */
static int run_decoded(int64_t M, int64_t N, int64_t K, const double *Ad, const double *Bd, const void *R,
                       int r_dtype, int64_t ldr, int epi, const float *bias, int out_dtype, void *C, int64_t ldc,
                       double *C_exact, double *S, int threads) {
    if (threads < 1) threads = 1;
    if (threads > M) threads = (int)M;
    gemm_job *jobs = (gemm_job *)calloc((size_t)threads, sizeof(gemm_job));
    pthread_t *tids = (pthread_t *)calloc((size_t)threads, sizeof(pthread_t));
    int rc = 0;
    if (!jobs || !tids) rc = -2;
    for (int t = 0; rc == 0 && t < threads; ++t) {
        gemm_job *jb = &jobs[t];
        jb->M = M; jb->N = N; jb->K = K;
        jb->R = R; jb->r_dtype = r_dtype; jb->ldr = ldr;
        jb->Ad = Ad; jb->Bd = Bd;
        jb->epi = epi; jb->bias = bias;
        jb->out_dtype = out_dtype; jb->C = C; jb->ldc = ldc;
        jb->C_exact = C_exact; jb->S = S;
        jb->row_begin = M * t / threads;
        jb->row_end = M * (t + 1) / threads;
    }
    int started = 0;
    for (int t = 0; rc == 0 && t < threads; ++t) {
        if (pthread_create(&tids[t], NULL, gemm_rows, &jobs[t]) != 0) {
            /* run the rest on this thread */
            for (int u = t; u < threads; ++u)
                if (gemm_rows(&jobs[u]) != NULL) rc = -2;
            break;
        }
        ++started;
    }
    for (int t = 0; t < started; ++t) {
        void *ret = NULL;
        pthread_join(tids[t], &ret);
        if (ret != NULL) rc = -2;
    }
    free(jobs);
    free(tids);
    return rc;
}

/* ------------------------------------------------ integer-coded B operand
 *
 * Tolk.Stage, "Decoded panels on the host": one operand of the product is
 * decoded from integer codes, as a quantised matrix's is.  The page names no
 * code format; the reading taken here: B is given as signed 8-bit codes q_kj
 * (two's complement, row-major K x N, pitch ldq) and one fp32 scale s_j per
 * column, and its value is b_kj = s_j * q_kj.  That product is exact in fp64
 * (24 + 8 significant bits), so the decoded B below is the value itself and
 * the rest is orc_gemm's definition: C = epilogue(sum_k a_ik b_kj), S_ij =
 * sum_k |a_ik b_kj|.  Where the decode happens (once per panel, as the page
 * stages it, or at every use) cannot change the value; the oracle has no
 * panel at all. */
int orc_gemm_qb(int64_t M, int64_t N, int64_t K, const void *A, int64_t lda, int in_dtype, const int8_t *Q,
                int64_t ldq, const float *scale, int epi, const float *bias, int out_dtype, void *C, int64_t ldc,
                double *C_exact, double *S, int threads) {
    if (M < 0 || N < 0 || K < 0) return -1;
    if (!valid_in(in_dtype) || !valid_out(out_dtype) || !valid_epi(epi)) return -1;
    if ((epi == ORC_EPI_BIAS_RELU) != (bias != NULL)) return -1;
    if (lda < K || ldq < N || ldc < N || (N > 0 && !scale)) return -1;
    if (M == 0 || N == 0) return 0;
    double *Ad = decode_matrix(in_dtype, A, M, K, lda);
    double *Bd = (double *)malloc((size_t)(K * N > 0 ? K * N : 1) * sizeof(double));
    if (!Ad || !Bd) {
        free(Ad);
        free(Bd);
        return -2;
    }
    for (int64_t k = 0; k < K; ++k)
        for (int64_t j = 0; j < N; ++j) {
            const double s_j = orc_decode(ORC_FP32, load_bits(ORC_FP32, scale, j));
            Bd[k * N + j] = s_j * (double)Q[k * ldq + j];
        }
    const int rc = run_decoded(M, N, K, Ad, Bd, NULL, ORC_FP32, 0, epi, bias, out_dtype, C, ldc, C_exact, S, threads);
    free(Ad);
    free(Bd);
    return rc;
}

int orc_gemm(int64_t M, int64_t N, int64_t K, const void *A, int64_t lda, const void *B, int64_t ldb,
             int in_dtype, int epi, const float *bias, int out_dtype, void *C, int64_t ldc, double *C_exact,
             double *S, int threads) {
    return orc_gemm_residual(M, N, K, A, lda, B, ldb, NULL, ORC_FP32, 0, in_dtype, epi, bias, out_dtype, C, ldc,
                             C_exact, S, threads);
}

/* --------------------------------------------------- selected (i, j) only */

typedef struct {
    int64_t K;
    const void *R; int r_dtype; int64_t ldr;
    const void *A; int64_t lda;
    const void *B; int64_t ldb;
    int in_dtype, epi, out_dtype;
    const float *bias;
    const int64_t *rows, *cols;
    uint32_t *out_bits;
    double *out_exact, *out_S;
    int64_t begin, end;
} at_job;

static void *gemm_at_range(void *arg) {
    at_job *jb = (at_job *)arg;
    for (int64_t t = jb->begin; t < jb->end; ++t) {
        const int64_t i = jb->rows[t], j = jb->cols[t];
        double acc = 0.0, sab = 0.0;
        for (int64_t k = 0; k < jb->K; ++k) {
            const double p = orc_decode(jb->in_dtype, load_bits(jb->in_dtype, jb->A, i * jb->lda + k)) *
                             orc_decode(jb->in_dtype, load_bits(jb->in_dtype, jb->B, k * jb->ldb + j));
            acc += p;
            sab += fabs(p);
        }
        if (jb->R) acc += orc_decode(jb->r_dtype, load_bits(jb->r_dtype, jb->R, i * jb->ldr + j));
        const double v = epilogue(jb->epi, acc, jb->bias, j);
        if (jb->out_exact) jb->out_exact[t] = v;
        if (jb->out_S) jb->out_S[t] = sab;
        if (jb->out_bits) jb->out_bits[t] = orc_encode(jb->out_dtype, v);
    }
    return NULL;
}

/* The same definition at n chosen output positions (rows[t], cols[t]): the
 * dot product of row i of A with column j of B over ascending k.  Used where
 * the full product is too large to recompute on the host. */
int orc_gemm_residual_at(int64_t M, int64_t N, int64_t K, const void *A, int64_t lda, const void *B, int64_t ldb,
                         const void *R, int r_dtype, int64_t ldr, int in_dtype, int epi, const float *bias,
                         int out_dtype, int64_t n, const int64_t *rows, const int64_t *cols, uint32_t *out_bits,
                         double *out_exact, double *out_S, int threads) {
    if (M < 0 || N < 0 || K < 0 || n < 0) return -1;
    if (R && (!valid_out(r_dtype) || ldr < N)) return -1;
    if (!valid_in(in_dtype) || !valid_out(out_dtype) || !valid_epi(epi)) return -1;
    if ((epi == ORC_EPI_BIAS_RELU) != (bias != NULL)) return -1;
    if (lda < K || ldb < N) return -1;
    for (int64_t t = 0; t < n; ++t)
        if (rows[t] < 0 || rows[t] >= M || cols[t] < 0 || cols[t] >= N) return -1;
    if (n == 0) return 0;
    if (threads < 1) threads = 1;
    if (threads > n) threads = (int)n;
    at_job *jobs = (at_job *)calloc((size_t)threads, sizeof(at_job));
    pthread_t *tids = (pthread_t *)calloc((size_t)threads, sizeof(pthread_t));
    if (!jobs || !tids) {
        free(jobs);
        free(tids);
        return -2;
    }
    for (int t = 0; t < threads; ++t) {
        at_job *jb = &jobs[t];
        jb->K = K; jb->A = A; jb->lda = lda; jb->B = B; jb->ldb = ldb;
        jb->R = R; jb->r_dtype = r_dtype; jb->ldr = ldr;
        jb->in_dtype = in_dtype; jb->epi = epi; jb->out_dtype = out_dtype; jb->bias = bias;
        jb->rows = rows; jb->cols = cols;
        jb->out_bits = out_bits; jb->out_exact = out_exact; jb->out_S = out_S;
        jb->begin = n * t / threads;
        jb->end = n * (t + 1) / threads;
    }
    int started = 0;
    for (int t = 0; t < threads; ++t) {
        if (pthread_create(&tids[t], NULL, gemm_at_range, &jobs[t]) != 0) {
            for (int u = t; u < threads; ++u) gemm_at_range(&jobs[u]);
            break;
        }
        ++started;
    }
    for (int t = 0; t < started; ++t) pthread_join(tids[t], NULL);
    free(jobs);
    free(tids);
    return 0;
}

int orc_gemm_at(int64_t M, int64_t N, int64_t K, const void *A, int64_t lda, const void *B, int64_t ldb,
                int in_dtype, int epi, const float *bias, int out_dtype, int64_t n, const int64_t *rows,
                const int64_t *cols, uint32_t *out_bits, double *out_exact, double *out_S, int threads) {
    return orc_gemm_residual_at(M, N, K, A, lda, B, ldb, NULL, ORC_FP32, 0, in_dtype, epi, bias, out_dtype, n, rows,
                                cols, out_bits, out_exact, out_S, threads);
}

/* Elementwise decode / encode of arrays, for the tests. */
void orc_decode_array(int dtype, const void *bits, int64_t n, double *out) {
    for (int64_t t = 0; t < n; ++t) out[t] = orc_decode(dtype, load_bits(dtype, bits, t));
}

void orc_encode_array(int dtype, const double *x, int64_t n, void *bits) {
    for (int64_t t = 0; t < n; ++t) store_bits(dtype, bits, t, orc_encode(dtype, x[t]));
}
