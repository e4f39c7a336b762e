/*
 * CPU oracle for the packed-int4 integer GEMMs.  TEST INFRASTRUCTURE ONLY:
 * tests, the smoke check and the benchmark's CPU-baseline leg call it; the
 * library never does.  It shares no code with the CUDA path.
 *
 * What it computes (the plain definition, nothing reordered or blocked):
 *
 *   C[m,n] = sum_{k<K} a[m,k] * b[n,k]                         (NT product)
 *
 * with a, b the logical signed integers, accumulated in int64 and narrowed
 * to int32 after checking the no-overflow bound |C| <= K*max|a|*max|b|.
 *   - "[CUDA] Support int4 T.gemm" (tilelang PR #2063),
 *     examples/gemm_int4/example_tilelang_gemm_int4.py, matmul_nt_int4:
 *     A (M,K) int4, B (N,K) int4, C (M,N) int32, gemm with transpose_B.
 *   - "[Example] add w4a8 gemm kernel" (tilelang PR #815), review of
 *     ref_program: A int8 times the unpacked int4 B, taken in integers.
 *   - TileLang tutorial low_precision_gemm.py, matmul_int4 (int4 inputs,
 *     int32 accumulator).
 *
 * Packing (tutorial low_precision_gemm.py, pack_int4): byte j of a packed row
 * holds logical element 2j in its low nibble and element 2j+1 in its high
 * nibble, each masked to 4 bits.
 *
 * Unpacking ("[Example] add w4a8 gemm kernel", reviewer's vectorised
 * torch_convert): the nibble at position pos (0 = low, 1 = high) is
 * (byte >> 4*pos) & 0xF, read as a 4-bit two's-complement number, i.e. minus
 * 16 when it is 8 or more.
 *
 * Every function here is pinned by the CPU tests (closed forms, brute force,
 * numpy int64 matmul, round trips, hand-computed bytes).
 *
 * ORACLE_MUTANT (compile-time, tests only): plants one known mistake so that
 * the pin suite can show it catches it.  Never defined in a normal build.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <pthread.h>

#ifndef ORACLE_MUTANT
#define ORACLE_MUTANT 0
#endif

/* Signed value of nibble `pos` (0 = low = even k, 1 = high = odd k). */
int oracle_nibble(uint8_t byte, int pos)
{
#if ORACLE_MUTANT == 1 /* planted: nibble order swapped */
    pos = 1 - pos;
#endif
    int v = (byte >> (4 * pos)) & 0xF;
#if ORACLE_MUTANT == 2 /* planted: no sign extension */
    return v;
#else
    return v >= 8 ? v - 16 : v;
#endif
}

/* logical [rows, K] int8 -> packed [rows, K/2] bytes.  K must be even. */
void oracle_pack_int4(const int8_t *logical, uint8_t *packed, int64_t rows, int64_t K)
{
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t j = 0; j < K / 2; ++j) {
            int lo = logical[r * K + 2 * j] & 0xF;
            int hi = logical[r * K + 2 * j + 1] & 0xF;
            packed[r * (K / 2) + j] = (uint8_t)(lo | (hi << 4));
        }
    }
}

/* packed [rows, K/2] -> logical [rows, K] int8 in [-8, 7]. */
void oracle_unpack_int4(const uint8_t *packed, int8_t *logical, int64_t rows, int64_t K)
{
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t k = 0; k < K; ++k)
            logical[r * K + k] = (int8_t)oracle_nibble(packed[r * (K / 2) + k / 2], (int)(k % 2));
}

/* One output element, int64 accumulation over the full K. */
static int64_t dot_i64(const int8_t *a_row, const int8_t *b_row, int64_t K)
{
    int64_t s = 0;
#if ORACLE_MUTANT == 4 /* planted: last k dropped */
    K -= 1;
#endif
    for (int64_t k = 0; k < K; ++k) {
#if ORACLE_MUTANT == 5 /* planted: sign of one product flipped (k == 1) */
        if (k == 1) { s -= (int64_t)a_row[k] * (int64_t)b_row[k]; continue; }
#endif
        s += (int64_t)a_row[k] * (int64_t)b_row[k];
    }
    return s;
}

struct job {
    const int8_t *a;  /* [M, K] logical */
    const int8_t *b;  /* [N, K] logical */
    int32_t *c;       /* [M, N] */
    int64_t M, N, K, bound;
    int64_t m_begin, m_end;
    int violated;
};

static void *run_rows(void *arg)
{
    struct job *j = (struct job *)arg;
    for (int64_t m = j->m_begin; m < j->m_end; ++m) {
        for (int64_t n = 0; n < j->N; ++n) {
#if ORACLE_MUTANT == 3 /* planted: operands transposed (b indexed by m) */
            int64_t s = dot_i64(j->a + m * j->K, j->b + (m % j->N) * j->K, j->K);
#else
            int64_t s = dot_i64(j->a + m * j->K, j->b + n * j->K, j->K);
#endif
            if (s > j->bound || s < -j->bound) j->violated = 1;
            j->c[m * j->N + n] = (int32_t)s;
        }
    }
    return NULL;
}

/* C = A . B^T over logical int8 rows, `nthreads` threads over m.
 * `amax`, `bmax` are the largest magnitudes the operands may take (8 for int4,
 * 128 for int8); the bound checked is K*amax*bmax.  Returns 0, or 4 if the
 * bound was exceeded (inputs outside the stated ranges), or -1 on a thread
 * error. */
static int gemm_logical(const int8_t *a, const int8_t *b, int32_t *c, int64_t M, int64_t N,
                        int64_t K, int64_t amax, int64_t bmax, int nthreads)
{
    if (nthreads < 1) nthreads = 1;
    if (nthreads > M) nthreads = (int)(M > 0 ? M : 1);
    struct job *jobs = (struct job *)calloc((size_t)nthreads, sizeof(struct job));
    pthread_t *tids = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !tids) { free(jobs); free(tids); return -1; }
    int rc = 0;
    for (int t = 0; t < nthreads; ++t) {
        jobs[t] = (struct job){a, b, c, M, N, K, K * amax * bmax,
                               M * t / nthreads, M * (t + 1) / nthreads, 0};
        if (pthread_create(&tids[t], NULL, run_rows, &jobs[t]) != 0) {
            run_rows(&jobs[t]);
            tids[t] = 0;
        }
    }
    for (int t = 0; t < nthreads; ++t) {
        if (tids[t]) pthread_join(tids[t], NULL);
        if (jobs[t].violated) rc = 4;
    }
    free(jobs);
    free(tids);
    return rc;
}

/* int4 x int4: Ap [M, K/2], Bp [N, K/2] packed; C [M, N] int32. */
int oracle_i4i4_gemm(const uint8_t *Ap, const uint8_t *Bp, int32_t *C, int64_t M, int64_t N,
                     int64_t K, int nthreads)
{
    int8_t *a = (int8_t *)malloc((size_t)(M * K));
    int8_t *b = (int8_t *)malloc((size_t)(N * K));
    if (!a || !b) { free(a); free(b); return -1; }
    oracle_unpack_int4(Ap, a, M, K);
    oracle_unpack_int4(Bp, b, N, K);
    int rc = gemm_logical(a, b, C, M, N, K, 8, 8, nthreads);
    free(a);
    free(b);
    return rc;
}

/* W4A8: A [M, K] int8 activations, Bp [N, K/2] packed int4 weights. */
int oracle_w4a8_gemm(const int8_t *A, const uint8_t *Bp, int32_t *C, int64_t M, int64_t N,
                     int64_t K, int nthreads)
{
    int8_t *b = (int8_t *)malloc((size_t)(N * K));
    if (!b) return -1;
    oracle_unpack_int4(Bp, b, N, K);
    int rc = gemm_logical(A, b, C, M, N, K, 128, 8, nthreads);
    free(b);
    return rc;
}

/* Single elements, for sampled checks at sizes too large for the full loop.
 * `ms`, `ns` list `count` (m, n) pairs; out[i] receives C[ms[i], ns[i]].
 * Returns 0, 4 if an entry exceeds the no-overflow bound K*amax*bmax (as
 * gemm_logical does), or -1 on an allocation error. */
int oracle_i4i4_entries(const uint8_t *Ap, const uint8_t *Bp, int64_t K, const int64_t *ms,
                        const int64_t *ns, int64_t count, int64_t *out)
{
    int8_t *a = (int8_t *)malloc((size_t)(K > 0 ? K : 1));
    int8_t *b = (int8_t *)malloc((size_t)(K > 0 ? K : 1));
    if (!a || !b) { free(a); free(b); return -1; }
    const int64_t bound = K * 8 * 8;
    int rc = 0;
    for (int64_t i = 0; i < count; ++i) {
        oracle_unpack_int4(Ap + ms[i] * (K / 2), a, 1, K);
        oracle_unpack_int4(Bp + ns[i] * (K / 2), b, 1, K);
        out[i] = dot_i64(a, b, K);
        if (out[i] > bound || out[i] < -bound) rc = 4;
    }
    free(a);
    free(b);
    return rc;
}

int oracle_w4a8_entries(const int8_t *A, const uint8_t *Bp, int64_t K, const int64_t *ms,
                        const int64_t *ns, int64_t count, int64_t *out)
{
    int8_t *b = (int8_t *)malloc((size_t)(K > 0 ? K : 1));
    if (!b) return -1;
    const int64_t bound = K * 128 * 8;
    int rc = 0;
    for (int64_t i = 0; i < count; ++i) {
        oracle_unpack_int4(Bp + ns[i] * (K / 2), b, 1, K);
        out[i] = dot_i64(A + ms[i] * K, b, K);
        if (out[i] > bound || out[i] < -bound) rc = 4;
    }
    free(b);
    return rc;
}

/* ---------------------------------------------------------------- fp8 GEMM
 * TileLang tutorial low_precision_gemm.py, gemm_fp8: A (M,K) and B (N,K) in an
 * fp8 dtype, C = A . B^T accumulated in float32 (accum_dtype).  The oracle
 * takes the plain definition in double: every fp8 value is exact in double and
 * so is every product; the sum of K products is kept in double next to the sum
 * of their magnitudes, which bounds the rounding of any float32 accumulation
 * order.
 *
 * E4M3 ("fn" variant of the OCP 8-bit floating point formats): 1 sign bit, 4
 * exponent bits with bias 7, 3 mantissa bits; exponent 0 holds the subnormals
 * m/8 * 2^-6; S.1111.111 is NaN; there are no infinities (largest finite 448).
 */
double oracle_e4m3_value(uint8_t byte)
{
    int s = byte >> 7, e = (byte >> 3) & 15, m = byte & 7;
    if (e == 15 && m == 7) return 0.0 / 0.0;
#if ORACLE_MUTANT == 6 /* planted: exponent bias 8 instead of 7 */
    double v = e == 0 ? (m / 8.0) / 128.0 : (1.0 + m / 8.0) * (double)(1u << e) / 256.0;
#else
    double v = e == 0 ? (m / 8.0) / 64.0 : (1.0 + m / 8.0) * (double)(1u << e) / 128.0;
#endif
    return s ? -v : v;
}

/*
 * E5M2 (the other 8-bit format of the tutorial's gemm_fp8; OCP 8-bit floating
 * point, IEEE-like): 1 sign bit, 5 exponent bits with bias 15, 2 mantissa bits;
 * exponent 0 holds the subnormals m/4 * 2^-14; exponent 31 is infinity (m = 0)
 * or NaN (m != 0).  Largest finite value 57344.
 */
double oracle_e5m2_value(uint8_t byte)
{
    int s = byte >> 7, e = (byte >> 2) & 31, m = byte & 3;
    double v;
    if (e == 31) {
        if (m) return 0.0 / 0.0;
        v = 1.0 / 0.0;
    } else if (e == 0) {
#if ORACLE_MUTANT == 9 /* planted: subnormals decoded with the implicit leading one */
        v = (1.0 + m / 4.0) / 16384.0;
#else
        v = (m / 4.0) / 16384.0;
#endif
    } else {
        v = (1.0 + m / 4.0) * (double)(1u << e) / 32768.0;
    }
    return s ? -v : v;
}

/* Value of an fp8 byte in the given format (0 = E4M3, 1 = E5M2); -1 if unknown. */
static int decode_fp8(const uint8_t *src, double *dst, int64_t count, int format)
{
    if (format != 0 && format != 1) return -1;
    for (int64_t i = 0; i < count; ++i) dst[i] = format ? oracle_e5m2_value(src[i]) : oracle_e4m3_value(src[i]);
    return 0;
}

struct fjob {
    const double *a, *b;
    double *c, *cabs;
    int64_t N, K, m_begin, m_end;
};

static void *run_rows_f(void *arg)
{
    struct fjob *j = (struct fjob *)arg;
    for (int64_t m = j->m_begin; m < j->m_end; ++m) {
        for (int64_t n = 0; n < j->N; ++n) {
            const double *ar = j->a + m * j->K, *br = j->b + n * j->K;
            double s = 0.0, sa = 0.0;
            for (int64_t k = 0; k < j->K; ++k) {
                const double p = ar[k] * br[k];
                s += p;
                sa += p < 0 ? -p : p;
            }
            j->c[m * j->N + n] = s;
            j->cabs[m * j->N + n] = sa;
        }
    }
    return NULL;
}

/* A [M, K], B [N, K] fp8 bytes of `format` (0 = E4M3, 1 = E5M2, both operands);
 * C [M, N] = sum_k a*b and Cabs = sum_k |a*b| in double.  Returns 0, or -1 on an
 * allocation error or an unknown format. */
int oracle_fp8_gemm(const uint8_t *A, const uint8_t *B, double *C, double *Cabs, int64_t M, int64_t N,
                    int64_t K, int format, int nthreads)
{
    double *a = (double *)malloc(sizeof(double) * (size_t)(M * K > 0 ? M * K : 1));
    double *b = (double *)malloc(sizeof(double) * (size_t)(N * K > 0 ? N * K : 1));
    if (!a || !b || decode_fp8(A, a, M * K, format) || decode_fp8(B, b, N * K, format)) {
        free(a);
        free(b);
        return -1;
    }
    if (nthreads < 1) nthreads = 1;
    if (nthreads > M) nthreads = (int)(M > 0 ? M : 1);
    struct fjob *jobs = (struct fjob *)calloc((size_t)nthreads, sizeof(struct fjob));
    pthread_t *tids = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !tids) { free(a); free(b); free(jobs); free(tids); return -1; }
    for (int t = 0; t < nthreads; ++t) {
        jobs[t] = (struct fjob){a, b, C, Cabs, N, K, M * t / nthreads, M * (t + 1) / nthreads};
        if (pthread_create(&tids[t], NULL, run_rows_f, &jobs[t]) != 0) {
            run_rows_f(&jobs[t]);
            tids[t] = 0;
        }
    }
    for (int t = 0; t < nthreads; ++t)
        if (tids[t]) pthread_join(tids[t], NULL);
    free(jobs);
    free(tids);
    free(a);
    free(b);
    return 0;
}

/*
 * Block-scaled fp8 GEMM (the tutorial's gemm_blockscaled, low_precision_gemm.py):
 * A [M, K], B [N, K] fp8 bytes of `format` (0 = E4M3, 1 = E5M2); SFA [M, KB],
 * SFB [N, KB] float32 scales with
 * KB = ceil(K / g): the scales are applied along K per block of g values,
 *
 *   C[m,n] = sum_{kb} SFA[m,kb] * SFB[n,kb] * sum_{k in block kb} a[m,k]*b[n,k]
 *
 * in double; Cabs takes the same sums of magnitudes (the scale of any rounding).
 * Returns 0, or -1 on an allocation error or an unknown format.
 */
struct bjob {
    const double *a, *b;
    const float *sfa, *sfb;
    double *c, *cabs;
    int64_t N, K, g, KB, m_begin, m_end;
};

static void *run_rows_b(void *arg)
{
    struct bjob *j = (struct bjob *)arg;
    for (int64_t m = j->m_begin; m < j->m_end; ++m) {
        for (int64_t n = 0; n < j->N; ++n) {
            const double *ar = j->a + m * j->K, *br = j->b + n * j->K;
            double s = 0.0, sa = 0.0;
            for (int64_t kb = 0; kb < j->KB; ++kb) {
                double part = 0.0, pabs = 0.0;
                const int64_t k1 = (kb + 1) * j->g < j->K ? (kb + 1) * j->g : j->K;
                for (int64_t k = kb * j->g; k < k1; ++k) {
                    const double p = ar[k] * br[k];
                    part += p;
                    pabs += p < 0 ? -p : p;
                }
#if ORACLE_MUTANT == 7 /* planted: every block takes the scales of block 0 */
                const int64_t ks = 0;
#else
                const int64_t ks = kb;
#endif
#if ORACLE_MUTANT == 8 /* planted: SFA indexed by the B row */
                const double sc = (double)j->sfa[(n % (j->m_end > 0 ? j->m_end : 1)) * j->KB + ks] *
                                  (double)j->sfb[n * j->KB + ks];
#else
                const double sc = (double)j->sfa[m * j->KB + ks] * (double)j->sfb[n * j->KB + ks];
#endif
                s += sc * part;
                sa += (sc < 0 ? -sc : sc) * pabs;
            }
            j->c[m * j->N + n] = s;
            j->cabs[m * j->N + n] = sa;
        }
    }
    return NULL;
}

int oracle_fp8_blockscaled(const uint8_t *A, const uint8_t *B, const float *SFA, const float *SFB, double *C,
                           double *Cabs, int64_t M, int64_t N, int64_t K, int64_t g, int format, int nthreads)
{
    if (g < 1) return -1;
    const int64_t KB = (K + g - 1) / g;
    double *a = (double *)malloc(sizeof(double) * (size_t)(M * K > 0 ? M * K : 1));
    double *b = (double *)malloc(sizeof(double) * (size_t)(N * K > 0 ? N * K : 1));
    if (!a || !b || decode_fp8(A, a, M * K, format) || decode_fp8(B, b, N * K, format)) {
        free(a);
        free(b);
        return -1;
    }
    if (nthreads < 1) nthreads = 1;
    if (nthreads > M) nthreads = (int)(M > 0 ? M : 1);
    struct bjob *jobs = (struct bjob *)calloc((size_t)nthreads, sizeof(struct bjob));
    pthread_t *tids = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !tids) { free(a); free(b); free(jobs); free(tids); return -1; }
    for (int t = 0; t < nthreads; ++t) {
        jobs[t] = (struct bjob){a, b, SFA, SFB, C, Cabs, N, K, g, KB, M * t / nthreads, M * (t + 1) / nthreads};
        if (pthread_create(&tids[t], NULL, run_rows_b, &jobs[t]) != 0) {
            run_rows_b(&jobs[t]);
            tids[t] = 0;
        }
    }
    for (int t = 0; t < nthreads; ++t)
        if (tids[t]) pthread_join(tids[t], NULL);
    free(jobs);
    free(tids);
    free(a);
    free(b);
    return 0;
}

