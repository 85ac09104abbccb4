/*
 * CPU FP64 oracle for the dense tiled GEMM C = A·B: test infrastructure only.
 *
 * Only the tests, the package's smoke check and the benchmark's CPU-baseline
 * leg use this file. The product path never links or calls it.
 *
 * It computes the definition the tiled kernel computes. "Two Waves, One Stage
 * Apart: Warp-Pipelining Triton GEMMs on AMD Instinct" (opening paragraph)
 * defines tiled GEMM as computing on one pair of operand tiles after another,
 * with each output tile the sum over K of A-tile·B-tile products. Summed over
 * all tiles, that is
 *
 *     C[i][j] = sum_{k=0}^{K-1} a[i][k] * b[k][j]
 *
 * and the oracle evaluates it in FP64, with k ascending, over the exact
 * values of the FP16/BF16 or FP8 (E4M3, E5M2) operands. It also returns
 *
 *     C_abs[i][j] = sum_k |a[i][k] * b[k][j]|
 *
 * which the acceptance bound uses. Every product of two FP16 values (11-bit
 * significands), two BF16 values (8-bit) or two FP8 values (4-bit E4M3,
 * 3-bit E5M2) is exact in FP64, so the only rounding is in the FP64 running
 * sum. No blocking or reordering: one plain i-k-j loop per output row, with
 * rows shared among threads.
 *
 * Block-scaled (MX) inputs: "Two Waves, One Stage Apart" (section "MI450",
 * Table 1) measures MXFP8 and MXFP4 GEMMs without defining the formats; the
 * reading taken is OCP Microscaling: elements E4M3/E5M2 (MXFP8) or E2M1
 * (MXFP4), and one E8M0 scale 2^(e-127) shared by each run of 32 consecutive
 * K elements of a row of A, and of a column of B. oracle_gemm_mx computes
 *
 *     C[i][j] = sum_k (sa[i][k/32] * a[i][k]) * (sb[j][k/32] * b[k][j])
 *
 * with each scaled operand formed exactly in FP64 before the product (the
 * scaled values are powers of two times short significands).
 *
 * FP8 inputs follow "Porting High-Performance HIP Kernels to FlyDSL"
 * (section "A More Complex Kernel"): E4M3 operands, FP32 accumulation and a
 * block scale of 1.0 on every operand (the identity scale), so the scaled
 * product is the plain product and the definition above is unchanged. The
 * same page's BF8 sibling (E5M2, named among the FP8/BF8 formats of the RDNA
 * instruction-set pages) is decoded too.
 *
 * Operand storage (the reading taken for the "K-major" wording of the pages'
 * kernels, whose B operand is passed transposed, "B_T"); elements are 16-bit
 * words for FP16/BF16 and bytes for FP8:
 *   A       : M x K row-major, a[i][k] at A[i*K + k]
 *   B k-major : N x K, K contiguous, b[k][j] at B[j*K + k]
 *   B mn-major: K x N, N contiguous, b[k][j] at B[k*N + j]
 *
 * Build: plain C99, gcc -O2 -ffp-contract=off (no fused multiply-add, so
 * x86 and Arm hosts give identical bits), -pthread.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

enum { ORACLE_F16 = 0, ORACLE_BF16 = 1, ORACLE_E4M3 = 3, ORACLE_E5M2 = 4, ORACLE_E2M1 = 5 };
enum { ORACLE_MX_BLOCK = 32 };
enum { ORACLE_K_MAJOR = 0, ORACLE_MN_MAJOR = 1 };

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits.
 * Normal:    (1024 + f) * 2^(e - 15 - 10)
 * Subnormal: f * 2^(1 - 15 - 10) = f * 2^-24                                */
double oracle_decode_f16(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);
    else if (e == 0x1f)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + f), e - 25);
    return sign ? -v : v;
}

/* bfloat16: the upper half of an IEEE binary32: 1 sign bit, 8 exponent bits
 * (bias 127), 7 fraction bits.
 * Normal:    (128 + f) * 2^(e - 127 - 7)
 * Subnormal: f * 2^(1 - 127 - 7) = f * 2^-133                               */
double oracle_decode_bf16(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 7) & 0xff;
    int f = h & 0x7f;
    double v;
    if (e == 0)
        v = ldexp((double)f, -133);
    else if (e == 0xff)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(128 + f), e - 134);
    return sign ? -v : v;
}

/* FP8 E4M3 in its "FN" form (finite, NaN only): 1 sign bit, 4 exponent bits
 * (bias 7), 3 fraction bits, no infinities; S.1111.111 is NaN, so the largest
 * finite magnitude is 1.75 * 2^8 = 448.
 * Normal:    (8 + f) * 2^(e - 7 - 3)
 * Subnormal: f * 2^(1 - 7 - 3) = f * 2^-9                                   */
double oracle_decode_e4m3(uint8_t h)
{
    int sign = (h >> 7) & 1;
    int e = (h >> 3) & 0xf;
    int f = h & 0x7;
    double v;
    if (e == 0)
        v = ldexp((double)f, -9);
    else if (e == 0xf && f == 0x7)
        v = NAN;
    else
        v = ldexp((double)(8 + f), e - 10);
    return sign ? -v : v;
}

/* FP8 E5M2: 1 sign bit, 5 exponent bits (bias 15), 2 fraction bits, with
 * IEEE infinities and NaNs at exponent 31; largest finite 1.75 * 2^15.
 * Normal:    (4 + f) * 2^(e - 15 - 2)
 * Subnormal: f * 2^(1 - 15 - 2) = f * 2^-16                                 */
double oracle_decode_e5m2(uint8_t h)
{
    int sign = (h >> 7) & 1;
    int e = (h >> 2) & 0x1f;
    int f = h & 0x3;
    double v;
    if (e == 0)
        v = ldexp((double)f, -16);
    else if (e == 0x1f)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(4 + f), e - 17);
    return sign ? -v : v;
}

/* FP4 E2M1 (OCP): 1 sign bit, 2 exponent bits (bias 1), 1 fraction bit, no
 * infinities or NaNs; magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6.
 * Normal:    (2 + f) * 2^(e - 1 - 1)
 * Subnormal: f * 2^(1 - 1 - 1) = f * 0.5                                    */
double oracle_decode_e2m1(uint8_t h)
{
    int sign = (h >> 3) & 1;
    int e = (h >> 1) & 0x3;
    int f = h & 0x1;
    double v = e == 0 ? ldexp((double)f, -1) : ldexp((double)(2 + f), e - 2);
    return sign ? -v : v;
}

/* E8M0 scale (OCP): an 8-bit biased exponent, value 2^(e - 127); 0xFF is NaN. */
double oracle_decode_e8m0(uint8_t e)
{
    return e == 0xFF ? NAN : ldexp(1.0, (int)e - 127);
}

static int is_fp8(int dtype)
{
    return dtype == ORACLE_E4M3 || dtype == ORACLE_E5M2;
}

/* element idx of an operand array holding dtype's patterns. E2M1 elements
 * are packed two per byte, the lower index in the low nibble; `idx` then
 * counts nibbles. */
static double decode(const void *base, int64_t idx, int dtype)
{
    switch (dtype) {
    case ORACLE_E2M1: {
        const uint8_t byte = ((const uint8_t *)base)[idx >> 1];
        return oracle_decode_e2m1((idx & 1) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 0xF));
    }
    case ORACLE_BF16: return oracle_decode_bf16(((const uint16_t *)base)[idx]);
    case ORACLE_E4M3: return oracle_decode_e4m3(((const uint8_t *)base)[idx]);
    case ORACLE_E5M2: return oracle_decode_e5m2(((const uint8_t *)base)[idx]);
    default:          return oracle_decode_f16(((const uint16_t *)base)[idx]);
    }
}

typedef struct {
    /* shared */
    const void *A;
    const double *Bd;      /* decoded b[k][j], K x N row-major */
    const void *B;         /* raw B, for the decode phase */
    const uint8_t *sfa, *sfb;  /* MX scales (E8M0), rows x n_blocks; NULL: unscaled */
    int64_t n_blocks;      /* scale blocks per row = ceil(K / 32) */
    int64_t row_elems;     /* element slots per stored row (K, or K rounded up to even for E2M1) */
    int64_t M, N, K;
    int dtype, layout_b;
    const int64_t *rows;
    int64_t n_rows;
    double *C, *C_abs;
    /* per thread */
    int64_t lo, hi;        /* range of output rows (decode: range of k) */
    int phase;             /* 0: decode B, 1: rows of C */
} job_t;

static void decode_b_rows(const job_t *j)
{
    double *Bd = (double *)j->Bd;
    for (int64_t k = j->lo; k < j->hi; ++k)
        for (int64_t c = 0; c < j->N; ++c) {
            int64_t idx = j->layout_b == ORACLE_K_MAJOR ? c * j->row_elems + k : k * j->N + c;
            double v = decode(j->B, idx, j->dtype);
            if (j->sfb)
                v *= oracle_decode_e8m0(j->sfb[c * j->n_blocks + k / ORACLE_MX_BLOCK]);
            Bd[k * j->N + c] = v;
        }
}

static void gemm_rows(const job_t *j)
{
    const int64_t N = j->N, K = j->K;
    for (int64_t r = j->lo; r < j->hi; ++r) {
        const int64_t i = j->rows ? j->rows[r] : r;
        double *c = j->C + r * N;
        double *cabs = j->C_abs + r * N;
        for (int64_t col = 0; col < N; ++col) {
            c[col] = 0.0;
            cabs[col] = 0.0;
        }
        for (int64_t k = 0; k < K; ++k) {
            double a = decode(j->A, i * j->row_elems + k, j->dtype);
            if (j->sfa)
                a *= oracle_decode_e8m0(j->sfa[i * j->n_blocks + k / ORACLE_MX_BLOCK]);
            const double *b = j->Bd + k * N;
            for (int64_t col = 0; col < N; ++col) {
                const double p = a * b[col];
                c[col] += p;
                cabs[col] += fabs(p);
            }
        }
    }
}

static void *worker(void *arg)
{
    const job_t *j = (const job_t *)arg;
    if (j->phase == 0)
        decode_b_rows(j);
    else
        gemm_rows(j);
    return NULL;
}

static int run_threads(job_t *base, int64_t count, int n_threads)
{
    if (count <= 0)
        return 0;
    if (n_threads > count)
        n_threads = (int)count;
    pthread_t *tid = (pthread_t *)calloc((size_t)n_threads, sizeof(pthread_t));
    char *started = (char *)calloc((size_t)n_threads, 1);
    job_t *jobs = (job_t *)calloc((size_t)n_threads, sizeof(job_t));
    if (!tid || !jobs || !started) {
        free(tid);
        free(started);
        free(jobs);
        return -2;
    }
    for (int t = 0; t < n_threads; ++t) {
        jobs[t] = *base;
        jobs[t].lo = count * t / n_threads;
        jobs[t].hi = count * (t + 1) / n_threads;
        if (t == n_threads - 1)
            worker(&jobs[t]);   /* the calling thread takes the last share */
        else if (pthread_create(&tid[t], NULL, worker, &jobs[t]) == 0)
            started[t] = 1;
        else
            worker(&jobs[t]);   /* no thread available: do the share inline */
    }
    for (int t = 0; t < n_threads - 1; ++t)
        if (started[t])
            pthread_join(tid[t], NULL);
    free(tid);
    free(started);
    free(jobs);
    return 0;
}

static int run_gemm(const void *A, const void *B, const uint8_t *sfa, const uint8_t *sfb, int64_t M,
                    int64_t N, int64_t K, int dtype, int layout_b, const int64_t *rows, int64_t n_rows,
                    double *C, double *C_abs, int n_threads)
{
    if (rows) {
        for (int64_t r = 0; r < n_rows; ++r)
            if (rows[r] < 0 || rows[r] >= M)
                return -1;
    } else {
        n_rows = M;
    }
    if (n_threads <= 0) {
        long n = sysconf(_SC_NPROCESSORS_ONLN);
        n_threads = n > 0 ? (int)n : 1;
    }
    double *Bd = (double *)malloc((size_t)K * (size_t)N * sizeof(double));
    if (!Bd)
        return -2;
    job_t base;
    memset(&base, 0, sizeof(base));
    base.A = A;
    base.B = B;
    base.Bd = Bd;
    base.sfa = sfa;
    base.sfb = sfb;
    base.n_blocks = (K + ORACLE_MX_BLOCK - 1) / ORACLE_MX_BLOCK;
    base.row_elems = dtype == ORACLE_E2M1 ? (K + 1) / 2 * 2 : K;
    base.M = M;
    base.N = N;
    base.K = K;
    base.dtype = dtype;
    base.layout_b = layout_b;
    base.rows = rows;
    base.n_rows = n_rows;
    base.C = C;
    base.C_abs = C_abs;

    /* phase 0 decodes (and scales) b[k][j] into FP64 once; phase 1 runs the row loops */
    base.phase = 0;
    int rc = run_threads(&base, K, n_threads);
    if (rc == 0) {
        base.phase = 1;
        rc = run_threads(&base, n_rows, n_threads);
    }
    free(Bd);
    return rc;
}

/*
 * Compute selected rows of C = A·B in FP64.
 *   A, B      : raw operand patterns (16-bit words for ORACLE_F16 and
 *               ORACLE_BF16, bytes for ORACLE_E4M3 and ORACLE_E5M2),
 *               layouts as described above
 *   dtype     : the element type of both operands
 *   layout_b  : ORACLE_K_MAJOR or ORACLE_MN_MAJOR
 *   rows      : indices of the output rows to compute, or NULL for all M
 *   n_rows    : number of entries in rows (ignored when rows is NULL)
 *   C, C_abs  : n_rows x N (or M x N) row-major outputs
 *   n_threads : worker threads (<= 0: all online CPUs)
 * Returns 0 on success, -1 for invalid arguments, -2 when memory runs out.
 */
int oracle_gemm(const void *A, const void *B, int64_t M, int64_t N, int64_t K,
                int dtype, int layout_b, const int64_t *rows, int64_t n_rows,
                double *C, double *C_abs, int n_threads)
{
    if (!A || !B || !C || !C_abs || M <= 0 || N <= 0 || K <= 0)
        return -1;
    if (dtype != ORACLE_F16 && dtype != ORACLE_BF16 && !is_fp8(dtype))
        return -1;
    if (layout_b != ORACLE_K_MAJOR && layout_b != ORACLE_MN_MAJOR)
        return -1;
    return run_gemm(A, B, NULL, NULL, M, N, K, dtype, layout_b, rows, n_rows, C, C_abs, n_threads);
}

/*
 * Block-scaled (MX) GEMM rows in FP64: C = (SFA ∘ A)·(SFB ∘ B), see the top
 * of this file.
 *   A         : M x K elements, row-major; bytes for ORACLE_E4M3/ORACLE_E5M2,
 *               or E2M1 nibbles packed two per byte with each row padded to a
 *               whole byte (row pitch ceil(K/2) bytes), lower k in the low nibble
 *   B         : N x K (K-major, the same element layout as A)
 *   sfa, sfb  : E8M0 scales, M x ceil(K/32) and N x ceil(K/32) bytes, row-major
 *   other arguments as for oracle_gemm (B must be K-major)
 */
int oracle_gemm_mx(const void *A, const void *B, const uint8_t *sfa, const uint8_t *sfb, int64_t M,
                   int64_t N, int64_t K, int dtype, const int64_t *rows, int64_t n_rows, double *C,
                   double *C_abs, int n_threads)
{
    if (!A || !B || !sfa || !sfb || !C || !C_abs || M <= 0 || N <= 0 || K <= 0)
        return -1;
    if (!is_fp8(dtype) && dtype != ORACLE_E2M1)
        return -1;
    return run_gemm(A, B, sfa, sfb, M, N, K, dtype, ORACLE_K_MAJOR, rows, n_rows, C, C_abs, n_threads);
}
