/*
 * CPU FP64 oracle for the attention forward pass: test infrastructure only.
 *
 * Only the tests, the package's smoke check and the benchmark's CPU legs use
 * this file. The product path never links or calls it.
 *
 * "Two Waves, One Stage Apart" (section "Beyond GEMM: FlashAttention")
 * describes the inner loop of FlashAttention: QK and PV products alternating
 * with an online softmax over key/value blocks. The online form reaches, up
 * to rounding, the plain definition, which this oracle evaluates directly:
 *
 *     s[i][k] = scale * sum_c q[i][c] * k[k][c]          (k allowed for row i)
 *     m[i]    = max_k s[i][k]
 *     p[i][k] = exp(s[i][k] - m[i])
 *     l[i]    = sum_k p[i][k]
 *     O[i][j] = sum_k p[i][k] * v[k][j] / l[i]
 *     LSE[i]  = m[i] + log(l[i])
 *
 * plus O_abs[i][j] = sum_k p[i][k] * |v[k][j]| / l[i] for the acceptance
 * bound. Subtracting m[i] leaves the softmax unchanged (it only keeps exp in
 * range). Key k is allowed for query row i always, or, when causal, iff
 * k <= i + (Lk - Lq) (the last query row sees every key). Everything is FP64
 * over the exact FP16/BF16 operand values; sums run with k ascending.
 *
 * Storage: Q is [B][H][Lq][d], K and V are [B][H][Lk][d], all row-major and
 * densely packed 16-bit patterns; outputs are [n_rows][d] (O, O_abs) and
 * [n_rows] (LSE) for the selected flat query rows r = (b*H + h)*Lq + i.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

double oracle_decode_f16(uint16_t h);
double oracle_decode_bf16(uint16_t h);

enum { ATT_F16 = 0, ATT_BF16 = 1 };

typedef struct {
    const uint16_t *Q, *K, *V;
    int64_t B, H, Lq, Lk, d;
    int dtype, causal;
    double scale;
    const int64_t *rows;
    double *O, *O_abs, *LSE;
    int64_t lo, hi;
} att_job_t;

static double dec(uint16_t x, int dtype)
{
    return dtype == ATT_BF16 ? oracle_decode_bf16(x) : oracle_decode_f16(x);
}

static void *att_worker(void *arg)
{
    const att_job_t *j = (const att_job_t *)arg;
    const int64_t d = j->d, Lk = j->Lk;
    double *q = (double *)malloc((size_t)d * sizeof(double));
    double *s = (double *)malloc((size_t)Lk * sizeof(double));
    if (!q || !s) {
        free(q);
        free(s);
        return (void *)1;
    }
    for (int64_t r = j->lo; r < j->hi; ++r) {
        const int64_t flat = j->rows ? j->rows[r] : r;
        const int64_t bh = flat / j->Lq, i = flat % j->Lq;
        const uint16_t *qrow = j->Q + flat * d;
        const uint16_t *kmat = j->K + bh * Lk * d;
        const uint16_t *vmat = j->V + bh * Lk * d;
        for (int64_t c = 0; c < d; ++c)
            q[c] = dec(qrow[c], j->dtype);
        /* keys allowed for this row: [0, n_keys) */
        int64_t n_keys = Lk;
        if (j->causal) {
            n_keys = i + (Lk - j->Lq) + 1;
            if (n_keys > Lk)
                n_keys = Lk;
            if (n_keys < 0)
                n_keys = 0;
        }
        double m = -INFINITY;
        for (int64_t k = 0; k < n_keys; ++k) {
            double acc = 0.0;
            for (int64_t c = 0; c < d; ++c)
                acc += q[c] * dec(kmat[k * d + c], j->dtype);
            s[k] = j->scale * acc;
            if (s[k] > m)
                m = s[k];
        }
        double l = 0.0;
        for (int64_t k = 0; k < n_keys; ++k) {
            s[k] = exp(s[k] - m); /* now p[k] */
            l += s[k];
        }
        double *o = j->O + r * d, *oa = j->O_abs + r * d;
        for (int64_t c = 0; c < d; ++c) {
            o[c] = 0.0;
            oa[c] = 0.0;
        }
        for (int64_t k = 0; k < n_keys; ++k)
            for (int64_t c = 0; c < d; ++c) {
                const double pv = s[k] * dec(vmat[k * d + c], j->dtype);
                o[c] += pv;
                oa[c] += fabs(pv);
            }
        for (int64_t c = 0; c < d; ++c) {
            o[c] = n_keys ? o[c] / l : 0.0;
            oa[c] = n_keys ? oa[c] / l : 0.0;
        }
        j->LSE[r] = n_keys ? m + log(l) : -INFINITY;
    }
    free(q);
    free(s);
    return NULL;
}

/*
 * Attention forward rows in FP64 (see above).
 *   Q, K, V   : raw 16-bit patterns of dtype (0: FP16, 1: BF16)
 *   rows      : flat query rows to compute ((b*H + h)*Lq + i), NULL for all
 *   n_rows    : entries in rows (ignored when rows is NULL)
 *   scale     : the score scale (1/sqrt(d) in the usual form)
 *   O, O_abs  : n_rows x d outputs; LSE: n_rows outputs
 *   n_threads : worker threads (<= 0: all online CPUs)
 * Returns 0 on success, -1 for invalid arguments, -2 when memory runs out.
 */
int oracle_attention(const uint16_t *Q, const uint16_t *K, const uint16_t *V, int64_t B, int64_t H,
                     int64_t Lq, int64_t Lk, int64_t d, int dtype, int causal, double scale,
                     const int64_t *rows, int64_t n_rows, double *O, double *O_abs, double *LSE,
                     int n_threads)
{
    if (!Q || !K || !V || !O || !O_abs || !LSE || B <= 0 || H <= 0 || Lq <= 0 || Lk <= 0 || d <= 0)
        return -1;
    if (dtype != ATT_F16 && dtype != ATT_BF16)
        return -1;
    const int64_t total = B * H * Lq;
    if (rows) {
        for (int64_t r = 0; r < n_rows; ++r)
            if (rows[r] < 0 || rows[r] >= total)
                return -1;
    } else {
        n_rows = total;
    }
    if (n_threads <= 0) {
        long n = sysconf(_SC_NPROCESSORS_ONLN);
        n_threads = n > 0 ? (int)n : 1;
    }
    if (n_threads > n_rows)
        n_threads = (int)(n_rows > 0 ? n_rows : 1);
    att_job_t base;
    memset(&base, 0, sizeof(base));
    base.Q = Q;
    base.K = K;
    base.V = V;
    base.B = B;
    base.H = H;
    base.Lq = Lq;
    base.Lk = Lk;
    base.d = d;
    base.dtype = dtype;
    base.causal = causal;
    base.scale = scale;
    base.rows = rows;
    base.O = O;
    base.O_abs = O_abs;
    base.LSE = LSE;
    pthread_t *tid = (pthread_t *)calloc((size_t)n_threads, sizeof(pthread_t));
    char *started = (char *)calloc((size_t)n_threads, 1);
    att_job_t *jobs = (att_job_t *)calloc((size_t)n_threads, sizeof(att_job_t));
    if (!tid || !started || !jobs) {
        free(tid);
        free(started);
        free(jobs);
        return -2;
    }
    int rc = 0;
    for (int t = 0; t < n_threads; ++t) {
        jobs[t] = base;
        jobs[t].lo = n_rows * t / n_threads;
        jobs[t].hi = n_rows * (t + 1) / n_threads;
        if (t == n_threads - 1 || pthread_create(&tid[t], NULL, att_worker, &jobs[t]) != 0) {
            if (att_worker(&jobs[t]))
                rc = -2;
        } else {
            started[t] = 1;
        }
    }
    for (int t = 0; t < n_threads; ++t)
        if (started[t]) {
            void *ret = NULL;
            pthread_join(tid[t], &ret);
            if (ret)
                rc = -2;
        }
    free(tid);
    free(started);
    free(jobs);
    return rc;
}
