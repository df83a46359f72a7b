/*
 * fp64 CPU oracle for exact softmax attention.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path links, loads or calls
 * this file; only the tests, the bench's CPU-baseline leg and the smoke check
 * do. It shares no code, header or constant with the CUDA path.
 *
 * What it computes is the plain definition of attention, written out one query
 * row at a time:
 *
 *   S = Q Kᵀ · scale          (scores)
 *   P = softmax(S) over rows  (probabilities; causal: S[i,j] = -inf for j > i)
 *   O = P V                   (outputs)
 *
 * ("Mini FlashAttention", §1 "What attention is", the three-line math and the
 * causal-mask sentence after it; "How Did I Write My First FlashAttention
 * Kernel in CUDA?", the "Standard attention computes" paragraph.)
 *
 * Layout: Q, K, V, O are contiguous [B, H, N, d] row-major; LSE is [B, H, N].
 * The log-sum-exp of a row is LSE_i = ln Σ_j exp(S[i,j]) over the unmasked
 * keys, computed as M_i + ln Z_i with M_i the row maximum. A row whose keys
 * are all masked (not reachable with a square causal mask, kept for
 * completeness) gives O = 0 and LSE = -inf.
 *
 * A second entry point runs the chunked online-softmax loop of "Mini
 * FlashAttention", §4 "The flash trick: online softmax" (running max m,
 * running sum l, running output acc, rescaled by alpha = exp(m_old - m_new)
 * when a chunk raises the max, O = acc / l after the last chunk), with the
 * page's guard that pins m_new to 0 when it is still -inf. It exists so that
 * tests can check that the streaming form equals the definition, which is the
 * claim the method rests on ("Mini FlashAttention", §4; "How Did I Write My
 * First FlashAttention Kernel in CUDA?", the surrogate-output paragraph).
 *
 * A third entry point takes a variable-length batch: sequences with their
 * own query and key counts, tokens stored as rows of [total, H, d], and the
 * causal mask aligned so that each sequence's last query sees its last key
 * (the plainest reading for queries and keys of different lengths; with equal
 * lengths it is the mask above). It calls the same per-row definition.
 *
 * Every function returns 0 on success and a negative value on bad arguments.
 * Threads (POSIX) split independent query rows; each row is computed by one
 * thread in a fixed order, so results do not depend on the thread count.
 */
#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

/* ---------- one query row, by the definition ------------------------------ */

/* Row i of head (q_row, k, v): keys 0 .. n_keys-1 take part (n_keys = N, or
 * i+1 under the causal mask). Key j's row of K and V starts at j * kv_stride.
 * s_buf holds n_keys doubles of scratch. */
static void definition_row(const double *q_row, const double *k, const double *v,
                           long n_keys, long d, long kv_stride, double scale, double *s_buf,
                           double *o_row, double *lse_out)
{
    long j, c;
    if (n_keys <= 0) { /* every key masked */
        for (c = 0; c < d; ++c) o_row[c] = 0.0;
        *lse_out = -INFINITY;
        return;
    }
    /* S[i, j] = scale * <Q[i], K[j]> */
    for (j = 0; j < n_keys; ++j) {
        double x = 0.0;
        for (c = 0; c < d; ++c) x += q_row[c] * k[j * kv_stride + c];
        s_buf[j] = scale * x;
    }
    /* P[i, :] = softmax(S[i, :]): max, sum of exponentials, normalise */
    double m = -INFINITY;
    for (j = 0; j < n_keys; ++j) if (s_buf[j] > m) m = s_buf[j];
    double z = 0.0;
    for (j = 0; j < n_keys; ++j) z += exp(s_buf[j] - m);
    for (j = 0; j < n_keys; ++j) s_buf[j] = exp(s_buf[j] - m) / z; /* now P[i, j] */
    /* O[i, :] = P[i, :] V */
    for (c = 0; c < d; ++c) o_row[c] = 0.0;
    for (j = 0; j < n_keys; ++j) {
        const double p = s_buf[j];
        for (c = 0; c < d; ++c) o_row[c] += p * v[j * kv_stride + c];
    }
    *lse_out = m + log(z);
}

/* ---------- one query row, by the chunked online-softmax loop ------------- */

static void online_row(const double *q_row, const double *k, const double *v,
                       long n_keys, long d, double scale, long chunk,
                       double *s_buf, double *acc, double *o_row, double *lse_out)
{
    long c, j, j0;
    double m_i = -INFINITY; /* running max, starts at -inf */
    double l_i = 0.0;       /* running sum of exp, starts at 0 */
    for (c = 0; c < d; ++c) acc[c] = 0.0; /* running P V, starts at 0 */
    for (j0 = 0; j0 < n_keys; j0 += chunk) {
        long len = n_keys - j0 < chunk ? n_keys - j0 : chunk;
        double m_chunk = -INFINITY;
        for (j = 0; j < len; ++j) {
            double x = 0.0;
            for (c = 0; c < d; ++c) x += q_row[c] * k[(j0 + j) * d + c];
            s_buf[j] = scale * x;
            if (s_buf[j] > m_chunk) m_chunk = s_buf[j];
        }
        double m_new = m_i > m_chunk ? m_i : m_chunk;
        if (m_new == -INFINITY) m_new = 0.0; /* guard: a fully masked row stays finite */
        double alpha = exp(m_i - m_new);     /* rescale factor for the old state */
        double sum_p = 0.0;
        for (c = 0; c < d; ++c) acc[c] *= alpha;
        for (j = 0; j < len; ++j) {
            double p = exp(s_buf[j] - m_new);
            sum_p += p;
            for (c = 0; c < d; ++c) acc[c] += p * v[(j0 + j) * d + c];
        }
        l_i = l_i * alpha + sum_p;
        m_i = m_new;
    }
    if (l_i > 0.0) {
        for (c = 0; c < d; ++c) o_row[c] = acc[c] / l_i;
        *lse_out = m_i + log(l_i);
    } else {
        for (c = 0; c < d; ++c) o_row[c] = 0.0;
        *lse_out = -INFINITY;
    }
}

/* ---------- threading over independent rows ------------------------------ */

typedef struct {
    const double *q, *k, *v;
    double *o, *lse;
    long B, H, N, d;
    double scale;
    int causal;
    long chunk;            /* 0: definition; > 0: online loop with this chunk */
    const long *rows;      /* NULL: every row b*H*N + h*N + i; else a list */
    long n_rows;
    long next;             /* next row index to hand out (under lock) */
    pthread_mutex_t lock;
    int failed;
} job_t;

enum { ROWS_PER_GRAB = 16 };

static void *worker(void *arg)
{
    job_t *job = (job_t *)arg;
    const long N = job->N, d = job->d;
    double *s_buf = (double *)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1));
    double *acc = (double *)malloc(sizeof(double) * (size_t)d);
    if (!s_buf || !acc) {
        pthread_mutex_lock(&job->lock);
        job->failed = 1;
        pthread_mutex_unlock(&job->lock);
        free(s_buf);
        free(acc);
        return NULL;
    }
    for (;;) {
        pthread_mutex_lock(&job->lock);
        long start = job->next;
        job->next += ROWS_PER_GRAB;
        pthread_mutex_unlock(&job->lock);
        if (start >= job->n_rows) break;
        long stop = start + ROWS_PER_GRAB < job->n_rows ? start + ROWS_PER_GRAB : job->n_rows;
        for (long r = start; r < stop; ++r) {
            long flat = job->rows ? job->rows[r] : r; /* (b*H + h)*N + i */
            long head = flat / N, i = flat % N;
            const double *q_row = job->q + flat * d;
            const double *k = job->k + head * N * d;
            const double *v = job->v + head * N * d;
            long n_keys = job->causal ? i + 1 : N;
            double *o_row = job->o + r * d;
            double *lse = job->lse + r;
            if (job->chunk > 0)
                online_row(q_row, k, v, n_keys, d, job->scale, job->chunk, s_buf, acc, o_row, lse);
            else
                definition_row(q_row, k, v, n_keys, d, d, job->scale, s_buf, o_row, lse);
        }
    }
    free(s_buf);
    free(acc);
    return NULL;
}

static long host_threads(void)
{
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    return n > 0 ? n : 1;
}

static int run_job(job_t *job, int nthreads)
{
    long n = nthreads > 0 ? nthreads : host_threads();
    if (n > job->n_rows) n = job->n_rows > 0 ? job->n_rows : 1;
    pthread_t *tids = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)n);
    if (!tids) return -3;
    pthread_mutex_init(&job->lock, NULL);
    job->next = 0;
    job->failed = 0;
    long started = 0;
    for (long t = 0; t < n; ++t) {
        if (pthread_create(&tids[t], NULL, worker, job) != 0) break;
        ++started;
    }
    if (started == 0) worker(job); /* no thread could start: run inline */
    for (long t = 0; t < started; ++t) pthread_join(tids[t], NULL);
    pthread_mutex_destroy(&job->lock);
    free(tids);
    return job->failed ? -3 : 0;
}

static int check_shape(long B, long H, long N, long d)
{
    return (B < 0 || H < 0 || N < 0 || d <= 0) ? -2 : 0;
}

/* ---------- variable-length batches -------------------------------------- */

/* Sequence b holds query tokens cu_q[b] .. cu_q[b+1]-1 and key tokens
 * cu_k[b] .. cu_k[b+1]-1 (Nq and Nk of them). Tokens are rows of [total, H, d]
 * (a token's H heads side by side). Under the causal mask the last query of a
 * sequence lines up with its last key: query i (0-based in its sequence) sees
 * keys j <= i + Nk - Nq, a prefix of the sequence's keys; a query that sees
 * none gives O = 0 and LSE = -inf. Rows are numbered h * total_q + token,
 * which is also the LSE layout [H, total_q]. */
typedef struct {
    const double *q, *k, *v;
    double *o, *lse;
    const long *cu_q, *cu_k;
    long B, H, d, total_q;
    double scale;
    int causal;
    long max_nk;
    long next;
    pthread_mutex_t lock;
    int failed;
} vjob_t;

static void *varlen_worker(void *arg)
{
    vjob_t *job = (vjob_t *)arg;
    const long H = job->H, d = job->d, n_rows = job->H * job->total_q;
    double *s_buf = (double *)malloc(sizeof(double) * (size_t)(job->max_nk > 0 ? job->max_nk : 1));
    if (!s_buf) {
        pthread_mutex_lock(&job->lock);
        job->failed = 1;
        pthread_mutex_unlock(&job->lock);
        return NULL;
    }
    for (;;) {
        pthread_mutex_lock(&job->lock);
        long start = job->next;
        job->next += ROWS_PER_GRAB;
        pthread_mutex_unlock(&job->lock);
        if (start >= n_rows) break;
        long stop = start + ROWS_PER_GRAB < n_rows ? start + ROWS_PER_GRAB : n_rows;
        for (long r = start; r < stop; ++r) {
            long h = r / job->total_q, tok = r % job->total_q;
            long b = 0; /* the sequence holding query token tok */
            while (b + 1 < job->B && job->cu_q[b + 1] <= tok) ++b;
            long nq = job->cu_q[b + 1] - job->cu_q[b], nk = job->cu_k[b + 1] - job->cu_k[b];
            long i = tok - job->cu_q[b];
            long n_keys = nk;
            if (job->causal) {
                n_keys = i + nk - nq + 1;
                if (n_keys < 0) n_keys = 0;
                if (n_keys > nk) n_keys = nk;
            }
            const double *q_row = job->q + (tok * H + h) * d;
            const double *k = job->k + (job->cu_k[b] * H + h) * d;
            const double *v = job->v + (job->cu_k[b] * H + h) * d;
            definition_row(q_row, k, v, n_keys, d, H * d, job->scale, s_buf,
                           job->o + (tok * H + h) * d, job->lse + r);
        }
    }
    free(s_buf);
    return NULL;
}

/* ---------- exported entry points ----------------------------------------- */

/* Number of host threads the oracle uses when asked for 0. */
int oracle_host_threads(void) { return (int)host_threads(); }

/* Every row of every head, by the definition. o: [B,H,N,d], lse: [B,H,N]. */
int oracle_attn_fwd_f64(const double *q, const double *k, const double *v,
                        double *o, double *lse, long B, long H, long N, long d,
                        double scale, int causal, int nthreads)
{
    if (!q || !k || !v || !o || !lse) return -1;
    if (check_shape(B, H, N, d)) return -2;
    job_t job = {q, k, v, o, lse, B, H, N, d, scale, causal, 0, NULL, B * H * N};
    return run_job(&job, nthreads);
}

/* A chosen list of rows (flat index (b*H + h)*N + i), by the definition.
 * q, k, v are the full [B,H,N,d] inputs; o: [n_rows, d], lse: [n_rows]. */
int oracle_attn_rows_f64(const double *q, const double *k, const double *v,
                         double *o, double *lse, long B, long H, long N, long d,
                         double scale, int causal, const long *rows, long n_rows,
                         int nthreads)
{
    if (!q || !k || !v || !o || !lse || (!rows && n_rows > 0)) return -1;
    if (check_shape(B, H, N, d) || n_rows < 0) return -2;
    for (long r = 0; r < n_rows; ++r)
        if (rows[r] < 0 || rows[r] >= B * H * N) return -2;
    job_t job = {q, k, v, o, lse, B, H, N, d, scale, causal, 0, rows, n_rows};
    return run_job(&job, nthreads);
}

/* Every row, by the chunked online-softmax loop with `chunk` keys per step. */
int oracle_attn_online_f64(const double *q, const double *k, const double *v,
                           double *o, double *lse, long B, long H, long N, long d,
                           double scale, int causal, long chunk, int nthreads)
{
    if (!q || !k || !v || !o || !lse) return -1;
    if (check_shape(B, H, N, d) || chunk <= 0) return -2;
    job_t job = {q, k, v, o, lse, B, H, N, d, scale, causal, chunk, NULL, B * H * N};
    return run_job(&job, nthreads);
}

/* The probability matrix P = softmax(S) of one head (q, k: [N,d]; p: [N,N]),
 * masked entries 0. Single-threaded; meant for small N. */
int oracle_attn_probs_f64(const double *q, const double *k, double *p,
                          long N, long d, double scale, int causal)
{
    if (!q || !k || !p) return -1;
    if (check_shape(1, 1, N, d)) return -2;
    for (long i = 0; i < N; ++i) {
        long n_keys = causal ? i + 1 : N;
        double *row = p + i * N;
        for (long j = 0; j < N; ++j) row[j] = 0.0;
        double m = -INFINITY;
        for (long j = 0; j < n_keys; ++j) {
            double x = 0.0;
            for (long c = 0; c < d; ++c) x += q[i * d + c] * k[j * d + c];
            row[j] = scale * x;
            if (row[j] > m) m = row[j];
        }
        double z = 0.0;
        for (long j = 0; j < n_keys; ++j) z += exp(row[j] - m);
        for (long j = 0; j < n_keys; ++j) row[j] = exp(row[j] - m) / z;
    }
    return 0;
}

/* Variable-length batch by the definition. q, o: [total_q, H, d]; k, v:
 * [total_k, H, d]; lse: [H, total_q]; cu_q, cu_k: B+1 non-decreasing offsets
 * from 0 (total_q = cu_q[B], total_k = cu_k[B]). */
int oracle_attn_varlen_f64(const double *q, const double *k, const double *v,
                           double *o, double *lse, const long *cu_q, const long *cu_k,
                           long B, long H, long d, double scale, int causal, int nthreads)
{
    if (!q || !k || !v || !o || !lse || !cu_q || !cu_k) return -1;
    if (B < 1 || H < 1 || d <= 0 || cu_q[0] != 0 || cu_k[0] != 0) return -2;
    long max_nk = 0;
    for (long b = 0; b < B; ++b) {
        if (cu_q[b + 1] < cu_q[b] || cu_k[b + 1] < cu_k[b]) return -2;
        if (cu_k[b + 1] - cu_k[b] > max_nk) max_nk = cu_k[b + 1] - cu_k[b];
    }
    vjob_t job;
    memset(&job, 0, sizeof(job));
    job.q = q; job.k = k; job.v = v; job.o = o; job.lse = lse;
    job.cu_q = cu_q; job.cu_k = cu_k;
    job.B = B; job.H = H; job.d = d; job.total_q = cu_q[B];
    job.scale = scale; job.causal = causal; job.max_nk = max_nk;
    long n_rows = H * job.total_q;
    if (n_rows == 0) return 0;
    long n = nthreads > 0 ? nthreads : host_threads();
    if (n > n_rows) n = n_rows;
    pthread_t *tids = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)n);
    if (!tids) return -3;
    pthread_mutex_init(&job.lock, NULL);
    long started = 0;
    for (long t = 0; t < n; ++t) {
        if (pthread_create(&tids[t], NULL, varlen_worker, &job) != 0) break;
        ++started;
    }
    if (started == 0) varlen_worker(&job);
    for (long t = 0; t < started; ++t) pthread_join(tids[t], NULL);
    pthread_mutex_destroy(&job.lock);
    free(tids);
    return job.failed ? -3 : 0;
}
