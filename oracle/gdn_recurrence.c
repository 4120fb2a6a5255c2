/*
 * Gated Delta Rule prefill: the plain fp64 CPU definition.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the library calls this; only the tests,
 * the package smoke check and the benchmark's CPU-baseline leg load it.  It
 * shares no code with the CUDA path.
 *
 * What it computes (the Gated Delta Rule recurrence stated for the flashinfer
 * prefill kernels, "flashinfer.gdn_prefill": a chunked scan that initialises
 * the recurrent state from a full prompt; argument meanings from
 * "flashinfer.cudnn.cudnn_chunk_gated_delta_rule", Parameters):
 *
 *   for every token t of a sequence, with S the Dv x Dk state (row = value
 *   index, column = key index: the V-major layout of "flashinfer.cudnn",
 *   Linear attention):
 *       S_t = g_t * S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T
 *       o_t = scale * S_t q_t
 *
 * The product S (I - b k k^T) is evaluated as S - b (S k) k^T, which is the
 * same matrix by associativity; everything else is written out term by term.
 *
 * A "unit" is one (sequence, sab head) pair.  The caller gathers each unit's
 * rows into compact arrays (row r of unit u is input row off[u] + r), so this
 * file needs no notion of packing, head mapping or state pools.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    int64_t n_units;
    const int64_t* len;     /* [n_units] tokens per unit */
    const int64_t* off;     /* [n_units] first compact row of the unit */
    int dk, dv;
    const double* q;        /* [R, dk] */
    const double* k;        /* [R, dk] */
    const double* v;        /* [R, dv] */
    const double* g;        /* [R] or NULL (all ones) */
    const double* beta;     /* [R] or NULL (all ones) */
    double scale;
    int use_l2norm;
    double eps;
    const double* s0;       /* [n_units, dv, dk] or NULL (zero state) */
    double* out;            /* [R, dv] */
    double* s_final;        /* [n_units, dv, dk] */
    int64_t next;           /* work counter shared by the threads */
} job_t;

/* x / sqrt(sum(x^2) + eps), the L2 normalisation fused into the kernel when
 * use_qk_l2norm_in_kernel is set. */
static void l2normalise(const double* x, double* y, int n, double eps) {
    double ss = 0.0;
    for (int i = 0; i < n; ++i) ss += x[i] * x[i];
    double r = 1.0 / sqrt(ss + eps);
    for (int i = 0; i < n; ++i) y[i] = x[i] * r;
}

static void run_unit(const job_t* J, int64_t u, double* qv, double* kv, double* sk) {
    const int dk = J->dk, dv = J->dv;
    double* S = J->s_final + u * (int64_t)dv * dk;
    if (J->s0) memcpy(S, J->s0 + u * (int64_t)dv * dk, sizeof(double) * dv * dk);
    else memset(S, 0, sizeof(double) * dv * dk);

    for (int64_t r = J->off[u]; r < J->off[u] + J->len[u]; ++r) {
        const double* qt = J->q + r * dk;
        const double* kt = J->k + r * dk;
        const double* vt = J->v + r * dv;
        if (J->use_l2norm) {
            l2normalise(qt, qv, dk, J->eps);
            l2normalise(kt, kv, dk, J->eps);
        } else {
            memcpy(qv, qt, sizeof(double) * dk);
            memcpy(kv, kt, sizeof(double) * dk);
        }
        const double a = J->g ? J->g[r] : 1.0;
        const double b = J->beta ? J->beta[r] : 1.0;

        /* sk = S_{t-1} k_t */
        for (int i = 0; i < dv; ++i) {
            double acc = 0.0;
            for (int j = 0; j < dk; ++j) acc += S[i * dk + j] * kv[j];
            sk[i] = acc;
        }
        /* S_t = a (S_{t-1} - b (S_{t-1} k) k^T) + b v k^T */
        for (int i = 0; i < dv; ++i)
            for (int j = 0; j < dk; ++j)
                S[i * dk + j] = a * (S[i * dk + j] - b * sk[i] * kv[j]) + b * vt[i] * kv[j];
        /* o_t = scale S_t q_t */
        double* ot = J->out + r * dv;
        for (int i = 0; i < dv; ++i) {
            double acc = 0.0;
            for (int j = 0; j < dk; ++j) acc += S[i * dk + j] * qv[j];
            ot[i] = J->scale * acc;
        }
    }
}

static void* worker(void* arg) {
    job_t* J = (job_t*)arg;
    double* qv = (double*)malloc(sizeof(double) * J->dk);
    double* kv = (double*)malloc(sizeof(double) * J->dk);
    double* sk = (double*)malloc(sizeof(double) * J->dv);
    for (;;) {
        int64_t u = __atomic_fetch_add(&J->next, 1, __ATOMIC_RELAXED);
        if (u >= J->n_units) break;
        run_unit(J, u, qv, kv, sk);
    }
    free(qv);
    free(kv);
    free(sk);
    return NULL;
}

/* Returns 0 on success, -1 on bad arguments.  If a helper thread cannot be
 * started the remaining threads still process every unit. */
int gdn_oracle_recurrence(int64_t n_units, const int64_t* len, const int64_t* off,
                          int dk, int dv, const double* q, const double* k,
                          const double* v, const double* g, const double* beta,
                          double scale, int use_l2norm, double eps, const double* s0,
                          double* out, double* s_final, int nthreads) {
    if (n_units < 0 || dk <= 0 || dv <= 0 || !len || !off || !out || !s_final) return -1;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > n_units) nthreads = n_units > 0 ? (int)n_units : 1;
    job_t J = {n_units, len, off, dk, dv, q, k, v, g, beta, scale, use_l2norm, eps,
               s0, out, s_final, 0};
    pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * nthreads);
    int started = 0;
    for (int i = 1; i < nthreads; ++i) {
        if (pthread_create(&th[i], NULL, worker, &J) != 0) break;
        ++started;
    }
    worker(&J);
    for (int i = 1; i <= started; ++i) pthread_join(th[i], NULL);
    free(th);
    return 0;
}
