/*
 * kda_scan.c — the oracle's token-by-token Kimi Delta Attention scan, in fp64.
 *
 * TEST INFRASTRUCTURE. Only tests/, __graft_entry__.smoke() and bench.py's
 * CPU-baseline leg may load this file's library. The product path (the CUDA
 * library and its Python binding) never calls it and shares no code with it.
 *
 * What it computes is the plain definition of the method, one token at a time,
 * per (sequence, head), with the state S of shape d_k x d_v (row c = key
 * channel c):
 *
 *   a_t      = exp(g_t)                       per key channel, g_t <= 0
 *   S~_t     = Diag(a_t) S_{t-1}              decay first ...
 *   e_t      = beta_t (v_t - S~_t^T k_t)      ... then predict against the
 *                                              decayed state and take the error
 *   S_t      = S~_t + k_t e_t^T               rank-one corrective write
 *   o_t      = S_t^T (scale * q_t)            read with the scaled query
 *
 * Sources:
 *   "Understanding Kimi Delta Attention", box "KDA: Retain, predict, correct"
 *     (decay, prediction against the decayed state, corrective write) and the
 *     paragraph after Figure 02 (why decay comes before the prediction);
 *   "Understanding Kimi Delta Attention", box "A fixed-size associative
 *     memory" (the read o_t = S_t^T q_t);
 *   "Demystifying Kimi Delta Attention", the opening KDA update equations
 *     (the query is multiplied by d_k^{-1/2}; that page stores the transpose
 *     of S, the same map).
 *
 * Layouts (all row-major, fp64):
 *   q, k, g   [T_total][H][d_k]      v, out [T_total][H][d_v]
 *   beta      [T_total][H]
 *   init_state, final_state [num_seqs][H][d_k][d_v]   (init may be NULL = 0)
 *   cu_seqlens int64 [num_seqs + 1]: sequence n spans tokens
 *              [cu_seqlens[n], cu_seqlens[n+1]).
 *
 * Work is split over (sequence, head) pairs, which are independent, across
 * nthreads POSIX threads. The arithmetic inside a pair is strictly sequential
 * in token order.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

typedef struct {
    const double *q, *k, *v, *g, *beta;
    double scale;
    const double *init_state;
    const int64_t *cu_seqlens;
    int num_seqs, H, dk, dv;
    double *out, *final_state;
    int next_item; /* shared work counter */
    int error;
} scan_job;

static void scan_one(const scan_job *J, int item, double *S, double *vhat, double *e) {
    const int n = item / J->H, h = item % J->H;
    const int H = J->H, dk = J->dk, dv = J->dv;
    const size_t state_off = ((size_t)n * H + h) * (size_t)dk * dv;

    if (J->init_state)
        memcpy(S, J->init_state + state_off, sizeof(double) * (size_t)dk * dv);
    else
        memset(S, 0, sizeof(double) * (size_t)dk * dv);

    for (int64_t t = J->cu_seqlens[n]; t < J->cu_seqlens[n + 1]; ++t) {
        const double *qt = J->q + ((size_t)t * H + h) * dk;
        const double *kt = J->k + ((size_t)t * H + h) * dk;
        const double *gt = J->g + ((size_t)t * H + h) * dk;
        const double *vt = J->v + ((size_t)t * H + h) * dv;
        const double bt = J->beta[(size_t)t * H + h];
        double *ot = J->out + ((size_t)t * H + h) * dv;

        /* S~ = Diag(exp(g_t)) S: row c of the state is scaled by a_t[c]. */
        for (int c = 0; c < dk; ++c) {
            const double a = exp(gt[c]);
            for (int j = 0; j < dv; ++j) S[(size_t)c * dv + j] *= a;
        }
        /* vhat = S~^T k_t; e = beta (v - vhat). */
        for (int j = 0; j < dv; ++j) vhat[j] = 0.0;
        for (int c = 0; c < dk; ++c)
            for (int j = 0; j < dv; ++j) vhat[j] += S[(size_t)c * dv + j] * kt[c];
        for (int j = 0; j < dv; ++j) e[j] = bt * (vt[j] - vhat[j]);
        /* S = S~ + k_t e^T. */
        for (int c = 0; c < dk; ++c)
            for (int j = 0; j < dv; ++j) S[(size_t)c * dv + j] += kt[c] * e[j];
        /* o_t = S^T (scale q_t). */
        for (int j = 0; j < dv; ++j) {
            double acc = 0.0;
            for (int c = 0; c < dk; ++c) acc += S[(size_t)c * dv + j] * (J->scale * qt[c]);
            ot[j] = acc;
        }
    }
    if (J->final_state) memcpy(J->final_state + state_off, S, sizeof(double) * (size_t)dk * dv);
}

static void *scan_worker(void *arg) {
    scan_job *J = (scan_job *)arg;
    double *S = (double *)malloc(sizeof(double) * (size_t)J->dk * J->dv);
    double *vhat = (double *)malloc(sizeof(double) * (size_t)J->dv);
    double *e = (double *)malloc(sizeof(double) * (size_t)J->dv);
    if (!S || !vhat || !e) {
        __atomic_store_n(&J->error, 1, __ATOMIC_SEQ_CST);
    } else {
        const int items = J->num_seqs * J->H;
        for (;;) {
            const int it = __atomic_fetch_add(&J->next_item, 1, __ATOMIC_RELAXED);
            if (it >= items) break;
            scan_one(J, it, S, vhat, e);
        }
    }
    free(S);
    free(vhat);
    free(e);
    return NULL;
}

/* Number of hardware threads the host reports (the default pool size). */
int kda_oracle_hw_threads(void) {
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    return n > 0 ? (int)n : 1;
}

/*
 * Runs the scan. Returns 0 on success, -1 on bad arguments, -2 on allocation
 * failure. nthreads <= 0 means one thread per online processor; the count is
 * capped at the number of (sequence, head) pairs.
 */
int kda_oracle_scan(const double *q, const double *k, const double *v, const double *g,
                    const double *beta, double scale, const double *init_state,
                    const int64_t *cu_seqlens, int num_seqs, int H, int dk, int dv,
                    double *out, double *final_state, int nthreads) {
    if (!q || !k || !v || !g || !beta || !cu_seqlens || !out) return -1;
    if (num_seqs < 0 || H <= 0 || dk <= 0 || dv <= 0) return -1;
    for (int n = 0; n < num_seqs; ++n)
        if (cu_seqlens[n + 1] < cu_seqlens[n]) return -1;

    scan_job J;
    J.q = q; J.k = k; J.v = v; J.g = g; J.beta = beta; J.scale = scale;
    J.init_state = init_state; J.cu_seqlens = cu_seqlens;
    J.num_seqs = num_seqs; J.H = H; J.dk = dk; J.dv = dv;
    J.out = out; J.final_state = final_state;
    J.next_item = 0; J.error = 0;

    const int items = num_seqs * H;
    if (nthreads <= 0) nthreads = kda_oracle_hw_threads();
    if (nthreads > items) nthreads = items;
    if (nthreads <= 1) {
        scan_worker(&J);
        return J.error ? -2 : 0;
    }
    pthread_t *tid = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
    if (!tid) return -2;
    int started = 0;
    for (int i = 0; i < nthreads; ++i) {
        if (pthread_create(&tid[i], NULL, scan_worker, &J) != 0) break;
        ++started;
    }
    if (started == 0) scan_worker(&J);
    for (int i = 0; i < started; ++i) pthread_join(tid[i], NULL);
    free(tid);
    return J.error ? -2 : 0;
}
