/*
 * kda_oracle.c -- fp64 CPU oracle for the Kimi Delta Attention (KDA) state
 * recurrence.  TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the
 * benchmark's CPU-baseline leg call it; the library's product path never
 * does.  It shares no code, header, table or helper with the CUDA path.
 *
 * What it computes (GLM-5.3-Flash Architecture Mastery, course index,
 * "Course Outcomes": the delta-rule update written as five named operations
 * and expanded to the closed form (I - beta k k^T) D S + beta k v^T; and
 * Lecture 11, section 2, KDA row of the correctness matrix: the operator
 * order is (I - beta k k^T) D, not D (I - beta k k^T)):
 *
 *     S_t = (I - beta_t k_t k_t^T) D_t S_{t-1} + beta_t k_t v_t^T
 *     o_t = S_t^T q_t,            D_t = diag(exp(g_t))
 *
 * one token at a time, in this order (the plainest reading of the "five
 * named operations"; expanding them gives exactly the closed form):
 *
 *     1. decay   S' = D_t S_{t-1}          (D_t scales the d_k rows of S)
 *     2. read    vhat = S'^T k_t
 *     3. error   delta = v_t - vhat
 *     4. write   S_t = S' + beta_t k_t delta^T
 *     5. output  o_t = S_t^T q_t          (post-update state, scale 1)
 *
 * Packed documents (Lecture 11, section 2, "Padding / packing" row): the
 * state restarts at every cu_seqlens boundary from S0[seq] (or zero), so no
 * state crosses a document boundary.
 *
 * Layouts (row-major, all fp64):
 *   q, k, g : [T, H, dk]     v : [T, H, dv]     beta : [T, H]
 *   cu_seqlens : [N + 1] int32, cu[0] = 0, non-decreasing, cu[N] = T
 *   S0, S_final : [N, H, dk, dv]  (S0 may be NULL = zero initial state)
 *   o : [T, H, dv]
 *   snap_t : [n_snap] token counts; S_snap : [n_snap, N, H, dk, dv] holds the
 *            state of every (seq, head) after snap_t[j] tokens of that
 *            sequence (entries whose count exceeds the sequence length are
 *            left untouched; a count of 0 stores the initial state).
 *
 * Chains (seq, head) are independent; they are spread over POSIX threads.
 * Each chain is computed by one thread with a fixed operation order, so the
 * result does not depend on the thread count.
 */
#include <math.h>
#include <pthread.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    const double *q, *k, *v, *g, *beta;
    const int32_t *cu_seqlens;
    int32_t num_seqs, H, dk, dv;
    const double *S0;
    double *o, *S_final;
    int32_t n_snap;
    const int32_t *snap_t;
    double *S_snap;
    int64_t next_chain; /* shared work counter */
    int32_t failed;
} oracle_job;

/* 1. decay: S' = D_t S, row i of S scaled by exp(g_t[i]). */
static void decay_rows(double *S, const double *g_t, int dk, int dv) {
    for (int i = 0; i < dk; ++i) {
        const double d = exp(g_t[i]);
        for (int j = 0; j < dv; ++j) S[(size_t)i * dv + j] *= d;
    }
}

/* 2. read: vhat = S'^T k_t. */
static void read_state(const double *S, const double *k_t, double *vhat, int dk, int dv) {
    for (int j = 0; j < dv; ++j) vhat[j] = 0.0;
    for (int i = 0; i < dk; ++i)
        for (int j = 0; j < dv; ++j) vhat[j] += S[(size_t)i * dv + j] * k_t[i];
}

/* 3. error: delta = v_t - vhat. */
static void prediction_error(const double *v_t, const double *vhat, double *delta, int dv) {
    for (int j = 0; j < dv; ++j) delta[j] = v_t[j] - vhat[j];
}

/* 4. write: S = S' + beta_t k_t delta^T. */
static void write_state(double *S, const double *k_t, double beta_t, const double *delta, int dk, int dv) {
    for (int i = 0; i < dk; ++i)
        for (int j = 0; j < dv; ++j) S[(size_t)i * dv + j] += beta_t * k_t[i] * delta[j];
}

/* 5. output: o_t = S_t^T q_t. */
static void read_output(const double *S, const double *q_t, double *o_t, int dk, int dv) {
    for (int j = 0; j < dv; ++j) o_t[j] = 0.0;
    for (int i = 0; i < dk; ++i)
        for (int j = 0; j < dv; ++j) o_t[j] += S[(size_t)i * dv + j] * q_t[i];
}

static void store_snapshots(const oracle_job *J, int32_t seq, int32_t head, int32_t count, const double *S) {
    const size_t state = (size_t)J->dk * J->dv;
    for (int32_t j = 0; j < J->n_snap; ++j) {
        if (J->snap_t[j] != count) continue;
        double *dst = J->S_snap + (((size_t)j * J->num_seqs + seq) * J->H + head) * state;
        memcpy(dst, S, state * sizeof(double));
    }
}

static int run_chain(const oracle_job *J, int32_t seq, int32_t head) {
    const int dk = J->dk, dv = J->dv, H = J->H;
    const size_t state = (size_t)dk * dv;
    double *S = (double *)malloc(state * sizeof(double));
    double *vhat = (double *)malloc((size_t)dv * sizeof(double));
    double *delta = (double *)malloc((size_t)dv * sizeof(double));
    if (!S || !vhat || !delta) {
        free(S); free(vhat); free(delta);
        return 1;
    }
    if (J->S0) memcpy(S, J->S0 + ((size_t)seq * H + head) * state, state * sizeof(double));
    else memset(S, 0, state * sizeof(double));

    const int32_t t0 = J->cu_seqlens[seq], t1 = J->cu_seqlens[seq + 1];
    if (J->n_snap) store_snapshots(J, seq, head, 0, S);
    for (int32_t t = t0; t < t1; ++t) {
        const size_t th = (size_t)t * H + head;
        const double *q_t = J->q + th * dk, *k_t = J->k + th * dk, *g_t = J->g + th * dk;
        const double *v_t = J->v + th * dv;
        double *o_t = J->o + th * dv;
        decay_rows(S, g_t, dk, dv);
        read_state(S, k_t, vhat, dk, dv);
        prediction_error(v_t, vhat, delta, dv);
        write_state(S, k_t, J->beta[th], delta, dk, dv);
        read_output(S, q_t, o_t, dk, dv);
        if (J->n_snap) store_snapshots(J, seq, head, t - t0 + 1, S);
    }
    if (J->S_final) memcpy(J->S_final + ((size_t)seq * H + head) * state, S, state * sizeof(double));
    free(S); free(vhat); free(delta);
    return 0;
}

static void *worker(void *arg) {
    oracle_job *J = (oracle_job *)arg;
    const int64_t chains = (int64_t)J->num_seqs * J->H;
    for (;;) {
        const int64_t c = __atomic_fetch_add(&J->next_chain, 1, __ATOMIC_RELAXED);
        if (c >= chains) break;
        if (run_chain(J, (int32_t)(c / J->H), (int32_t)(c % J->H)))
            __atomic_store_n(&J->failed, 1, __ATOMIC_RELAXED);
    }
    return NULL;
}

/*
 * Runs the recurrence over every (seq, head) chain.
 * Returns 0 on success, 1 on invalid arguments, 2 on allocation failure.
 */
int kda_oracle_run(const double *q, const double *k, const double *v, const double *g, const double *beta,
                   const int32_t *cu_seqlens, int32_t num_seqs, int32_t H, int32_t dk, int32_t dv,
                   const double *S0, double *o, double *S_final,
                   int32_t n_snap, const int32_t *snap_t, double *S_snap, int32_t num_threads) {
    if (num_seqs < 0 || H <= 0 || dk <= 0 || dv <= 0 || !cu_seqlens || num_threads < 0) return 1;
    if (n_snap < 0 || (n_snap > 0 && (!snap_t || !S_snap))) return 1;
    if (cu_seqlens[0] != 0) return 1;
    for (int32_t i = 0; i < num_seqs; ++i)
        if (cu_seqlens[i + 1] < cu_seqlens[i]) return 1;
    if (cu_seqlens[num_seqs] > 0 && (!q || !k || !v || !g || !beta || !o)) return 1;

    oracle_job J;
    J.q = q; J.k = k; J.v = v; J.g = g; J.beta = beta;
    J.cu_seqlens = cu_seqlens; J.num_seqs = num_seqs; J.H = H; J.dk = dk; J.dv = dv;
    J.S0 = S0; J.o = o; J.S_final = S_final;
    J.n_snap = n_snap; J.snap_t = snap_t; J.S_snap = S_snap;
    J.next_chain = 0; J.failed = 0;

    int64_t chains = (int64_t)num_seqs * H;
    int nt = num_threads > 0 ? num_threads : 1;
    if (nt > chains) nt = chains > 0 ? (int)chains : 1;
    if (nt <= 1) {
        worker(&J);
    } else {
        pthread_t *tid = (pthread_t *)malloc((size_t)nt * sizeof(pthread_t));
        if (!tid) return 2;
        int started = 0;
        for (; started < nt; ++started)
            if (pthread_create(&tid[started], NULL, worker, &J) != 0) break;
        if (started == 0) worker(&J);
        for (int i = 0; i < started; ++i) pthread_join(tid[i], NULL);
        free(tid);
    }
    return J.failed ? 2 : 0;
}
