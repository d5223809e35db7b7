/*
 * gdn_ref.c -- CPU oracle for the gated delta-rule recurrence (Gated DeltaNet).
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, sequential definition
 * of what the GPU library computes.  Only the tests, the package's smoke check
 * and the benchmark's CPU-baseline leg may load it.  It shares no code, header
 * or constant with the CUDA library and includes nothing from it.
 *
 * Everything is float64.  Inputs arrive already widened from the exact values the
 * GPU sees (bf16/f16/fp32 rounded once by the input generator), so the oracle's
 * result is the recurrence's value up to float64 rounding.
 *
 * Sources (the pages it restates):
 *  - onnx-runtime-ep-cuda 0.1.0-dev.6, src/kernels/linear_attention.rs,
 *    `linear_attention_core`: the four steps per token -- Step 1 decay
 *    S *= exp(g_t); Step 2 retrieval r = S^T k_t over d_k; Step 3 delta update
 *    S += k_t (x) beta_t (v_t - r); Step 4 readout o_t = scale * q_t^T S with the
 *    UPDATED S.  Also its gate helpers `la_softplus`
 *    (max(x,0) + log1p(exp(-|x|))) and `la_sigmoid`, the fused gate chain
 *    g = -exp(A_log) * softplus(a + dt_bias), beta = sigmoid(b), the state
 *    layout [.., d_k, d_v], the GQA mapping (consecutive value heads share one
 *    key/query head) and the update rules {linear, gated, delta, gated_delta}.
 *  - onnxruntime-ep-mlx 0.31.1, src/ops/ssm.rs, `linear_attention_gate_op`:
 *    the gates are evaluated once in wide precision and never re-rounded per
 *    intermediate; and `linear_attention_op`'s zero-length time axis: no step
 *    runs and the present state equals the past state.
 *  - nuvec-core 0.6.1, src/fast/imp.rs, `gated_delta_graph`: the same four steps
 *    written with whole-array operations (a cross-check of the step order).
 *  - The CUDA page's gate variants: Step 1 with `decay_per_key_dim` (one decay per
 *    key dimension, S[i,:] *= exp(g_i), with A_log and dt_bias per (head, key dim))
 *    and a beta shared by all heads (`beta_per_head` false, beta [B, T, 1]).
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *  - `scale` multiplies the finished fp64 dot product q^T S (post-multiply).
 *  - A sequence of length 0 leaves its state unchanged; a NULL state_in is zeros.
 *  - Varlen: sequence n covers packed tokens [cu[n], cu[n+1]) and starts from
 *    state_in[n]; sequences never interact.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Update rules, numbered as in the pages' rule list. */
enum { RULE_GATED_DELTA = 0, RULE_DELTA = 1, RULE_GATED = 2, RULE_LINEAR = 3 };

/* softplus(x) = log(1 + e^x), in the overflow-free form max(x,0) + log1p(e^-|x|). */
double gdn_ref_softplus(double x) { return fmax(x, 0.0) + log1p(exp(-fabs(x))); }

/* sigmoid(x) = 1 / (1 + e^-x), split on the sign so e^(...) never overflows. */
double gdn_ref_sigmoid(double x) {
    if (x >= 0.0) return 1.0 / (1.0 + exp(-x));
    double e = exp(x);
    return e / (1.0 + e);
}

/* g = -exp(A_log) * softplus(a + dt_bias), the log-space per-token decay. */
double gdn_ref_decay(double a, double A_log, double dt_bias) {
    return -exp(A_log) * gdn_ref_softplus(a + dt_bias);
}

typedef struct {
    int64_t n_seq;
    const int64_t *cu;
    int32_t h_qk, h_v, d_k, d_v;
    const double *q, *k, *v, *a, *b, *A_log, *dt_bias, *g_in, *beta_in, *state_in;
    double scale;
    int32_t rule;
    double *o, *state_out;
    int32_t decay_per_key;   /* a / g_in [T, h_v, d_k]; A_log, dt_bias [h_v, d_k] */
    int32_t beta_shared;     /* b / beta_in [T] (one beta for every head) */
} job_t;

/* One (sequence n, value head h): the recurrence over its tokens, in order. */
static void run_unit(const job_t *J, int64_t n, int32_t h, double *S, double *r) {
    const int32_t dk = J->d_k, dv = J->d_v;
    const int32_t group = J->h_v / J->h_qk;          /* value heads per q/k head */
    const int32_t hq = h / group;                     /* consecutive heads share */
    const int has_decay = (J->rule == RULE_GATED_DELTA || J->rule == RULE_GATED);
    const int has_delta = (J->rule == RULE_GATED_DELTA || J->rule == RULE_DELTA);
    const size_t sz = (size_t)dk * dv;

    if (J->state_in)
        memcpy(S, J->state_in + ((size_t)n * J->h_v + h) * sz, sz * sizeof(double));
    else
        memset(S, 0, sz * sizeof(double));

    for (int64_t t = J->cu[n]; t < J->cu[n + 1]; ++t) {
        const double *qt = J->q + ((size_t)t * J->h_qk + hq) * dk;
        const double *kt = J->k + ((size_t)t * J->h_qk + hq) * dk;
        const double *vt = J->v + ((size_t)t * J->h_v + h) * dv;
        double *ot = J->o + ((size_t)t * J->h_v + h) * dv;
        const size_t gi = (size_t)t * J->h_v + h;
        const size_t bi = J->beta_shared ? (size_t)t : gi;
        double g = 0.0, beta;
        if (J->a) {
            if (!J->decay_per_key) g = gdn_ref_decay(J->a[gi], J->A_log[h], J->dt_bias[h]);
            beta = gdn_ref_sigmoid(J->b[bi]);
        } else {
            if (!J->decay_per_key) g = J->g_in ? J->g_in[gi] : 0.0;
            beta = J->beta_in ? J->beta_in[bi] : 1.0;
        }

        /* Step 1: decay, one factor per head or one per key dimension (row i of S). */
        if (has_decay && !J->decay_per_key) {
            const double alpha = exp(g);
            for (size_t e = 0; e < sz; ++e) S[e] *= alpha;
        } else if (has_decay) {
            for (int32_t i = 0; i < dk; ++i) {
                const size_t ki = gi * dk + i, hk = (size_t)h * dk + i;
                const double gk = J->a ? gdn_ref_decay(J->a[ki], J->A_log[hk], J->dt_bias[hk])
                                       : (J->g_in ? J->g_in[ki] : 0.0);
                const double alpha = exp(gk);
                for (int32_t j = 0; j < dv; ++j) S[(size_t)i * dv + j] *= alpha;
            }
        }
        if (has_delta) {
            /* Step 2: retrieval r_j = sum_i S_ij k_i, left to right over i. */
            for (int32_t j = 0; j < dv; ++j) r[j] = 0.0;
            for (int32_t i = 0; i < dk; ++i)
                for (int32_t j = 0; j < dv; ++j) r[j] += S[(size_t)i * dv + j] * kt[i];
            /* Step 3: delta update S_ij += k_i * beta * (v_j - r_j). */
            for (int32_t j = 0; j < dv; ++j) r[j] = beta * (vt[j] - r[j]);
            for (int32_t i = 0; i < dk; ++i)
                for (int32_t j = 0; j < dv; ++j) S[(size_t)i * dv + j] += kt[i] * r[j];
        } else {
            /* linear / gated rules: S_ij += k_i v_j. */
            for (int32_t i = 0; i < dk; ++i)
                for (int32_t j = 0; j < dv; ++j) S[(size_t)i * dv + j] += kt[i] * vt[j];
        }
        /* Step 4: readout with the updated state, o_j = scale * sum_i q_i S_ij. */
        for (int32_t j = 0; j < dv; ++j) r[j] = 0.0;
        for (int32_t i = 0; i < dk; ++i)
            for (int32_t j = 0; j < dv; ++j) r[j] += qt[i] * S[(size_t)i * dv + j];
        for (int32_t j = 0; j < dv; ++j) ot[j] = J->scale * r[j];
    }
    memcpy(J->state_out + ((size_t)n * J->h_v + h) * sz, S, sz * sizeof(double));
}

typedef struct {
    const job_t *J;
    int64_t first, stride, units;
    const int64_t *unit_list;   /* optional subset of units (n * h_v + h) */
    int rc;
} worker_t;

static void *worker(void *arg) {
    worker_t *W = (worker_t *)arg;
    const job_t *J = W->J;
    double *S = (double *)malloc((size_t)J->d_k * J->d_v * sizeof(double));
    double *r = (double *)malloc((size_t)J->d_v * sizeof(double));
    if (!S || !r) { W->rc = -2; free(S); free(r); return NULL; }
    for (int64_t u = W->first; u < W->units; u += W->stride) {
        const int64_t id = W->unit_list ? W->unit_list[u] : u;
        run_unit(J, id / J->h_v, (int32_t)(id % J->h_v), S, r);
    }
    free(S);
    free(r);
    return NULL;
}

/*
 * gdn_ref_scan_ex: the recurrence for every (sequence, value head), or for the
 * listed subset of them.
 *
 *   cu         [n_seq+1] token offsets of each sequence in the packed axis
 *   q, k       [T_total, h_qk, d_k]
 *   v          [T_total, h_v, d_v]
 *   a, b       [T_total, h_v] raw gate logits; if a == NULL the gates come from
 *              g_in (log-space decay, NULL = 0) and beta_in (NULL = 1)
 *   A_log, dt_bias [h_v]
 *   state_in   [n_seq, h_v, d_k, d_v] or NULL (zeros)
 *   rule       0 gated_delta, 1 delta, 2 gated, 3 linear
 *   decay_per_key  a (or g_in) is [T_total, h_v, d_k] and A_log, dt_bias are
 *              [h_v, d_k]: row i of S decays by its own factor
 *   beta_shared    b (or beta_in) is [T_total]: one beta for every head
 *   units      NULL for all n_seq*h_v units, else n_units ids (n*h_v + h);
 *              only those units' o rows and states are written
 *   o          [T_total, h_v, d_v];  state_out [n_seq, h_v, d_k, d_v]
 * Returns 0, or a negative code for bad arguments / allocation failure.
 */
int gdn_ref_scan_ex(int64_t n_seq, const int64_t *cu, int32_t h_qk, int32_t h_v,
                    int32_t d_k, int32_t d_v, const double *q, const double *k,
                    const double *v, const double *a, const double *b,
                    const double *A_log, const double *dt_bias, const double *g_in,
                    const double *beta_in, const double *state_in, double scale,
                    int32_t rule, int32_t decay_per_key, int32_t beta_shared,
                    const int64_t *units, int64_t n_units, int32_t n_threads, double *o,
                    double *state_out) {
    if (n_seq < 0 || !cu || h_qk <= 0 || h_v <= 0 || h_v % h_qk != 0 || d_k <= 0 ||
        d_v <= 0 || rule < 0 || rule > 3 || !o || !state_out)
        return -1;
    if (a && (!b || !A_log || !dt_bias)) return -1;
    for (int64_t n = 0; n < n_seq; ++n)
        if (cu[n + 1] < cu[n]) return -1;
    job_t J = {n_seq, cu, h_qk, h_v, d_k, d_v, q, k, v, a, b, A_log, dt_bias,
               g_in, beta_in, state_in, scale, rule, o, state_out, decay_per_key != 0,
               beta_shared != 0};
    const int64_t total = units ? n_units : n_seq * (int64_t)h_v;
    if (n_threads < 1) n_threads = 1;
    if (n_threads > 256) n_threads = 256;
    if ((int64_t)n_threads > total) n_threads = total > 0 ? (int32_t)total : 1;
    worker_t W[256];
    pthread_t th[256];
    for (int32_t i = 0; i < n_threads; ++i) {
        W[i].J = &J; W[i].first = i; W[i].stride = n_threads;
        W[i].units = total; W[i].unit_list = units; W[i].rc = 0;
    }
    int rc = 0;
    if (n_threads == 1) {
        worker(&W[0]);
    } else {
        int32_t started = 0;
        for (; started < n_threads; ++started)
            if (pthread_create(&th[started], NULL, worker, &W[started]) != 0) break;
        for (int32_t i = started; i < n_threads; ++i) worker(&W[i]);
        for (int32_t i = 0; i < started; ++i) pthread_join(th[i], NULL);
    }
    for (int32_t i = 0; i < n_threads; ++i)
        if (W[i].rc) rc = W[i].rc;
    return rc;
}

/* gdn_ref_scan_ex with one decay and one beta per (token, head). */
int gdn_ref_scan(int64_t n_seq, const int64_t *cu, int32_t h_qk, int32_t h_v,
                 int32_t d_k, int32_t d_v, const double *q, const double *k,
                 const double *v, const double *a, const double *b,
                 const double *A_log, const double *dt_bias, const double *g_in,
                 const double *beta_in, const double *state_in, double scale,
                 int32_t rule, const int64_t *units, int64_t n_units,
                 int32_t n_threads, double *o, double *state_out) {
    return gdn_ref_scan_ex(n_seq, cu, h_qk, h_v, d_k, d_v, q, k, v, a, b, A_log, dt_bias, g_in,
                           beta_in, state_in, scale, rule, 0, 0, units, n_units, n_threads, o,
                           state_out);
}
