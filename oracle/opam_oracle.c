/*
 * opam_oracle.c -- float64 CPU oracle for the outer-product associative-memory
 * layers (Tensor Cache, DeltaNet delta rule, BDH-style additive linear
 * attention).
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, obviously correct
 * statement of what the layers compute: one plain loop over tokens per
 * (batch, head) unit, in float64, in the order the pages give the steps.  It
 * shares no code, header, table or helper with the CUDA library; the only
 * callers are the test-suite, the package smoke check and the CPU-baseline leg
 * of the benchmark.  No product code path may call it.
 *
 * Parallelism: units (batch x head, or sequence x head for decode) are
 * independent, so they are spread over OpenMP threads.  Inside a unit nothing
 * is blocked, fused or reordered.
 *
 * State orientation: every state is stored key-major, element (a, b) of the
 * d_k x d_v matrix at [a * d_v + b].  For Tensor Cache this is A itself
 * (A = sum of k (x) v = k v^T).  DeltaNet and BDH write their state as
 * S in R^{d_v x d_k} with read S q; S is the transpose of that matrix, so
 * S_{i,j} sits at [j * d_v + i].
 *
 * Parity status: every function here is pinned by the CPU test-suite
 * (tests/test_oracle_*.py) against hand-derived fixtures, closed forms,
 * library routines, invariants or brute force; see the header of each test.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

void oracle_set_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

int oracle_get_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

static double logistic(double x) { return 1.0 / (1.0 + exp(-x)); }

/* ======================================================================
 * Tensor Cache (gist.science 2605.22884, "Tensor Cache: Eviction-conditioned
 * Associative Memory for Transformers", Methodology 1: two-level
 * architecture).
 *
 *  - L1 is a fixed-size KV ring buffer of the most recent W tokens; queries
 *    take exact softmax attention over it.
 *  - When the ring overwrites an entry, the displaced (k, v) is written into
 *    the fixed-size outer-product matrix A:  A <- lambda A + eta (k (x) v),
 *    with lambda (decay) and eta (write rate) learned per head.
 *  - A query reads the compressed past as r_t = m_t = q_t A, which by
 *    q (k (x) v) = <q, k> v retrieves every evicted token at once.
 *  - A learned scalar gate g fuses the two: y_t = y_local + sigmoid(g) m_t.
 *
 * Readings where the page is silent (each listed in the design notes):
 *  the window holds W tokens including the current one (its KV is inserted
 *  before it attends); the eviction write happens before the read of the same
 *  step; the softmax scale is a parameter (1/sqrt(d_k) by default); lambda,
 *  eta and g are one scalar per head; sigmoid is the logistic function.
 * ====================================================================== */

typedef struct {
    int W, dk, dv;
    double *ring_k;     /* [W][dk], slot = position mod W                  */
    double *ring_v;     /* [W][dv]                                         */
    int64_t *ring_tok;  /* [W] token position held by each slot, -1 empty  */
    double *A;          /* [dk][dv] L2 matrix                              */
    double lam, eta, gate, scale;
    double *score;      /* [W] scratch                                     */
} tc_unit;

/* One streaming step for token position t: ring insert (with eviction write
 * into A when a slot is overwritten), softmax over the ring, L2 read, gate. */
static void tc_step(tc_unit *u, int64_t t, const double *q, const double *k,
                    const double *v, double *y, double *m_out,
                    int *write_count, int64_t *write_time)
{
    const int W = u->W, dk = u->dk, dv = u->dv;
    const int slot = (int)(t % W);

    /* Eviction: the slot's previous (k, v) is written into A before the
     * slot is reused. */
    if (u->ring_tok[slot] >= 0) {
        const int64_t e = u->ring_tok[slot];
        const double *ke = u->ring_k + (size_t)slot * dk;
        const double *ve = u->ring_v + (size_t)slot * dv;
        for (int a = 0; a < dk; ++a)
            for (int b = 0; b < dv; ++b)
                u->A[(size_t)a * dv + b] = u->lam * u->A[(size_t)a * dv + b]
                                         + u->eta * ke[a] * ve[b];
        if (write_count) write_count[e] += 1;
        if (write_time) write_time[e] = t;
    }
    memcpy(u->ring_k + (size_t)slot * dk, k, sizeof(double) * dk);
    memcpy(u->ring_v + (size_t)slot * dv, v, sizeof(double) * dv);
    u->ring_tok[slot] = t;

    /* L1: exact softmax over every occupied slot (max-subtracted, two pass). */
    double mx = -INFINITY;
    for (int j = 0; j < W; ++j) {
        if (u->ring_tok[j] < 0) continue;
        double s = 0.0;
        for (int a = 0; a < dk; ++a) s += q[a] * u->ring_k[(size_t)j * dk + a];
        s *= u->scale;
        u->score[j] = s;
        if (s > mx) mx = s;
    }
    double z = 0.0;
    for (int b = 0; b < dv; ++b) y[b] = 0.0;
    for (int j = 0; j < W; ++j) {
        if (u->ring_tok[j] < 0) continue;
        const double p = exp(u->score[j] - mx);
        z += p;
        for (int b = 0; b < dv; ++b) y[b] += p * u->ring_v[(size_t)j * dv + b];
    }
    for (int b = 0; b < dv; ++b) y[b] /= z;

    /* L2 read m = q A, then the gated fuse. */
    const double sg = logistic(u->gate);
    for (int b = 0; b < dv; ++b) {
        double m = 0.0;
        for (int a = 0; a < dk; ++a) m += q[a] * u->A[(size_t)a * dv + b];
        if (m_out) m_out[b] = m;
        y[b] += sg * m;
    }
}

static int tc_unit_alloc(tc_unit *u, int W, int dk, int dv)
{
    u->W = W; u->dk = dk; u->dv = dv;
    u->ring_k = (double *)calloc((size_t)W * dk, sizeof(double));
    u->ring_v = (double *)calloc((size_t)W * dv, sizeof(double));
    u->ring_tok = (int64_t *)malloc(sizeof(int64_t) * (size_t)W);
    u->A = (double *)calloc((size_t)dk * dv, sizeof(double));
    u->score = (double *)malloc(sizeof(double) * (size_t)W);
    if (!u->ring_k || !u->ring_v || !u->ring_tok || !u->A || !u->score) return -1;
    for (int j = 0; j < W; ++j) u->ring_tok[j] = -1;
    return 0;
}

static void tc_unit_free(tc_unit *u)
{
    free(u->ring_k); free(u->ring_v); free(u->ring_tok); free(u->A); free(u->score);
}

/* Prefill from an empty state: tokens 0..T-1 through tc_step.
 * q,k: [B][H][T][dk]; v: [B][H][T][dv]; lam, eta, gate: [H].
 * y: [B][H][T][dv].  Optional outputs (NULL to skip): m_out [B][H][T][dv]
 * (the L2 read alone), the final state ring_k [B][H][W][dk],
 * ring_v [B][H][W][dv], A [B][H][dk][dv] (empty ring slots are zero), and
 * write_count / write_time [B][H][T] (how often, and at which step, each
 * token was written into A). Returns 0, or -1 on allocation failure. */
int oracle_tc_prefill(int B, int H, int T, int dk, int dv, int W,
                      const double *q, const double *k, const double *v,
                      const double *lam, const double *eta, const double *gate,
                      double scale, double *y, double *m_out,
                      double *ring_k_out, double *ring_v_out, double *A_out,
                      int *write_count, int64_t *write_time)
{
    int err = 0;
    const int units = B * H;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : err)
    for (int bh = 0; bh < units; ++bh) {
        const int h = bh % H;
        tc_unit u;
        if (tc_unit_alloc(&u, W, dk, dv)) { err |= 1; tc_unit_free(&u); continue; }
        u.lam = lam[h]; u.eta = eta[h]; u.gate = gate[h]; u.scale = scale;
        int *wc = write_count ? write_count + (size_t)bh * T : NULL;
        int64_t *wt = write_time ? write_time + (size_t)bh * T : NULL;
        if (wc) for (int t = 0; t < T; ++t) wc[t] = 0;
        if (wt) for (int t = 0; t < T; ++t) wt[t] = -1;
        for (int t = 0; t < T; ++t) {
            const size_t ik = ((size_t)bh * T + t) * dk, iv = ((size_t)bh * T + t) * dv;
            tc_step(&u, t, q + ik, k + ik, v + iv, y + iv, m_out ? m_out + iv : NULL, wc, wt);
        }
        if (ring_k_out) memcpy(ring_k_out + (size_t)bh * W * dk, u.ring_k, sizeof(double) * (size_t)W * dk);
        if (ring_v_out) memcpy(ring_v_out + (size_t)bh * W * dv, u.ring_v, sizeof(double) * (size_t)W * dv);
        if (A_out) memcpy(A_out + (size_t)bh * dk * dv, u.A, sizeof(double) * (size_t)dk * dv);
        tc_unit_free(&u);
    }
    return err ? -1 : 0;
}

/* Streaming decode continuing from an exported state (Methodology 1: the
 * same ring-buffer / eviction / read / fuse step, one token at a time).
 * State (in/out): ring_k [S][H][W][dk], ring_v [S][H][W][dv],
 * A [S][H][dk][dv], pos [S] (tokens seen; slot j holds the latest token
 * position p < pos with p mod W == j, and is empty when pos <= j).
 * Inputs q,k: [steps][S][H][dk]; v: [steps][S][H][dv]. y: [steps][S][H][dv]. */
int oracle_tc_decode(int S, int H, int dk, int dv, int W, int steps,
                     double *ring_k, double *ring_v, double *A, int64_t *pos,
                     const double *q, const double *k, const double *v,
                     const double *lam, const double *eta, const double *gate,
                     double scale, double *y)
{
    int err = 0;
    const int units = S * H;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : err)
    for (int sh = 0; sh < units; ++sh) {
        const int s = sh / H, h = sh % H;
        tc_unit u;
        if (tc_unit_alloc(&u, W, dk, dv)) { err |= 1; tc_unit_free(&u); continue; }
        u.lam = lam[h]; u.eta = eta[h]; u.gate = gate[h]; u.scale = scale;
        memcpy(u.ring_k, ring_k + (size_t)sh * W * dk, sizeof(double) * (size_t)W * dk);
        memcpy(u.ring_v, ring_v + (size_t)sh * W * dv, sizeof(double) * (size_t)W * dv);
        memcpy(u.A, A + (size_t)sh * dk * dv, sizeof(double) * (size_t)dk * dv);
        const int64_t p0 = pos[s];
        for (int j = 0; j < W; ++j) {
            /* latest position below p0 congruent to j mod W */
            if (p0 <= j) { u.ring_tok[j] = -1; continue; }
            u.ring_tok[j] = j + ((p0 - 1 - j) / W) * (int64_t)W;
        }
        for (int st = 0; st < steps; ++st) {
            const size_t ik = ((size_t)st * units + sh) * dk, iv = ((size_t)st * units + sh) * dv;
            tc_step(&u, p0 + st, q + ik, k + ik, v + iv, y + iv, NULL, NULL, NULL);
        }
        memcpy(ring_k + (size_t)sh * W * dk, u.ring_k, sizeof(double) * (size_t)W * dk);
        memcpy(ring_v + (size_t)sh * W * dv, u.ring_v, sizeof(double) * (size_t)W * dv);
        memcpy(A + (size_t)sh * dk * dv, u.A, sizeof(double) * (size_t)dk * dv);
        tc_unit_free(&u);
    }
    if (!err)
        for (int s = 0; s < S; ++s) pos[s] += steps;
    return err ? -1 : 0;
}

/* Closed form of the Tensor Cache output for selected positions of one unit,
 * written straight from the definitions: the softmax runs over the W most
 * recent positions max(0, t-W+1)..t, and A after step t holds every token
 * s <= t-W, written at step s+W and decayed once per later write, so
 *   m_t = sum_{s <= t-W} eta * lambda^(t-W-s) <q_t, k_s> v_s.
 * q,k: [T][dk]; v: [T][dv]; ts: [n] positions; y: [n][dv]. */
void oracle_tc_output_at(int T, int dk, int dv, int W,
                         const double *q, const double *k, const double *v,
                         double lam, double eta, double gate, double scale,
                         int n, const int64_t *ts, double *y)
{
    (void)T;
#pragma omp parallel for schedule(dynamic, 1)
    for (int i = 0; i < n; ++i) {
        const int64_t t = ts[i];
        const double *qt = q + (size_t)t * dk;
        double *yt = y + (size_t)i * dv;
        const int64_t s0 = t - W + 1 > 0 ? t - W + 1 : 0;
        double mx = -INFINITY;
        for (int64_t s = s0; s <= t; ++s) {
            double d = 0.0;
            for (int a = 0; a < dk; ++a) d += qt[a] * k[(size_t)s * dk + a];
            d *= scale;
            if (d > mx) mx = d;
        }
        double z = 0.0;
        for (int b = 0; b < dv; ++b) yt[b] = 0.0;
        for (int64_t s = s0; s <= t; ++s) {
            double d = 0.0;
            for (int a = 0; a < dk; ++a) d += qt[a] * k[(size_t)s * dk + a];
            const double p = exp(d * scale - mx);
            z += p;
            for (int b = 0; b < dv; ++b) yt[b] += p * v[(size_t)s * dv + b];
        }
        for (int b = 0; b < dv; ++b) yt[b] /= z;
        const double sg = logistic(gate);
        for (int64_t s = 0; s <= t - W; ++s) {
            double d = 0.0;
            for (int a = 0; a < dk; ++a) d += qt[a] * k[(size_t)s * dk + a];
            const double w = sg * eta * pow(lam, (double)(t - W - s)) * d;
            for (int b = 0; b < dv; ++b) yt[b] += w * v[(size_t)s * dv + b];
        }
    }
}

/* ======================================================================
 * DeltaNet delta rule (molayo1419.me, "DeltaNet-family linear attention
 * variants", section "DeltaNet: write the prediction error instead of the
 * value"): read the current prediction S_{t-1} k_t, write only the
 * difference,
 *     e_t = beta_t (v_t - S_{t-1} k_t),   S_t = S_{t-1} + e_t k_t^T,
 * with beta_t in [0, 1].  The read is o_t = S_t q_t, taken after the write of
 * the same step (the page's "read again right after writing").  No decay, no
 * normaliser, no query scaling.
 * q,k: [B][H][T][dk]; v: [B][H][T][dv]; beta: [B][H][T];
 * S0 / S_out: [B][H][dk][dv] key-major (NULL: zero start / no export);
 * y: [B][H][T][dv].
 * ====================================================================== */
int oracle_delta(int B, int H, int T, int dk, int dv,
                 const double *q, const double *k, const double *v,
                 const double *beta, const double *S0, double *S_out, double *y)
{
    int err = 0;
    const int units = B * H;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : err)
    for (int bh = 0; bh < units; ++bh) {
        double *ST = (double *)calloc((size_t)dk * dv, sizeof(double)); /* S_{i,j} at [j*dv+i] */
        double *e = (double *)malloc(sizeof(double) * (size_t)dv);
        if (!ST || !e) { err |= 1; free(ST); free(e); continue; }
        if (S0) memcpy(ST, S0 + (size_t)bh * dk * dv, sizeof(double) * (size_t)dk * dv);
        for (int t = 0; t < T; ++t) {
            const double *qt = q + ((size_t)bh * T + t) * dk;
            const double *kt = k + ((size_t)bh * T + t) * dk;
            const double *vt = v + ((size_t)bh * T + t) * dv;
            const double bt = beta[(size_t)bh * T + t];
            for (int i = 0; i < dv; ++i) {            /* e = beta (v - S k) */
                double pred = 0.0;
                for (int j = 0; j < dk; ++j) pred += ST[(size_t)j * dv + i] * kt[j];
                e[i] = bt * (vt[i] - pred);
            }
            for (int j = 0; j < dk; ++j)              /* S += e k^T */
                for (int i = 0; i < dv; ++i) ST[(size_t)j * dv + i] += e[i] * kt[j];
            double *yt = y + ((size_t)bh * T + t) * dv;
            for (int i = 0; i < dv; ++i) {            /* o = S q */
                double o = 0.0;
                for (int j = 0; j < dk; ++j) o += ST[(size_t)j * dv + i] * qt[j];
                yt[i] = o;
            }
        }
        if (S_out) memcpy(S_out + (size_t)bh * dk * dv, ST, sizeof(double) * (size_t)dk * dv);
        free(ST); free(e);
    }
    return err ? -1 : 0;
}

/* ======================================================================
 * BDH-style linear attention over wide, sparse, non-negative keys
 * (ainews.random.gg, BDH memory architecture post: keys and queries are
 * neuron activations in a very high-dimensional space, the state is the
 * accumulated connectivity and a read is propagation through it; it behaves
 * like a fixed-size hash table that sparse keys write a few buckets of).  The
 * write is the classical Hebbian outer-product sum (mo.ai.kr, "Hebbian memory
 * MLP", simple MLP construction: W = sum_i v_i k_i^T), applied per token:
 *     S_t = S_{t-1} + v_t k_t^T,     o_t = S_t q_t  (read after write).
 * No decay and no normaliser.  Everything is dense here: the oracle does no
 * sparse bookkeeping at all.
 * q,k: [B][H][T][N]; v: [B][H][T][dv]; S0 / S_out: [B][H][N][dv] key-major
 * (NULL allowed); y: [B][H][T][dv].
 * ====================================================================== */
int oracle_sparse_linattn(int B, int H, int T, int N, int dv,
                          const double *q, const double *k, const double *v,
                          const double *S0, double *S_out, double *y)
{
    int err = 0;
    const int units = B * H;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : err)
    for (int bh = 0; bh < units; ++bh) {
        double *ST = (double *)calloc((size_t)N * dv, sizeof(double));
        if (!ST) { err |= 1; continue; }
        if (S0) memcpy(ST, S0 + (size_t)bh * N * dv, sizeof(double) * (size_t)N * dv);
        for (int t = 0; t < T; ++t) {
            const double *qt = q + ((size_t)bh * T + t) * N;
            const double *kt = k + ((size_t)bh * T + t) * N;
            const double *vt = v + ((size_t)bh * T + t) * dv;
            for (int j = 0; j < N; ++j)               /* S += v k^T */
                for (int i = 0; i < dv; ++i) ST[(size_t)j * dv + i] += vt[i] * kt[j];
            double *yt = y + ((size_t)bh * T + t) * dv;
            for (int i = 0; i < dv; ++i) yt[i] = 0.0;
            for (int j = 0; j < N; ++j)               /* o = S q */
                for (int i = 0; i < dv; ++i) yt[i] += ST[(size_t)j * dv + i] * qt[j];
        }
        if (S_out) memcpy(S_out + (size_t)bh * N * dv, ST, sizeof(double) * (size_t)N * dv);
        free(ST);
    }
    return err ? -1 : 0;
}

/* Closed form of the additive read for selected positions of one unit:
 * unrolling S_t = S_0 + sum_{s<=t} v_s k_s^T gives
 *     o_t = S_0 q_t + sum_{s <= t} <k_s, q_t> v_s.
 * q,k: [T][N]; v: [T][dv]; S0: [N][dv] or NULL; ts: [n]; y: [n][dv]. */
void oracle_sparse_linattn_output_at(int T, int N, int dv,
                                     const double *q, const double *k, const double *v,
                                     const double *S0, int n, const int64_t *ts, double *y)
{
    (void)T;
#pragma omp parallel for schedule(dynamic, 1)
    for (int i = 0; i < n; ++i) {
        const int64_t t = ts[i];
        const double *qt = q + (size_t)t * N;
        double *yt = y + (size_t)i * dv;
        for (int b = 0; b < dv; ++b) yt[b] = 0.0;
        if (S0)
            for (int j = 0; j < N; ++j)
                for (int b = 0; b < dv; ++b) yt[b] += S0[(size_t)j * dv + b] * qt[j];
        for (int64_t s = 0; s <= t; ++s) {
            double d = 0.0;
            for (int j = 0; j < N; ++j) d += k[(size_t)s * N + j] * qt[j];
            for (int b = 0; b < dv; ++b) yt[b] += d * v[(size_t)s * dv + b];
        }
    }
}

/* ======================================================================
 * Backward passes (gradients of a scalar loss through the layers above).
 *
 * The Tensor Cache page presents the parallel weighted-sum scan as what makes
 * the layer trainable without chunk averaging (Methodology 2; Main
 * contributions); training needs the gradient of the layer.  The pages print
 * no backward formulas, so the definition used here is the plain one: the
 * derivative of L = sum_t <dy_t, y_t> with respect to every input, for a
 * given upstream gradient dy.  Each function below is reverse-mode
 * differentiation of the per-token recurrence above, written step by step:
 * the forward recurrence is run first and its states kept, then the steps
 * are undone in reverse order, each forward operation contributing its
 * partial derivatives.  Nothing is blocked or fused.
 * ====================================================================== */

/* Tensor Cache layer backward from an empty state.  Forward step t (see
 * tc_step): (c) if t >= W the token e = t-W is written,
 * A_t = lambda A_{t-1} + eta k_e v_e^T; the new token enters the ring;
 * (b) y_loc = sum_s p_s v_s over s in [max(0,t-W+1), t], p = softmax_s of
 * scale <q_t, k_s>; (a) m_t = q_t A_t, y_t = y_loc + sigmoid(g) m_t.
 * Reverse step t, with dA the gradient with respect to A_t:
 *   (a) dg += sigmoid'(g) <dy_t, m_t>; dm = sigmoid(g) dy_t;
 *       dq_t += A_t dm; dA += q_t dm^T
 *   (b) dv_s += p_s dy_t; dp_s = <dy_t, v_s>; D = sum_s p_s dp_s;
 *       ds_s = p_s (dp_s - D); dq_t += scale sum_s ds_s k_s;
 *       dk_s += scale ds_s q_t
 *   (c) if t >= W: dlambda += <dA, A_{t-1}>; deta += k_e^T dA v_e;
 *       dk_e += eta dA v_e; dv_e += eta dA^T k_e; then dA <- lambda dA
 *       (the gradient with respect to A_{t-1}).
 * q,k: [B][H][T][dk]; v, dy: [B][H][T][dv]; lam, eta, gate: [H].
 * Outputs dq, dk: [B][H][T][dk]; dv: [B][H][T][dv]; dlam, deta, dgate: [H]
 * (summed over the batch).  Returns 0, or -1 on allocation failure. */
int oracle_tc_backward(int B, int H, int T, int dk, int dv, int W,
                       const double *q, const double *k, const double *v,
                       const double *lam, const double *eta, const double *gate,
                       double scale, const double *dy,
                       double *dq, double *dk_out, double *dv_out,
                       double *dlam, double *deta, double *dgate)
{
    int err = 0;
    const int units = B * H;
    double *gl = (double *)calloc((size_t)units * 3, sizeof(double)); /* per-unit scalar grads */
    if (!gl) return -1;
    memset(dq, 0, sizeof(double) * (size_t)units * T * dk);
    memset(dk_out, 0, sizeof(double) * (size_t)units * T * dk);
    memset(dv_out, 0, sizeof(double) * (size_t)units * T * dv);
#pragma omp parallel for schedule(dynamic, 1) reduction(| : err)
    for (int bh = 0; bh < units; ++bh) {
        const int h = bh % H;
        const double lm = lam[h], et = eta[h], sg = logistic(gate[h]);
        const size_t dd = (size_t)dk * dv;
        const double *Q = q + (size_t)bh * T * dk, *K = k + (size_t)bh * T * dk;
        const double *V = v + (size_t)bh * T * dv, *DY = dy + (size_t)bh * T * dv;
        double *DQ = dq + (size_t)bh * T * dk, *DK = dk_out + (size_t)bh * T * dk;
        double *DV = dv_out + (size_t)bh * T * dv;
        /* States A_t after step t's write, t = -1..T-1 (A_{-1} = 0). */
        double *As = (double *)calloc((size_t)(T + 1) * dd, sizeof(double));
        double *dA = (double *)calloc(dd, sizeof(double));
        double *p = (double *)malloc(sizeof(double) * (size_t)(W + 1));
        double *dp = (double *)malloc(sizeof(double) * (size_t)(W + 1));
        double *m = (double *)malloc(sizeof(double) * (size_t)dv);
        double *dm = (double *)malloc(sizeof(double) * (size_t)dv);
        if (!As || !dA || !p || !dp || !m || !dm) {
            err |= 1;
            free(As); free(dA); free(p); free(dp); free(m); free(dm);
            continue;
        }
        for (int t = 0; t < T; ++t) {            /* forward: the states only */
            const double *prev = As + (size_t)t * dd;
            double *cur = As + (size_t)(t + 1) * dd;
            memcpy(cur, prev, sizeof(double) * dd);
            if (t >= W) {
                const double *ke = K + (size_t)(t - W) * dk, *ve = V + (size_t)(t - W) * dv;
                for (int a = 0; a < dk; ++a)
                    for (int b = 0; b < dv; ++b)
                        cur[(size_t)a * dv + b] = lm * prev[(size_t)a * dv + b] + et * ke[a] * ve[b];
            }
        }
        double g_lam = 0.0, g_eta = 0.0, g_gate = 0.0;
        for (int t = T - 1; t >= 0; --t) {
            const double *qt = Q + (size_t)t * dk, *dyt = DY + (size_t)t * dv;
            const double *At = As + (size_t)(t + 1) * dd;
            /* (a) read and gate */
            for (int b = 0; b < dv; ++b) {
                double s = 0.0;
                for (int a = 0; a < dk; ++a) s += qt[a] * At[(size_t)a * dv + b];
                m[b] = s;
                dm[b] = sg * dyt[b];
            }
            double dym = 0.0;
            for (int b = 0; b < dv; ++b) dym += dyt[b] * m[b];
            g_gate += sg * (1.0 - sg) * dym;
            for (int a = 0; a < dk; ++a) {
                double s = 0.0;
                for (int b = 0; b < dv; ++b) s += At[(size_t)a * dv + b] * dm[b];
                DQ[(size_t)t * dk + a] += s;
                for (int b = 0; b < dv; ++b) dA[(size_t)a * dv + b] += qt[a] * dm[b];
            }
            /* (b) window softmax */
            const int s0 = t - W + 1 > 0 ? t - W + 1 : 0, n = t - s0 + 1;
            double mx = -INFINITY;
            for (int i = 0; i < n; ++i) {
                const double *ks = K + (size_t)(s0 + i) * dk;
                double s = 0.0;
                for (int a = 0; a < dk; ++a) s += qt[a] * ks[a];
                p[i] = s * scale;
                if (p[i] > mx) mx = p[i];
            }
            double z = 0.0;
            for (int i = 0; i < n; ++i) { p[i] = exp(p[i] - mx); z += p[i]; }
            double D = 0.0;
            for (int i = 0; i < n; ++i) {
                p[i] /= z;
                const double *vs = V + (size_t)(s0 + i) * dv;
                double s = 0.0;
                for (int b = 0; b < dv; ++b) s += dyt[b] * vs[b];
                dp[i] = s;
                D += p[i] * s;
            }
            for (int i = 0; i < n; ++i) {
                const double *ks = K + (size_t)(s0 + i) * dk;
                const double ds = p[i] * (dp[i] - D);
                for (int b = 0; b < dv; ++b) DV[(size_t)(s0 + i) * dv + b] += p[i] * dyt[b];
                for (int a = 0; a < dk; ++a) {
                    DQ[(size_t)t * dk + a] += scale * ds * ks[a];
                    DK[(size_t)(s0 + i) * dk + a] += scale * ds * qt[a];
                }
            }
            /* (c) the eviction write of step t */
            if (t >= W) {
                const int e = t - W;
                const double *ke = K + (size_t)e * dk, *ve = V + (size_t)e * dv;
                const double *Ap = As + (size_t)t * dd;  /* A_{t-1} */
                for (int a = 0; a < dk; ++a) {
                    double sv = 0.0;
                    for (int b = 0; b < dv; ++b) {
                        const double g = dA[(size_t)a * dv + b];
                        g_lam += g * Ap[(size_t)a * dv + b];
                        sv += g * ve[b];
                    }
                    g_eta += ke[a] * sv;
                    DK[(size_t)e * dk + a] += et * sv;
                }
                for (int b = 0; b < dv; ++b) {
                    double sk = 0.0;
                    for (int a = 0; a < dk; ++a) sk += dA[(size_t)a * dv + b] * ke[a];
                    DV[(size_t)e * dv + b] += et * sk;
                }
                for (size_t i = 0; i < dd; ++i) dA[i] *= lm;
            }
        }
        gl[(size_t)bh * 3 + 0] = g_lam;
        gl[(size_t)bh * 3 + 1] = g_eta;
        gl[(size_t)bh * 3 + 2] = g_gate;
        free(As); free(dA); free(p); free(dp); free(m); free(dm);
    }
    if (!err) {
        for (int h = 0; h < H; ++h) dlam[h] = deta[h] = dgate[h] = 0.0;
        for (int bh = 0; bh < units; ++bh) {  /* batch sums in a fixed order */
            dlam[bh % H] += gl[(size_t)bh * 3 + 0];
            deta[bh % H] += gl[(size_t)bh * 3 + 1];
            dgate[bh % H] += gl[(size_t)bh * 3 + 2];
        }
    }
    free(gl);
    return err ? -1 : 0;
}

/* DeltaNet delta-rule backward.  Forward step t (oracle_delta):
 * u_t = v_t - S_{t-1} k_t, S_t = S_{t-1} + beta_t u_t k_t^T, o_t = S_t q_t
 * (S is d_v x d_k).  Reverse step t, with dS the gradient with respect to S_t:
 *   dq_t = S_t^T do_t;  dS += do_t q_t^T;
 *   g = dS k_t;  dv_t = beta_t g;  dbeta_t = <u_t, g>;
 *   dk_t = beta_t dS^T u_t - S_{t-1}^T (beta_t g);
 *   dS <- dS - beta_t g k_t^T  (the gradient with respect to S_{t-1}).
 * q,k: [B][H][T][dk]; v, dy: [B][H][T][dv]; beta: [B][H][T];
 * S0: NULL or [B][H][dk][dv] key-major start state; dS_T: NULL or the
 * gradient with respect to the final state, same layout.  Outputs dq, dk,
 * dv, dbeta as their inputs; dS0: NULL or the gradient with respect to S0.
 * Returns 0, or -1 on allocation failure. */
int oracle_delta_backward(int B, int H, int T, int dk, int dv,
                          const double *q, const double *k, const double *v,
                          const double *beta, const double *S0, const double *dy,
                          const double *dS_T, double *dq, double *dk_out,
                          double *dv_out, double *dbeta, double *dS0)
{
    int err = 0;
    const int units = B * H;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : err)
    for (int bh = 0; bh < units; ++bh) {
        const size_t dd = (size_t)dk * dv;
        const double *Q = q + (size_t)bh * T * dk, *K = k + (size_t)bh * T * dk;
        const double *V = v + (size_t)bh * T * dv, *DY = dy + (size_t)bh * T * dv;
        const double *Bt = beta + (size_t)bh * T;
        /* Ss[t] = S_{t-1} (t = 0..T), stored key-major like the API: element
         * S_{i,j} (row i of d_v, column j of d_k) at [j * dv + i]. */
        double *Ss = (double *)calloc((size_t)(T + 1) * dd, sizeof(double));
        double *U = (double *)malloc(sizeof(double) * (size_t)T * dv);
        double *dS = (double *)calloc(dd, sizeof(double));
        double *g = (double *)malloc(sizeof(double) * (size_t)dv);
        if (!Ss || !U || !dS || !g) {
            err |= 1;
            free(Ss); free(U); free(dS); free(g);
            continue;
        }
        if (S0) memcpy(Ss, S0 + (size_t)bh * dd, sizeof(double) * dd);
        for (int t = 0; t < T; ++t) {
            const double *Sp = Ss + (size_t)t * dd;
            double *Sc = Ss + (size_t)(t + 1) * dd;
            const double *kt = K + (size_t)t * dk, *vt = V + (size_t)t * dv;
            double *ut = U + (size_t)t * dv;
            for (int i = 0; i < dv; ++i) {
                double s = 0.0;
                for (int j = 0; j < dk; ++j) s += Sp[(size_t)j * dv + i] * kt[j];
                ut[i] = vt[i] - s;
            }
            for (int j = 0; j < dk; ++j)
                for (int i = 0; i < dv; ++i)
                    Sc[(size_t)j * dv + i] = Sp[(size_t)j * dv + i] + Bt[t] * ut[i] * kt[j];
        }
        if (dS_T) memcpy(dS, dS_T + (size_t)bh * dd, sizeof(double) * dd);
        for (int t = T - 1; t >= 0; --t) {
            const double *St = Ss + (size_t)(t + 1) * dd, *Sp = Ss + (size_t)t * dd;
            const double *qt = Q + (size_t)t * dk, *kt = K + (size_t)t * dk;
            const double *dot = DY + (size_t)t * dv, *ut = U + (size_t)t * dv;
            const double bt = Bt[t];
            double *dqt = dq + ((size_t)bh * T + t) * dk, *dkt = dk_out + ((size_t)bh * T + t) * dk;
            double *dvt = dv_out + ((size_t)bh * T + t) * dv;
            for (int j = 0; j < dk; ++j) {                 /* dq = S_t^T do */
                double s = 0.0;
                for (int i = 0; i < dv; ++i) s += St[(size_t)j * dv + i] * dot[i];
                dqt[j] = s;
            }
            for (int j = 0; j < dk; ++j)                   /* dS += do q^T */
                for (int i = 0; i < dv; ++i) dS[(size_t)j * dv + i] += dot[i] * qt[j];
            double db = 0.0;
            for (int i = 0; i < dv; ++i) {                 /* g = dS k */
                double s = 0.0;
                for (int j = 0; j < dk; ++j) s += dS[(size_t)j * dv + i] * kt[j];
                g[i] = s;
                dvt[i] = bt * s;
                db += ut[i] * s;
            }
            dbeta[(size_t)bh * T + t] = db;
            for (int j = 0; j < dk; ++j) {                 /* dk = beta dS^T u - S_{t-1}^T (beta g) */
                double s = 0.0;
                for (int i = 0; i < dv; ++i)
                    s += bt * dS[(size_t)j * dv + i] * ut[i] - Sp[(size_t)j * dv + i] * bt * g[i];
                dkt[j] = s;
            }
            for (int j = 0; j < dk; ++j)                   /* dS -= beta g k^T */
                for (int i = 0; i < dv; ++i) dS[(size_t)j * dv + i] -= bt * g[i] * kt[j];
        }
        if (dS0) memcpy(dS0 + (size_t)bh * dd, dS, sizeof(double) * dd);
        free(Ss); free(U); free(dS); free(g);
    }
    return err ? -1 : 0;
}

/* ======================================================================
 * BDH key generation (ainews.random.gg, BDH memory-architecture post: the
 * wide, sparse, non-negative activations come from a low-rank factorisation
 * followed by ReLU thresholding).  For one head h, a token's R-dimensional
 * input x is lifted to the N-wide activation
 *     a[n] = max(0, sum_r x[r] U_h[r][n] - theta),
 * the same U_h serving queries and keys.  Plain float64 loops, no blocking.
 * x: [B][H][T][R]; U: [H][R][N]; out: [B][H][T][N].
 * ====================================================================== */
void oracle_bdh_keys(int B, int H, int T, int R, int N, const double *x, const double *U,
                     double theta, double *out)
{
    const long rows = (long)B * H * T;
#pragma omp parallel for schedule(static)
    for (long row = 0; row < rows; ++row) {
        const int h = (int)((row / T) % H);
        const double *xr = x + (size_t)row * R;
        const double *Uh = U + (size_t)h * R * N;
        double *o = out + (size_t)row * N;
        for (int n = 0; n < N; ++n) {
            double s = 0.0;
            for (int r = 0; r < R; ++r) s += xr[r] * Uh[(size_t)r * N + n];
            s -= theta;
            o[n] = s > 0.0 ? s : 0.0;
        }
    }
}
