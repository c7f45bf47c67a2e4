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
