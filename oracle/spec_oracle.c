/*
 * spec_oracle.c -- CPU oracle for the speculative-decoding verification step.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or calls
 * this file; only the tests, the package's smoke check and the benchmark's CPU
 * baseline do.  It shares no code, header, table or constant generator with the
 * CUDA path.
 *
 * Everything is computed in IEEE double, one request at a time, in the order the
 * method states it, with no blocking or fusion:
 *
 *   "Спекулятивный декодинг в проде" (kiosknews.app), section "Немного теории":
 *     - notation: p is the target distribution *after temperature*, q the draft
 *       distribution, x the proposed token;
 *     - "Правило проверки": accept x with probability min(1, p(x)/q(x)); on a
 *       rejection sample a new token from the normalised residual max(0, p - q);
 *     - "Утверждение 1": the emitted token is distributed exactly as p whatever q;
 *     - "Утверждение 2": a pass yields the accepted tokens plus one token of the
 *       target model itself.
 *   "speculative decoding от черновика до проверки" (braintools.ru), section
 *   "Как это работает", steps 2-3 and the six-token remark: all drafts are
 *   checked left to right in one target pass; the target's own token is placed
 *   at the first mismatch, and when all K are accepted one more token comes from
 *   the same pass (position K+1).  Section "Почему ответ не портится": at
 *   temperature 0 the check reduces to comparing with the target argmax.
 *   "DSpark: ... верификацией по уверенности" (iitog.ru): the verify length is
 *   chosen per request from the estimated survival probability of the draft
 *   prefix.
 *
 * Readings where the pages are silent:
 *   - the same per-request temperature T divides both target and draft logits;
 *   - T <= 0, T not finite, or T below the smallest normal float => greedy;
 *   - acceptance test "u * q(x) < p(x)" with u in [0,1) on a 2^-24 grid;
 *   - argmax ties resolve to the lowest token index;
 *   - inverse-CDF sampling: the smallest v with C_v > u * Z, C the inclusive
 *     prefix sum in ascending token order, u in [0,1) on a 2^-53 grid; if no
 *     such v exists (rounding) the largest v with positive weight;
 *   - a residual whose mass Z is 0 falls back to sampling from p;
 *   - output positions after the emitted token hold -1;
 *   - verify_len is clamped to [0, K]; a draft token outside [0, V) at
 *     position k cuts the verify length to k;
 *   - schedule: L = number of leading positions whose float32 running product
 *     of draft max-probabilities stays >= threshold (left to right, every
 *     product rounded to float32, no fused multiply-add);
 *   - candidate trees: the functions of the two tree sections state their
 *     readings (the greedy walk; sibling candidates checked in index order
 *     against successively updated residuals).
 *
 * Random numbers: Philox4x32-10 as published by Salmon, Moraes, Dror and Shaw,
 * "Parallel random numbers: as easy as 1, 2, 3" (SC'11), written here from the
 * paper's definition.  Key = (lo32(seed), hi32(seed)); counter = (request b,
 * position k, draw, 0); draw 0 is the acceptance test at position k, draw 1 is
 * the residual / bonus sample at the emitted position.
 */
#include <math.h>
#include <float.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define SVO_F32 0
#define SVO_BF16 1
#define SVO_F64 2

#define SVO_BAD_TOKEN 1u
#define SVO_BAD_LEN 2u

/* ------------------------------------------------------------------ Philox */

static void svo_mulhilo(uint32_t a, uint32_t b, uint32_t *hi, uint32_t *lo) {
    uint64_t p = (uint64_t)a * (uint64_t)b;
    *hi = (uint32_t)(p >> 32);
    *lo = (uint32_t)p;
}

/* One Philox4x32 bijection followed by 10 rounds with a Weyl key schedule. */
void svo_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
    const uint32_t M0 = 0xD2511F53u, M1 = 0xCD9E8D57u;
    const uint32_t W0 = 0x9E3779B9u, W1 = 0xBB67AE85u;
    uint32_t x0 = ctr[0], x1 = ctr[1], x2 = ctr[2], x3 = ctr[3];
    uint32_t k0 = key[0], k1 = key[1];
    for (int r = 0; r < 10; ++r) {
        uint32_t hi0, lo0, hi1, lo1;
        svo_mulhilo(M0, x0, &hi0, &lo0);
        svo_mulhilo(M1, x2, &hi1, &lo1);
        uint32_t y0 = hi1 ^ x1 ^ k0;
        uint32_t y1 = lo1;
        uint32_t y2 = hi0 ^ x3 ^ k1;
        uint32_t y3 = lo0;
        x0 = y0; x1 = y1; x2 = y2; x3 = y3;
        k0 += W0; k1 += W1;
    }
    out[0] = x0; out[1] = x1; out[2] = x2; out[3] = x3;
}

static void svo_draw(uint64_t seed, uint32_t b, uint32_t k, uint32_t draw, uint32_t out[4]) {
    uint32_t ctr[4] = {b, k, draw, 0u};
    uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    svo_philox4x32_10(ctr, key, out);
}

/* Acceptance uniform at position k: top 24 bits of word 0, times 2^-24. */
double svo_u_accept(uint64_t seed, uint32_t b, uint32_t k) {
    uint32_t w[4];
    svo_draw(seed, b, k, 0u, w);
    return (double)(w[0] >> 8) * (1.0 / 16777216.0);
}

/* Sampling uniform at emitted position: top 53 bits of (w0:w1), times 2^-53. */
double svo_u_sample(uint64_t seed, uint32_t b, uint32_t pos) {
    uint32_t w[4];
    svo_draw(seed, b, pos, 1u, w);
    uint64_t v = ((uint64_t)w[0] << 32) | (uint64_t)w[1];
    return (double)(v >> 11) * (1.0 / 9007199254740992.0);
}

/* ------------------------------------------------------------------ rows */

static double svo_logit(const void *row, int dtype, int v) {
    if (dtype == SVO_F32) return (double)((const float *)row)[v];
    if (dtype == SVO_F64) return ((const double *)row)[v];
    uint16_t h = ((const uint16_t *)row)[v];
    uint32_t bits = (uint32_t)h << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

static size_t svo_esize(int dtype) {
    return dtype == SVO_F32 ? 4u : dtype == SVO_BF16 ? 2u : 8u;
}

static const void *svo_row(const void *base, int dtype, size_t row_index, int V) {
    return (const char *)base + row_index * (size_t)V * svo_esize(dtype);
}

/* Greedy iff T is not a positive normal float. */
int svo_is_greedy(float T) {
    return !(isfinite(T) && T >= FLT_MIN);
}

/* Temperature softmax of one row: y_v = z_v / T, m = max y, e_v = exp(y_v - m),
 * S = sum e_v (ascending v), p_v = e_v / S.  p may be NULL. */
void svo_row_softmax(const void *row, int dtype, int V, double T, double *p,
                     double *m_out, double *S_out) {
    double m = -INFINITY;
    for (int v = 0; v < V; ++v) {
        double y = svo_logit(row, dtype, v) / T;
        if (y > m) m = y;
    }
    double S = 0.0;
    for (int v = 0; v < V; ++v) {
        double e = exp(svo_logit(row, dtype, v) / T - m);
        if (p) p[v] = e;
        S += e;
    }
    if (p)
        for (int v = 0; v < V; ++v) p[v] /= S;
    if (m_out) *m_out = m;
    if (S_out) *S_out = S;
}

/* Probability of one token under the temperature softmax of a row. */
double svo_row_prob(const void *row, int dtype, int V, double T, int x) {
    double m, S;
    svo_row_softmax(row, dtype, V, T, NULL, &m, &S);
    return exp(svo_logit(row, dtype, x) / T - m) / S;
}

/* Lowest index of the largest raw logit. */
int svo_row_argmax(const void *row, int dtype, int V) {
    int best = 0;
    double bv = svo_logit(row, dtype, 0);
    for (int v = 1; v < V; ++v) {
        double z = svo_logit(row, dtype, v);
        if (z > bv) { bv = z; best = v; }
    }
    return best;
}

/* Acceptance rule, division free: accept iff u * q(x) < p(x). */
int svo_accept(double p_x, double q_x, double u) {
    return u * q_x < p_x;
}

/* Inverse CDF over non-negative weights w (not necessarily normalised):
 * smallest v with C_v > u * Z; fallback: largest v with w_v > 0 (or V-1).
 * If margin is non-NULL it receives the distance from u to the nearest
 * boundary of the chosen interval on the normalised CDF. */
int svo_inverse_cdf(const double *w, int V, double u, double *margin) {
    double Z = 0.0;
    for (int v = 0; v < V; ++v) Z += w[v];
    double thr = u * Z;
    double C = 0.0, prev = 0.0;
    int tok = -1;
    for (int v = 0; v < V; ++v) {
        prev = C;
        C += w[v];
        if (C > thr) { tok = v; break; }
    }
    if (tok < 0) {
        tok = V - 1;
        for (int v = V - 1; v >= 0; --v)
            if (w[v] > 0.0) { tok = v; break; }
        if (margin) *margin = 0.0;
        return tok;
    }
    if (margin) {
        double lo = (thr - prev) / Z, hi = (C - thr) / Z;
        *margin = lo < hi ? lo : hi;
    }
    return tok;
}

/* Residual sample at a rejected position: weights max(0, p - q); if their
 * total is 0 the sample is taken from p instead. */
int svo_sample_residual(const double *p, const double *q, int V, double u, double *r_scratch,
                        double *margin) {
    double Z = 0.0;
    for (int v = 0; v < V; ++v) {
        double d = p[v] - q[v];
        r_scratch[v] = d > 0.0 ? d : 0.0;
        Z += r_scratch[v];
    }
    if (Z == 0.0) return svo_inverse_cdf(p, V, u, margin);
    return svo_inverse_cdf(r_scratch, V, u, margin);
}

/* ------------------------------------------------------------- one request */

typedef struct {
    double accept_margin; /* min |u - p/q| over evaluated positions (q > 0) */
    double cdf_margin;    /* distance of u to the nearest boundary, or +inf */
    uint32_t status;      /* SVO_BAD_TOKEN / SVO_BAD_LEN */
} svo_diag;

/* Effective verify length after clamping and token validation. */
static int svo_effective_len(const int32_t *tokens, int K, int V, int L_in, uint32_t *status) {
    int L = L_in;
    if (L < 0) { L = 0; *status |= SVO_BAD_LEN; }
    if (L > K) { L = K; *status |= SVO_BAD_LEN; }
    for (int k = 0; k < L; ++k)
        if (tokens[k] < 0 || tokens[k] >= V) { L = k; *status |= SVO_BAD_TOKEN; break; }
    return L;
}

/* Verify one request with given uniforms.  tgt points at K+1 rows of V logits,
 * drf at K rows (unused when greedy).  u_acc[k] is the acceptance uniform of
 * position k (k < L); u_s[a] is the sampling uniform used when the emitted
 * position is a (u_s holds K+1 entries).  work must hold 3*V doubles.
 * Returns the accept length a and writes out[0..K]. */
int svo_verify_request_u(const void *tgt, const void *drf, int dtype, const int32_t *tokens,
                         int K, int V, int L_in, float T, const double *u_acc, const double *u_s,
                         int32_t *out, double *work, svo_diag *diag) {
    svo_diag d = {INFINITY, INFINITY, 0u};
    int L = svo_effective_len(tokens, K, V, L_in, &d.status);
    int a = L;
    int emitted;
    if (svo_is_greedy(T)) {
        /* compare each draft token with the target argmax, left to right */
        for (int k = 0; k < L; ++k) {
            int am = svo_row_argmax(svo_row(tgt, dtype, (size_t)k, V), dtype, V);
            if (tokens[k] != am) { a = k; break; }
        }
        emitted = svo_row_argmax(svo_row(tgt, dtype, (size_t)a, V), dtype, V);
    } else {
        double Td = (double)T;
        double *p = work, *q = work + V, *r = work + 2 * (size_t)V;
        for (int k = 0; k < L; ++k) {
            double pk = svo_row_prob(svo_row(tgt, dtype, (size_t)k, V), dtype, V, Td, tokens[k]);
            double qk = svo_row_prob(svo_row(drf, dtype, (size_t)k, V), dtype, V, Td, tokens[k]);
            if (qk > 0.0) {
                double gap = fabs(u_acc[k] - pk / qk);
                if (gap < d.accept_margin) d.accept_margin = gap;
            }
            if (!svo_accept(pk, qk, u_acc[k])) { a = k; break; }
        }
        svo_row_softmax(svo_row(tgt, dtype, (size_t)a, V), dtype, V, Td, p, NULL, NULL);
        if (a < L) {
            svo_row_softmax(svo_row(drf, dtype, (size_t)a, V), dtype, V, Td, q, NULL, NULL);
            emitted = svo_sample_residual(p, q, V, u_s[a], r, &d.cdf_margin);
        } else {
            emitted = svo_inverse_cdf(p, V, u_s[a], &d.cdf_margin);
        }
    }
    for (int k = 0; k < a; ++k) out[k] = tokens[k];
    out[a] = emitted;
    for (int k = a + 1; k <= K; ++k) out[k] = -1;
    if (diag) *diag = d;
    return a;
}

/* ------------------------------------------------------------- batch */

typedef struct {
    const void *tgt; size_t tgt_bstride; /* elements between requests */
    const void *drf; size_t drf_bstride;
    int dtype;
    const int32_t *tokens; size_t tok_bstride;
    const int32_t *verify_len; /* NULL => K */
    const float *temperature;
    uint64_t seed;
    int K, V;
    int b0, b1;
    int32_t *out_tokens; int32_t *accept_len;
    double *accept_margin; double *cdf_margin; uint32_t *status;
} svo_batch;

typedef struct { const svo_batch *job; int lo, hi; int rc; } svo_slice;

static void *svo_run_slice(void *arg) {
    svo_slice *s = (svo_slice *)arg;
    const svo_batch *j = s->job;
    int K = j->K, V = j->V;
    double *work = (double *)malloc(sizeof(double) * 3 * (size_t)V);
    double *u_acc = (double *)malloc(sizeof(double) * (size_t)K);
    double *u_s = (double *)malloc(sizeof(double) * (size_t)(K + 1));
    if (!work || !u_acc || !u_s) { free(work); free(u_acc); free(u_s); s->rc = -1; return NULL; }
    size_t es = svo_esize(j->dtype);
    for (int b = s->lo; b < s->hi; ++b) {
        const void *tgt = (const char *)j->tgt + (size_t)b * j->tgt_bstride * es;
        const void *drf = j->drf ? (const char *)j->drf + (size_t)b * j->drf_bstride * es : NULL;
        const int32_t *tok = j->tokens + (size_t)b * j->tok_bstride;
        int L_in = j->verify_len ? j->verify_len[b] : K;
        for (int k = 0; k < K; ++k) u_acc[k] = svo_u_accept(j->seed, (uint32_t)b, (uint32_t)k);
        for (int k = 0; k <= K; ++k) u_s[k] = svo_u_sample(j->seed, (uint32_t)b, (uint32_t)k);
        svo_diag d;
        int32_t *out = j->out_tokens + (size_t)(b - j->b0) * (size_t)(K + 1);
        int a = svo_verify_request_u(tgt, drf, j->dtype, tok, K, V, L_in, j->temperature[b], u_acc,
                                     u_s, out, work, &d);
        j->accept_len[b - j->b0] = a;
        if (j->accept_margin) j->accept_margin[b - j->b0] = d.accept_margin;
        if (j->cdf_margin) j->cdf_margin[b - j->b0] = d.cdf_margin;
        if (j->status) j->status[b - j->b0] = d.status;
    }
    free(work);
    free(u_acc);
    free(u_s);
    s->rc = 0;
    return NULL;
}

/* Verify requests [b0, b1) of a batch.  Outputs are indexed from b0 (row 0 of
 * out_tokens is request b0).  nthreads > 1 splits the requests over POSIX
 * threads.  Returns 0 on success. */
int svo_verify_batch(const void *tgt, size_t tgt_bstride, const void *drf, size_t drf_bstride,
                     int dtype, const int32_t *tokens, size_t tok_bstride,
                     const int32_t *verify_len, const float *temperature, uint64_t seed,
                     int K, int V, int b0, int b1, int nthreads, int32_t *out_tokens,
                     int32_t *accept_len, double *accept_margin, double *cdf_margin,
                     uint32_t *status) {
    if (K < 1 || V < 1 || b1 < b0) return -2;
    svo_batch job = {tgt, tgt_bstride, drf, drf_bstride, dtype, tokens, tok_bstride, verify_len,
                     temperature, seed, K, V, b0, b1, out_tokens, accept_len, accept_margin,
                     cdf_margin, status};
    int n = b1 - b0;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > n) nthreads = n > 0 ? n : 1;
    svo_slice *sl = (svo_slice *)calloc((size_t)nthreads, sizeof(svo_slice));
    pthread_t *th = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!sl || !th) { free(sl); free(th); return -1; }
    for (int t = 0; t < nthreads; ++t) {
        sl[t].job = &job;
        sl[t].lo = b0 + (int)((long long)n * t / nthreads);
        sl[t].hi = b0 + (int)((long long)n * (t + 1) / nthreads);
    }
    int rc = 0;
    if (nthreads == 1) {
        svo_run_slice(&sl[0]);
        rc = sl[0].rc;
    } else {
        for (int t = 0; t < nthreads; ++t) pthread_create(&th[t], NULL, svo_run_slice, &sl[t]);
        for (int t = 0; t < nthreads; ++t) {
            pthread_join(th[t], NULL);
            if (sl[t].rc) rc = sl[t].rc;
        }
    }
    free(sl);
    free(th);
    return rc;
}

/* Row intermediates of one logit row at temperature T: max of z/T, log of
 * sum exp(z/T - max), and the probability of token x (x < 0: skipped). */
void svo_row_intermediates(const void *row, int dtype, int V, float T, int x, double *m,
                           double *logS, double *px) {
    double mm, S;
    svo_row_softmax(row, dtype, V, (double)T, NULL, &mm, &S);
    *m = mm;
    *logS = log(S);
    if (x >= 0 && x < V) *px = exp(svo_logit(row, dtype, x) / (double)T - mm) / S;
}

/* ------------------------------------------------------------- tree (greedy) */

/* Greedy verification of a candidate tree ("speculative decoding от черновика до
 * проверки" (braintools.ru), Medusa / EAGLE-2 passages: the drafts form a tree of
 * candidates that the target checks in one pass; "Почему ответ не портится?": at
 * temperature 0 a draft token is kept when it equals the target's argmax).
 * Node 0 is the root (the last committed token); node n >= 1 carries token[n]
 * and parent[n] < n.  Row n of the target logits predicts the token after node
 * n.  Walk from the root: t = argmax of the current node's row (lowest index);
 * the next node is the lowest-index child carrying t; without one, t is the
 * emitted token.  Writes the path's tokens (accepted, then the emitted one) and
 * node indices, -1 after; returns the number of accepted nodes.  A node whose
 * parent is not an earlier node belongs to no path. */
int svo_verify_tree_greedy(const void *target, int dtype, const int32_t *parent,
                           const int32_t *token, int N, int V, int32_t *out_tokens,
                           int32_t *out_nodes) {
    const size_t esz = dtype == SVO_BF16 ? 2 : (dtype == SVO_F64 ? 8 : 4);
    for (int i = 0; i < N; ++i) {
        out_tokens[i] = -1;
        out_nodes[i] = -1;
    }
    int cur = 0, depth = 0;
    for (;;) {
        const int t = svo_row_argmax((const char *)target + (size_t)cur * V * esz, dtype, V);
        int next = -1;
        for (int c = cur + 1; c < N; ++c)
            if (parent[c] == cur && token[c] == t) {
                next = c;
                break;
            }
        out_tokens[depth] = t;  /* accepted, or emitted when no child carries it */
        if (next < 0) return depth;  /* a path has at most N - 1 accepted nodes */
        out_nodes[depth] = next;
        cur = next;
        ++depth;
    }
}

/* ------------------------------------------------------------- tree (sampled) */

/* Sampled verification of a candidate tree.  The pages give the acceptance rule
 * for one candidate per position ("Спекулятивный декодинг в проде"
 * (kiosknews.app), "Правило проверки") and let the drafts form a tree (the
 * Medusa and EAGLE-2 passages of the braintools.ru page); several children of
 * one node are checked against successively updated residuals, the
 * multi-candidate form of the same rule (reading):
 *   at node u the weights r start as p_u (target row u at T) with normaliser
 *   Z = 1; each child c of u, in index order, proposes x = token[c] (a token
 *   outside [0, V) is no candidate) and is accepted iff u_acc[c] * q_u(x) <
 *   r(x) / Z (q_u = draft row u at T); a rejection replaces r by
 *   max(0, r / Z - q_u) and Z by its sum (when that sum is 0, r = p_u and
 *   Z = 1 again).  An accepted child becomes the current node; when no child is
 *   accepted the emitted token is the inverse CDF of r at u_s[u].
 * With one child per node this is the linear rule step for step: the first
 * residual is max(0, p - q) and a node without candidates samples p.  Each
 * child's proposal drawn independently from q_u keeps the emitted token's law
 * equal to p_u.  Greedy T: the greedy tree walk.  work holds 3 * V doubles.
 *
 * distinct != 0: the siblings of a node are distinct tokens, drawn one after
 * another WITHOUT replacement from q_u (the top-k candidates per position of
 * the EAGLE and DFlash 2 passages: "Спекулятивное декодирование в vLLM и
 * SGLang" (alesha.pro), EAGLE-3 tree flags; kiosknews.app, "7. DFlash 2", 16
 * candidates per position).  Each child's draft law is then q_u without the
 * tokens of the siblings checked before it, renormalised (reading): after a
 * rejected sibling with token x, q(x) is set to 0 and q is divided by its
 * remaining mass 1 - q(x) before the next sibling is checked, and the residual
 * update uses that q.  A sibling repeating a rejected sibling's token, or one
 * met when q has no mass left, could not have been drawn: no candidate.
 *
 * Writes the path (tokens, node indices, -1 after) and returns the number of
 * accepted nodes; diag receives the smallest |u_acc - (r(x)/Z)/q_u(x)| over the
 * evaluated candidates and the inverse CDF's margin. */
int svo_verify_tree_u(const void *target, const void *draft, int dtype, const int32_t *parent,
                      const int32_t *token, int N, int V, float T, int distinct,
                      const double *u_acc, const double *u_s, int32_t *out_tokens,
                      int32_t *out_nodes, double *work, svo_diag *diag) {
    svo_diag d = {INFINITY, INFINITY, 0u};
    if (svo_is_greedy(T)) {
        int a = svo_verify_tree_greedy(target, dtype, parent, token, N, V, out_tokens, out_nodes);
        if (diag) *diag = d;
        return a;
    }
    for (int i = 0; i < N; ++i) {
        out_tokens[i] = -1;
        out_nodes[i] = -1;
    }
    const double Td = (double)T;
    double *p = work, *q = work + V, *r = work + 2 * (size_t)V;
    int cur = 0, depth = 0;
    for (;;) {
        svo_row_softmax(svo_row(target, dtype, (size_t)cur, V), dtype, V, Td, p, NULL, NULL);
        memcpy(r, p, (size_t)V * sizeof(double));
        double Z = 1.0;
        int have_q = 0, next = -1;
        int q_empty = 0;  /* distinct: q has no mass left */
        for (int c = cur + 1; c < N; ++c) {
            if (parent[c] != cur) continue;
            const int x = token[c];
            if (x < 0 || x >= V) continue;
            if (distinct) {  /* a token no draw without replacement could give */
                int dup = 0;
                for (int i = cur + 1; i < c; ++i)
                    if (parent[i] == cur && token[i] == x) dup = 1;
                if (dup || q_empty) continue;
            }
            if (!have_q) {
                svo_row_softmax(svo_row(draft, dtype, (size_t)cur, V), dtype, V, Td, q, NULL, NULL);
                have_q = 1;
            }
            const double rx = r[x] / Z;
            if (q[x] > 0.0) {
                double gap = fabs(u_acc[c] - rx / q[x]);
                if (gap < d.accept_margin) d.accept_margin = gap;
            }
            if (svo_accept(rx, q[x], u_acc[c])) {
                next = c;
                break;
            }
            double Zn = 0.0;
            for (int v = 0; v < V; ++v) {
                double w = r[v] / Z - q[v];
                r[v] = w > 0.0 ? w : 0.0;
                Zn += r[v];
            }
            if (Zn == 0.0) {
                memcpy(r, p, (size_t)V * sizeof(double));
                Zn = 1.0;
            }
            Z = Zn;
            if (distinct) {  /* the next sibling is drawn from q without x */
                const double rest = 1.0 - q[x];
                q[x] = 0.0;
                if (rest > 0.0) {
                    for (int v = 0; v < V; ++v) q[v] = q[v] / rest;
                } else {
                    q_empty = 1;
                }
            }
        }
        if (next < 0) {
            out_tokens[depth] = svo_inverse_cdf(r, V, u_s[cur], &d.cdf_margin);
            break;
        }
        out_tokens[depth] = token[next];
        out_nodes[depth] = next;
        cur = next;
        ++depth;
    }
    if (diag) *diag = d;
    return depth;
}

/* A batch of sampled trees with the oracle's own Philox: candidate node c >= 1
 * of request b takes the acceptance uniform of position c - 1 and node u's
 * emitted token the sampling uniform of position u, so a chain tree draws the
 * same numbers as the linear verification.  target and draft [B, N, V];
 * parent, token [B, N]; outputs [B, N] and per-request accepted counts and
 * margins.  Row b of the arrays is request b0 + b of the batch (its Philox
 * index). */
int svo_verify_tree_sampled(const void *target, const void *draft, int dtype,
                            const int32_t *parent, const int32_t *token, int b0, int B, int N,
                            int V, const float *temperature, uint64_t seed, int distinct,
                            int32_t *out_tokens, int32_t *out_nodes, int32_t *accepted,
                            double *accept_margin, double *cdf_margin) {
    const size_t esz = svo_esize(dtype);
    double *work = (double *)malloc(3 * (size_t)V * sizeof(double));
    double *ua = (double *)malloc((size_t)N * sizeof(double));
    double *us = (double *)malloc((size_t)N * sizeof(double));
    if (!work || !ua || !us) {
        free(work);
        free(ua);
        free(us);
        return -1;
    }
    for (int b = 0; b < B; ++b) {
        ua[0] = 0.0;
        for (int n = 0; n < N; ++n) {
            if (n > 0) ua[n] = svo_u_accept(seed, (uint32_t)(b0 + b), (uint32_t)(n - 1));
            us[n] = svo_u_sample(seed, (uint32_t)(b0 + b), (uint32_t)n);
        }
        const size_t off = (size_t)b * N;
        svo_diag d;
        accepted[b] = svo_verify_tree_u((const char *)target + off * V * esz,
                                        (const char *)draft + off * V * esz, dtype, parent + off,
                                        token + off, N, V, temperature[b], distinct, ua, us,
                                        out_tokens + off, out_nodes + off, work, &d);
        accept_margin[b] = d.accept_margin;
        cdf_margin[b] = d.cdf_margin;
    }
    free(work);
    free(ua);
    free(us);
    return 0;
}

/* ------------------------------------------------------------- LM head */

/* Logits of the LM-head product ("speculative decoding от черновика до
 * проверки" (braintools.ru), "Как это работает", step 2: the target scores the
 * drafts in one pass, whose last step maps each hidden state to vocabulary
 * logits): z[i][v] = sum_j h[i][j] * w[v][j] over j = 0..d-1 in ascending
 * order, in double, from bf16 hidden states h [M, d] and weights w [V, d]
 * (raw bit patterns).  Each product of two bf16 values is exact in double. */
static double svo_bf16_value(uint16_t bits) {
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

void svo_lm_logits(const uint16_t *h, const uint16_t *w, int M, int V, int d, double *z) {
    for (int i = 0; i < M; ++i) {
        const uint16_t *hr = h + (size_t)i * d;
        for (int v = 0; v < V; ++v) {
            const uint16_t *wr = w + (size_t)v * d;
            double s = 0.0;
            for (int j = 0; j < d; ++j) s += svo_bf16_value(hr[j]) * svo_bf16_value(wr[j]);
            z[(size_t)i * V + v] = s;
        }
    }
}

/* ------------------------------------------------------------- confidence */

/* Draft confidence of one position: the largest probability of the draft
 * distribution q at the request's temperature, max_v q(v) = 1 / sum_v exp(z_v/T
 * - max z/T).  A greedy request's q is a point mass: 1. */
void svo_draft_confidence(const void *draft, int dtype, int B, int K, int V,
                          const float *temperature, double *out) {
    const size_t esz = dtype == SVO_BF16 ? 2 : (dtype == SVO_F64 ? 8 : 4);
    for (int b = 0; b < B; ++b) {
        for (int k = 0; k < K; ++k) {
            const char *row = (const char *)draft + ((size_t)b * K + k) * (size_t)V * esz;
            double m, S;
            if (svo_is_greedy(temperature[b])) {
                out[(size_t)b * K + k] = 1.0;
                continue;
            }
            svo_row_softmax(row, dtype, V, (double)temperature[b], NULL, &m, &S);
            out[(size_t)b * K + k] = 1.0 / S;
        }
    }
}

/* ------------------------------------------------------------- schedule */

/* Confidence-scheduled verify length (DSpark): the number of leading draft
 * positions whose running float32 product of draft max-probabilities stays at
 * or above the threshold.  Each product is rounded to float32 on its own. */
/* Survival probability of draft prefix k of request b: the running float32
 * product c_0 * ... * c_k of the draft max-probabilities, each product rounded
 * on its own, with every c clamped to [0, 1] (NaN counts as 0). */
static void svo_survival(const float *maxprob, int B, int K, float *s) {
    for (int b = 0; b < B; ++b) {
        volatile float prod = 1.0f;
        for (int k = 0; k < K; ++k) {
            float c = maxprob[(size_t)b * K + k];
            if (!(c >= 0.0f)) c = 0.0f;
            if (c > 1.0f) c = 1.0f;
            volatile float cv = c;
            prod = prod * cv;
            s[(size_t)b * K + k] = prod;
        }
    }
}

static const float *g_sort_s;
static int svo_cmp_survival(const void *x, const void *y) {
    const int i = *(const int *)x, j = *(const int *)y;
    if (g_sort_s[i] != g_sort_s[j]) return g_sort_s[i] > g_sort_s[j] ? -1 : 1;
    return i < j ? -1 : (i > j ? 1 : 0);
}

/* Load-aware schedule (DSpark: the verify length follows both the prefix's
 * survival probability and the engine's current load): given a budget of
 * positions the engine verifies this step, keep the `budget` positions (b, k)
 * with the largest survival probabilities, ties to the lower b then the lower
 * k.  Survival never grows along a request, so the kept set is a prefix of
 * every request; verify_len[b] is its length. */
void svo_schedule_budget(const float *maxprob, int B, int K, long long budget, int32_t *out) {
    const size_t n = (size_t)B * K;
    float *s = (float *)malloc(n * sizeof(float));
    int *idx = (int *)malloc(n * sizeof(int));
    svo_survival(maxprob, B, K, s);
    for (size_t i = 0; i < n; ++i) idx[i] = (int)i;
    g_sort_s = s;
    qsort(idx, n, sizeof(int), svo_cmp_survival);
    for (int b = 0; b < B; ++b) out[b] = 0;
    const size_t take = budget <= 0 ? 0 : ((size_t)budget < n ? (size_t)budget : n);
    for (size_t i = 0; i < take; ++i) out[idx[i] / K] += 1;
    free(s);
    free(idx);
}

void svo_schedule_len(const float *maxprob, float threshold, int B, int K, int32_t *out) {
    for (int b = 0; b < B; ++b) {
        volatile float prod = 1.0f;
        int L = 0;
        for (int k = 0; k < K; ++k) {
            volatile float c = maxprob[(size_t)b * K + k];
            prod = prod * c;
            if (prod >= threshold) L = k + 1;
            else break;
        }
        out[b] = L;
    }
}
