/*
 * sdv_oracle.c -- plain CPU oracle for batched speculative-decoding
 * verification.  TEST INFRASTRUCTURE ONLY (see sdv_oracle.h): only the
 * tests, the smoke check and the bench's CPU-baseline leg use it.
 *
 * Everything is IEEE double, single-threaded, one request at a time, one
 * vocabulary row at a time, in the order each method states its steps.
 *
 * Notation (per request b, draft k, depth j):
 *   target row (b,k,j) -> P_j = softmax(logits / T)      (j = 0..L_b)
 *   draft  row (b,k,j) -> Q_j = softmax(logits / T)      (j = 0..L_b-1)
 *   X^k_{j+1} = tokens[b][k][j], the token draft k drew from Q_j.
 * Drafts that share a prefix share a node of the draft trie; a node's rows
 * are those of the lowest-index draft through it ("owner").
 *
 * Readings (the pages name the methods but print none of their formulas):
 *  - Standard speculative sampling [SD]: accept X with probability
 *    min(1, P(X)/Q(X)); on rejection draw from norm(max(P - Q, 0)); when
 *    every position is accepted draw a bonus token from the last target row.
 *    With K > 1 drafts the per-position multi-draft rule [SPECTR] is read as
 *    recursive rejection sampling over the trie: at an accepted node the
 *    draws of the drafts through it are tried in index order against the
 *    running residual r (r <- norm(max(r - Q, 0)) after each rejection);
 *    the first accepted draw moves to its child; if every draw is rejected
 *    the correction token comes from r.
 *  - Greedy block verification [GBV] (single draft): the published block
 *    rule: p_0 = 1, p_i = min(p_{i-1} P_{i-1}(X_i)/Q_{i-1}(X_i), 1),
 *    h_i = S_i/(S_i + 1 - p_i) with S_i = sum_x max(p_i P_i(x) - Q_i(x), 0)
 *    for i < L, h_L = p_L; tau = max{i : eta_i <= h_i}; the correction comes
 *    from P_L when tau = L, else from norm(max(p_tau P_tau - Q_tau, 0)).
 *  - SpecTr-GBV [ALG1]: at node v (weight p_v, root p = 1) with draws
 *    y_1..y_n (tokens of the drafts through v, in index order):
 *        R_0 = p_v P_v,  D_0 = 1
 *        a_j = min(R_{j-1}(y_j) / (D_{j-1} Q_v(y_j)), 1)
 *        R_j = max(R_{j-1} - D_{j-1} Q_v, 0),  S_j = sum R_j,
 *        D_j = 1 - p_v + S_j
 *    The child reached first by draw j gets weight a_j.  h_v = S_n / D_n is
 *    the block acceptance probability h_ik of the sub-block ending at v
 *    (Eq. 2) and R_n / S_n is the residual the correction token is drawn
 *    from (Eq. 4); the sequence R_j is the adjustment of the target at the
 *    unaccepted positions (Algorithm 2).  The decision walks the trie depth
 *    first, children in order of first appearance, and ends at the first
 *    node whose test eta <= h_v passes on the way back up (the root always
 *    passes); a draft whose token was already rejected at a node has
 *    R(y) = 0, which is the rejected-set H of step 3.  With K = 1 this is
 *    exactly GBV; at p = 1 a node is exactly the recursive residual above.
 *  - Degenerate cases: a = 1 when D*Q(y) = 0; h = 1 when D = 0; the
 *    correction is drawn from P_v when S_n = 0.
 *  - Acceptance tests are "u <= threshold"; the inverse CDF takes the first
 *    token in index order whose running sum exceeds u*S, else the last
 *    token of nonzero mass.
 *  - T = 0 in a sampling mode gives the greedy result.
 */
#include "sdv_oracle.h"

#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* input access                                                              */

static size_t elem_size(int dtype) { return dtype == SDVO_BF16 ? 2u : dtype == SDVO_F64 ? 8u : 4u; }

static const unsigned char* row_of(const sdvo_problem* pb, int is_target, int b, int k, int j)
{
    long long rows = is_target ? (long long)pb->L + 1 : (long long)pb->L;
    long long r = ((long long)b * pb->K + k) * rows + j;
    const unsigned char* base = (const unsigned char*)(is_target ? pb->target : pb->draft);
    return base + (size_t)r * (size_t)pb->row_stride * elem_size(pb->dtype);
}

static double bf16_value(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

static double logit(const sdvo_problem* pb, const unsigned char* row, int x)
{
    float f;
    if (pb->dtype == SDVO_F64) {
        double g;
        memcpy(&g, row + 8 * (size_t)x, 8);
        return g;
    }
    if (pb->dtype == SDVO_BF16) {
        uint16_t h;
        uint32_t u;
        memcpy(&h, row + 2 * (size_t)x, 2);
        u = (uint32_t)h << 16;
        memcpy(&f, &u, 4);
    } else {
        memcpy(&f, row + 4 * (size_t)x, 4);
    }
    return (double)f;
}

/* A row can be used iff it holds no NaN, no +Inf and some value above -Inf. */
static int row_usable(const sdvo_problem* pb, const unsigned char* row)
{
    double m = -INFINITY;
    for (int x = 0; x < pb->V; ++x) {
        double l = logit(pb, row, x);
        if (isnan(l) || l == INFINITY) return 0;
        if (l > m) m = l;
    }
    return m > -INFINITY;
}

/* P(x) = exp((l(x) - max l) / T) / sum, T > 0. */
static void softmax(const sdvo_problem* pb, const unsigned char* row, double T, double* P)
{
    double m = -INFINITY, Z = 0.0;
    for (int x = 0; x < pb->V; ++x) {
        double l = logit(pb, row, x);
        if (l > m) m = l;
    }
    for (int x = 0; x < pb->V; ++x) {
        P[x] = exp((logit(pb, row, x) - m) / T);
        Z += P[x];
    }
    for (int x = 0; x < pb->V; ++x) P[x] /= Z;
}

/* Index of the largest raw logit, lowest index on ties. */
static int argmax_row(const sdvo_problem* pb, const unsigned char* row)
{
    int best = 0;
    double m = logit(pb, row, 0);
    for (int x = 1; x < pb->V; ++x) {
        double l = logit(pb, row, x);
        if (l > m) {
            m = l;
            best = x;
        }
    }
    return best;
}

/* ------------------------------------------------------------------------ */
/* per-request state                                                         */

typedef struct {
    const sdvo_problem* pb;
    int b, Lb, greedy;
    int owner[SDVO_MAX_L + 1][SDVO_MAX_K]; /* lowest draft sharing k's prefix of length j */
    double a[SDVO_MAX_L][SDVO_MAX_K];      /* acceptance probability of draft k's draw at depth j */
    double h[SDVO_MAX_L + 1][SDVO_MAX_K];  /* node (j, owner) block acceptance probability */
    double S[SDVO_MAX_L + 1][SDVO_MAX_K];  /* node residual mass S_n */
    int am[SDVO_MAX_L + 1][SDVO_MAX_K];    /* node argmax (greedy) */
    double rho[SDVO_MAX_L + 1][SDVO_MAX_K];   /* K-SEQ: node scaling factor rho */
    double gam[SDVO_MAX_L + 1][SDVO_MAX_K];   /* K-SEQ: node factor (1 - (1 - beta)^n) / beta */
    double margin;
    sdvo_trace* tr;
    double *P, *Q, *R;                     /* V-sized scratch */
} req_t;

static int tok(const req_t* r, int k, int j)
{
    const sdvo_problem* pb = r->pb;
    return pb->tokens[((size_t)r->b * pb->K + k) * pb->L + j];
}

static void trace_add(req_t* r, int kind, int index, double lo, double hi)
{
    sdvo_trace* t = r->tr;
    if (!t) return;
    if (t->n < t->cap) {
        t->e[t->n].kind = kind;
        t->e[t->n].index = index;
        t->e[t->n].lo = lo;
        t->e[t->n].hi = hi;
    }
    t->n++;
}

/* Accept test of draft k at depth j: u <= thr with u = accept_u[b][k][j]. */
static int accept_test(req_t* r, int k, int j, double thr)
{
    const sdvo_problem* pb = r->pb;
    int idx = (r->b * pb->K + k) * pb->L + j;
    double u = pb->accept_u[idx];
    trace_add(r, 0, idx, thr, thr);
    if (fabs(u - thr) < r->margin) r->margin = fabs(u - thr);
    return u <= thr;
}

/* Inverse-CDF draw from the nonnegative weights w (sum > 0) with
 * u = sample_u[b][k][j]. */
static int sample_icdf(req_t* r, const double* w, int k, int j)
{
    const sdvo_problem* pb = r->pb;
    int idx = (r->b * pb->K + k) * (pb->L + 1) + j;
    double u = pb->sample_u[idx];
    double S = 0.0, cum = 0.0, lo = 0.0, hi = INFINITY, last_prev = 0.0;
    int chosen = -1, last = -1;
    for (int x = 0; x < pb->V; ++x) S += w[x];
    for (int x = 0; x < pb->V; ++x) {
        if (w[x] > 0.0) {
            double prev = cum;
            cum += w[x];
            last = x;
            last_prev = prev;
            if (cum > u * S) {
                chosen = x;
                lo = prev / S;
                hi = cum / S;
                break;
            }
        }
    }
    if (chosen < 0) { /* rounding: every running sum stayed at or below u*S */
        chosen = last;
        lo = last_prev / S;
        hi = INFINITY;
    }
    trace_add(r, 1, idx, lo, hi);
    if (u - lo < r->margin) r->margin = u - lo;
    if (hi - u < r->margin) r->margin = hi - u;
    return chosen;
}

/* Draft trie: owner[j][k] = lowest k' whose first j tokens equal draft k's. */
static void build_trie(req_t* r)
{
    int K = r->pb->K;
    for (int j = 0; j <= r->Lb; ++j) {
        for (int k = 0; k < K; ++k) {
            int o = k;
            for (int k2 = 0; k2 < k; ++k2) {
                int same = 1;
                for (int i = 0; i < j && same; ++i) same = tok(r, k2, i) == tok(r, k, i);
                if (same) {
                    o = k2;
                    break;
                }
            }
            r->owner[j][k] = o;
        }
    }
}

/* Request status: bad length, else bad token, else an unusable row among
 * the rows every decision reads: each inner trie node's target row, and its
 * draft row in the sampling rules.  A leaf's row enters nothing but the
 * token drawn there (in the sampling rules its residual is p P, of mass p;
 * greedy takes its argmax as the correction), so it is read, and checked,
 * only when the decision ends at that leaf (draw_correction, run_greedy),
 * just as rows past L_b are never read. */
static int request_status(req_t* r)
{
    const sdvo_problem* pb = r->pb;
    int st = 0;
    if (r->Lb < 0 || r->Lb > pb->L) return SDVO_REQ_BAD_LENGTH;
    for (int k = 0; k < pb->K; ++k)
        for (int j = 0; j < r->Lb; ++j)
            if (tok(r, k, j) < 0 || tok(r, k, j) >= pb->V) st = SDVO_REQ_BAD_TOKEN;
    if (st) return st;
    build_trie(r);
    for (int j = 0; j <= r->Lb; ++j)
        for (int o = 0; o < pb->K; ++o) {
            if (r->owner[j][o] != o) continue;
            if (j < r->Lb && !row_usable(pb, row_of(pb, 1, r->b, o, j)))
                st = SDVO_REQ_NONFINITE;
            if (!r->greedy && j < r->Lb && !row_usable(pb, row_of(pb, 0, r->b, o, j)))
                st = SDVO_REQ_NONFINITE;
        }
    return st;
}

/* ------------------------------------------------------------------------ */
/* node evaluation: residual recursion of SpecTr-GBV at node (j, o) with
 * weight p (p = 1 gives recursive rejection sampling).  Leaves R_n in r->R,
 * P_v in r->P; stores a, h and S.  Returns S_n.  A leaf has no draws:
 * S = h = p, and its row is not read here. */
static double eval_node(req_t* r, int j, int o, double p)
{
    const sdvo_problem* pb = r->pb;
    int V = pb->V;
    double S = 0.0, D = 1.0;
    if (j == r->Lb) {
        r->S[j][o] = p;
        r->h[j][o] = p;
        return p;
    }
    softmax(pb, row_of(pb, 1, r->b, o, j), pb->temperature, r->P);
    for (int x = 0; x < V; ++x) r->R[x] = p * r->P[x];
    for (int x = 0; x < V; ++x) S += r->R[x];
    if (j < r->Lb) {
        softmax(pb, row_of(pb, 0, r->b, o, j), pb->temperature, r->Q);
        for (int k = 0; k < pb->K; ++k) {
            if (r->owner[j][k] != o) continue; /* draws of the drafts through this node */
            int y = tok(r, k, j);
            double denom = D * r->Q[y];
            r->a[j][k] = denom > 0.0 ? fmin(r->R[y] / denom, 1.0) : 1.0;
            for (int x = 0; x < V; ++x) r->R[x] = fmax(r->R[x] - D * r->Q[x], 0.0);
            S = 0.0;
            for (int x = 0; x < V; ++x) S += r->R[x];
            D = 1.0 - p + S;
        }
    }
    r->S[j][o] = S;
    r->h[j][o] = D > 0.0 ? S / D : 1.0;
    return S;
}

/* weight of node (j, o) under SpecTr-GBV: the a of the draw that first
 * reached it (its owner's draw one level up); root 1. */
static double node_weight(const req_t* r, int j, int o) { return j == 0 ? 1.0 : r->a[j - 1][o]; }

/* Depth-first search of SpecTr-GBV: children in order of first appearance,
 * then the node's own test on the way back. */
static int dfs_accept(req_t* r, int j, int o, int* ej, int* eo)
{
    if (j < r->Lb) {
        for (int k = 0; k < r->pb->K; ++k) {
            if (r->owner[j][k] == o && r->owner[j + 1][k] == k) {
                if (dfs_accept(r, j + 1, k, ej, eo)) return 1;
            }
        }
    }
    if (j == 0) {
        *ej = 0;
        *eo = 0;
        return 1;
    }
    if (accept_test(r, o, j - 1, r->h[j][o])) {
        *ej = j;
        *eo = o;
        return 1;
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* modes                                                                     */

typedef struct {
    int tau, kstar, token;
    double mass;
} outcome_t;

/* Draw the correction from the end node's residual (R_n / S_n), or from
 * P_v when S_n = 0 or at a leaf (the bonus token; R = p P there).  Returns
 * SDVO_REQ_NONFINITE, drawing nothing, when the end node is a leaf whose
 * target row is unusable; else 0. */
static int draw_correction(req_t* r, int ej, int eo, double p, outcome_t* out, double* residual_out)
{
    const sdvo_problem* pb = r->pb;
    int V = pb->V;
    double S;
    const double* w;
    double tot = 0.0;
    if (ej == r->Lb) {
        const unsigned char* row = row_of(pb, 1, r->b, eo, ej);
        if (!row_usable(pb, row)) return SDVO_REQ_NONFINITE;
        softmax(pb, row, pb->temperature, r->P);
        S = p;
        w = r->P;
    } else {
        S = eval_node(r, ej, eo, p);
        w = S > 0.0 ? r->R : r->P;
    }
    out->tau = ej;
    out->kstar = eo;
    out->mass = S;
    out->token = sample_icdf(r, w, eo, ej);
    if (residual_out) {
        for (int x = 0; x < V; ++x) tot += w[x];
        for (int x = 0; x < V; ++x) residual_out[x] = w[x] / tot;
    }
    return 0;
}

/* Token-level speculative sampling (K = 1) and its per-position
 * multi-draft form (K > 1): every node at p = 1, then the walk. */
static int run_token(req_t* r, float* accept_prob, outcome_t* out, double* residual_out)
{
    const sdvo_problem* pb = r->pb;
    int j = 0, o = 0;
    for (int d = 0; d <= r->Lb; ++d)
        for (int v = 0; v < pb->K; ++v)
            if (r->owner[d][v] == v) eval_node(r, d, v, 1.0);
    if (accept_prob)
        for (int k = 0; k < pb->K; ++k)
            for (int d = 0; d < r->Lb; ++d) accept_prob[k * pb->L + d] = (float)r->a[d][k];
    while (j < r->Lb) {
        int acc = -1;
        for (int k = 0; k < pb->K && acc < 0; ++k)
            if (r->owner[j][k] == o && accept_test(r, k, j, r->a[j][k])) acc = k;
        if (acc < 0) break;
        o = r->owner[j + 1][acc];
        ++j;
    }
    return draw_correction(r, j, o, 1.0, out, residual_out);
}

/* SpecTr-GBV: nodes in breadth-first order (a node's weight comes from its
 * parent), then the depth-first decision. */
static int run_multidraft(req_t* r, float* accept_prob, outcome_t* out, double* residual_out)
{
    const sdvo_problem* pb = r->pb;
    int ej = 0, eo = 0;
    for (int d = 0; d <= r->Lb; ++d)
        for (int v = 0; v < pb->K; ++v)
            if (r->owner[d][v] == v) eval_node(r, d, v, node_weight(r, d, v));
    if (accept_prob)
        for (int k = 0; k < pb->K; ++k)
            for (int d = 0; d < r->Lb; ++d) {
                int v = r->owner[d + 1][k];
                accept_prob[k * pb->L + d] = (float)r->h[d + 1][v];
            }
    dfs_accept(r, 0, 0, &ej, &eo);
    return draw_correction(r, ej, eo, node_weight(r, ej, eo), out, residual_out);
}

/* Greedy block verification, single draft, written from its own steps. */
static int run_block(req_t* r, float* accept_prob, outcome_t* out, double* residual_out)
{
    const sdvo_problem* pb = r->pb;
    int V = pb->V, Lb = r->Lb, tau = 0;
    double p[SDVO_MAX_L + 1], h[SDVO_MAX_L + 1], Si = 0.0;
    const double* w;
    double tot = 0.0;
    p[0] = 1.0;
    for (int i = 1; i <= Lb; ++i) {
        int X = tok(r, 0, i - 1);
        softmax(pb, row_of(pb, 1, r->b, 0, i - 1), pb->temperature, r->P);
        softmax(pb, row_of(pb, 0, r->b, 0, i - 1), pb->temperature, r->Q);
        p[i] = r->Q[X] > 0.0 ? fmin(p[i - 1] * r->P[X] / r->Q[X], 1.0) : 1.0;
    }
    for (int i = 1; i < Lb; ++i) {
        double S = 0.0;
        softmax(pb, row_of(pb, 1, r->b, 0, i), pb->temperature, r->P);
        softmax(pb, row_of(pb, 0, r->b, 0, i), pb->temperature, r->Q);
        for (int x = 0; x < V; ++x) S += fmax(p[i] * r->P[x] - r->Q[x], 0.0);
        h[i] = S + (1.0 - p[i]) > 0.0 ? S / (S + (1.0 - p[i])) : 1.0;
    }
    if (Lb >= 1) h[Lb] = p[Lb];
    if (accept_prob)
        for (int i = 1; i <= Lb; ++i) accept_prob[i - 1] = (float)h[i];
    for (int i = Lb; i >= 1; --i)
        if (accept_test(r, 0, i - 1, h[i])) {
            tau = i;
            break;
        }
    /* correction: P_L when tau = L, else norm(max(p_tau P_tau - Q_tau, 0));
     * target row L_b is read only here */
    if (tau == Lb && !row_usable(pb, row_of(pb, 1, r->b, 0, tau))) return SDVO_REQ_NONFINITE;
    softmax(pb, row_of(pb, 1, r->b, 0, tau), pb->temperature, r->P);
    if (tau < Lb) {
        softmax(pb, row_of(pb, 0, r->b, 0, tau), pb->temperature, r->Q);
        for (int x = 0; x < V; ++x) r->R[x] = fmax(p[tau] * r->P[x] - r->Q[x], 0.0);
        for (int x = 0; x < V; ++x) Si += r->R[x];
        w = Si > 0.0 ? r->R : r->P;
    } else {
        for (int x = 0; x < V; ++x) Si += p[tau] * r->P[x];
        w = r->P;
    }
    out->tau = tau;
    out->kstar = 0;
    out->mass = Si;
    out->token = sample_icdf(r, w, 0, tau);
    if (residual_out) {
        for (int x = 0; x < V; ++x) tot += w[x];
        for (int x = 0; x < V; ++x) residual_out[x] = w[x] / tot;
    }
    return 0;
}

/* SpecTr's K-SEQ at a node (the pages name it and its binary search for a
 * scaling factor rho: SpecTr-GBV page, sections 3-4; the rule is written
 * here from its published definition).  The n drafts through the node are
 * i.i.d. candidates from Q.  For rho >= 1 let
 *   beta(rho) = sum_x min(Q(x), P(x) / rho),
 *   gamma(rho) = (1 - (1 - beta)^n) / beta   (n when beta = 0).
 * Candidate i is accepted with probability min(1, P(y_i) / (rho Q(y_i))),
 * tried in index order; if every one is rejected the token is drawn from
 * P - gamma min(Q, P / rho).  That residual is nonnegative, and the emitted
 * token follows P exactly, whenever gamma(rho) <= rho (true at rho = n).
 * The search for a small such rho (acceptance falls as rho grows) is fixed
 * here so that a parallel implementation can take the same decisions: rho
 * = 1 if it qualifies; else, starting from [lo, hi] = [1, n], KSEQ_PASSES
 * rounds each test the three points lo + (hi - lo) i / 4 (i = 1, 2, 3) and
 * keep the quarter holding the first that qualifies (the last quarter if
 * none does).  rho is the final hi, which always qualifies.
 * Stores a, rho and gamma; leaves P, Q in r->P, r->Q. */
#define KSEQ_PASSES 10

static double kseq_beta(const req_t* r, double rho)
{
    double beta = 0.0;
    for (int x = 0; x < r->pb->V; ++x) beta += fmin(r->Q[x], r->P[x] / rho);
    return beta;
}

/* gamma with 1 - (1 - beta)^n = -expm1(n log1p(-beta)): the same value,
 * without the cancellation of the plain form when beta is small */
static double kseq_gamma(double beta, int n)
{
    beta = fmin(fmax(beta, 0.0), 1.0);
    return beta > 0.0 ? -expm1((double)n * log1p(-beta)) / beta : (double)n;
}

static int kseq_ok(const req_t* r, double rho, int n) { return kseq_gamma(kseq_beta(r, rho), n) <= rho; }

static void kseq_node(req_t* r, int j, int o)
{
    const sdvo_problem* pb = r->pb;
    int n = 0;
    double lo = 1.0, hi;
    softmax(pb, row_of(pb, 1, r->b, o, j), pb->temperature, r->P);
    softmax(pb, row_of(pb, 0, r->b, o, j), pb->temperature, r->Q);
    for (int k = 0; k < pb->K; ++k) n += r->owner[j][k] == o;
    hi = (double)n;
    if (kseq_ok(r, 1.0, n)) {
        hi = 1.0;
    } else {
        for (int it = 0; it < KSEQ_PASSES; ++it) {
            double m[4];
            int i = 1;
            m[0] = lo;
            for (int t = 1; t < 4; ++t) m[t] = lo + (hi - lo) * t / 4.0;
            while (i < 4 && !kseq_ok(r, m[i], n)) ++i;
            if (i < 4) {
                lo = m[i - 1];
                hi = m[i];
            } else {
                lo = m[3];
            }
        }
    }
    r->rho[j][o] = hi;
    r->gam[j][o] = kseq_gamma(kseq_beta(r, hi), n);
    for (int k = 0; k < pb->K; ++k) {
        if (r->owner[j][k] != o) continue;
        int y = tok(r, k, j);
        double den = hi * r->Q[y];
        r->a[j][k] = den > 0.0 ? fmin(r->P[y] / den, 1.0) : 1.0;
    }
}

/* K-SEQ at every node, then the walk of the token rule; the correction
 * comes from the end node's K-SEQ residual (P where it has no mass), or
 * P at a leaf. */
static int run_kseq(req_t* r, float* accept_prob, outcome_t* out, double* residual_out)
{
    const sdvo_problem* pb = r->pb;
    int V = pb->V, j = 0, o = 0;
    double S = 0.0, tot = 0.0;
    const double* w;
    for (int d = 0; d < r->Lb; ++d)
        for (int v = 0; v < pb->K; ++v)
            if (r->owner[d][v] == v) kseq_node(r, d, v);
    if (accept_prob)
        for (int k = 0; k < pb->K; ++k)
            for (int d = 0; d < r->Lb; ++d) accept_prob[k * pb->L + d] = (float)r->a[d][k];
    while (j < r->Lb) {
        int acc = -1;
        for (int k = 0; k < pb->K && acc < 0; ++k)
            if (r->owner[j][k] == o && accept_test(r, k, j, r->a[j][k])) acc = k;
        if (acc < 0) break;
        o = r->owner[j + 1][acc];
        ++j;
    }
    if (j == r->Lb) return draw_correction(r, j, o, 1.0, out, residual_out); /* the bonus token */
    kseq_node(r, j, o);
    for (int x = 0; x < V; ++x) {
        r->R[x] = fmax(r->P[x] - r->gam[j][o] * fmin(r->Q[x], r->P[x] / r->rho[j][o]), 0.0);
        S += r->R[x];
    }
    w = S > 0.0 ? r->R : r->P;
    out->tau = j;
    out->kstar = o;
    out->mass = S;
    out->token = sample_icdf(r, w, o, j);
    if (residual_out) {
        for (int x = 0; x < V; ++x) tot += w[x];
        for (int x = 0; x < V; ++x) residual_out[x] = w[x] / tot;
    }
    return 0;
}

/* Greedy T = 0: a draft position matches when its token is the row's
 * argmax; the longest matching draft wins (lowest k on ties); the
 * correction is the argmax after the accepted prefix. */
static int run_greedy(req_t* r, float* accept_prob, outcome_t* out, double* residual_out)
{
    const sdvo_problem* pb = r->pb;
    int best = -1, bestk = 0;
    for (int d = 0; d < r->Lb; ++d) /* the inner nodes' argmaxes decide the matches */
        for (int v = 0; v < pb->K; ++v)
            if (r->owner[d][v] == v) r->am[d][v] = argmax_row(pb, row_of(pb, 1, r->b, v, d));
    for (int k = 0; k < pb->K; ++k) {
        int m = 0;
        while (m < r->Lb && tok(r, k, m) == r->am[m][r->owner[m][k]]) ++m;
        if (m > best) {
            best = m;
            bestk = k;
        }
        if (accept_prob)
            for (int d = 0; d < r->Lb; ++d)
                accept_prob[k * pb->L + d] = tok(r, k, d) == r->am[d][r->owner[d][k]] ? 1.0f : 0.0f;
    }
    out->tau = best;
    out->kstar = bestk;
    if (best == r->Lb) { /* a leaf: its row is read only now, for the correction */
        const unsigned char* row = row_of(pb, 1, r->b, r->owner[best][bestk], best);
        if (!row_usable(pb, row)) return SDVO_REQ_NONFINITE;
        out->token = argmax_row(pb, row);
    } else {
        out->token = r->am[best][r->owner[best][bestk]];
    }
    out->mass = 1.0;
    if (residual_out) {
        for (int x = 0; x < pb->V; ++x) residual_out[x] = 0.0;
        residual_out[out->token] = 1.0;
    }
    return 0;
}

/* ------------------------------------------------------------------------ */

int sdvo_verify(int mode, const sdvo_problem* pb, int* accept_len, int* accept_draft, int* out_token,
                float* accept_prob, double* residual_mass, double* margin, double* residual_out,
                int* req_status, sdvo_trace* trace)
{
    req_t r;
    int greedy;
    if (!pb || mode < SDVO_MODE_TOKEN || mode > SDVO_MODE_KSEQ) return SDVO_ERR_INVALID;
    if (pb->B < 0 || pb->K < 1 || pb->K > SDVO_MAX_K || pb->L < 0 || pb->L > SDVO_MAX_L || pb->V < 1 ||
        pb->row_stride < pb->V || (pb->dtype != SDVO_F32 && pb->dtype != SDVO_BF16 && pb->dtype != SDVO_F64))
        return SDVO_ERR_INVALID;
    if (isnan(pb->temperature) || pb->temperature < 0.0 || isinf(pb->temperature)) return SDVO_ERR_INVALID;
    if (mode == SDVO_MODE_BLOCK && pb->K != 1) return SDVO_ERR_INVALID;
    greedy = mode == SDVO_MODE_GREEDY || pb->temperature == 0.0;
    if (pb->B == 0) return SDVO_OK;
    if (!pb->target || (pb->L > 0 && !pb->tokens) || !accept_len || !accept_draft || !out_token)
        return SDVO_ERR_INVALID;
    if (!greedy && (!pb->sample_u || (pb->L > 0 && (!pb->draft || !pb->accept_u)))) return SDVO_ERR_INVALID;

    memset(&r, 0, sizeof r);
    r.pb = pb;
    r.greedy = greedy;
    r.tr = trace;
    r.P = (double*)malloc(sizeof(double) * (size_t)pb->V);
    r.Q = (double*)malloc(sizeof(double) * (size_t)pb->V);
    r.R = (double*)malloc(sizeof(double) * (size_t)pb->V);
    if (!r.P || !r.Q || !r.R) {
        free(r.P);
        free(r.Q);
        free(r.R);
        return SDVO_ERR_NOMEM;
    }
    for (int b = 0; b < pb->B; ++b) {
        outcome_t out = {0, 0, -1, 0.0};
        float* ap = accept_prob ? accept_prob + (size_t)b * pb->K * pb->L : NULL;
        double* ro = residual_out ? residual_out + (size_t)b * pb->V : NULL;
        int st;
        r.b = b;
        r.Lb = pb->lengths ? pb->lengths[b] : pb->L;
        r.margin = INFINITY;
        if (ap) memset(ap, 0, sizeof(float) * (size_t)pb->K * pb->L);
        if (ro) memset(ro, 0, sizeof(double) * (size_t)pb->V);
        st = request_status(&r);
        if (st == 0) {
            if (greedy) st = run_greedy(&r, ap, &out, ro);
            else if (mode == SDVO_MODE_TOKEN) st = run_token(&r, ap, &out, ro);
            else if (mode == SDVO_MODE_BLOCK) st = run_block(&r, ap, &out, ro);
            else if (mode == SDVO_MODE_KSEQ) st = run_kseq(&r, ap, &out, ro);
            else st = run_multidraft(&r, ap, &out, ro);
            if (st) { /* the decision ended at a leaf with an unusable row */
                out.tau = out.kstar = 0;
                out.token = -1;
                out.mass = 0.0;
                if (ro) memset(ro, 0, sizeof(double) * (size_t)pb->V);
            }
        }
        if (st && ap) memset(ap, 0, sizeof(float) * (size_t)pb->K * pb->L);
        accept_len[b] = out.tau;
        accept_draft[b] = out.kstar;
        out_token[b] = out.token;
        if (residual_mass) residual_mass[b] = st ? 0.0 : out.mass;
        if (margin) margin[b] = r.margin;
        if (req_status) req_status[b] = st;
    }
    free(r.P);
    free(r.Q);
    free(r.R);
    return SDVO_OK;
}

long long sdvo_prefix_index(const int* tokens, int j, int V)
{
    long long off = 0, pw = 1, num = 0;
    for (int i = 0; i < j; ++i) {
        off += pw;
        pw *= V;
    }
    for (int i = 0; i < j; ++i) num = num * V + tokens[i];
    return off + num;
}

/* ------------------------------------------------------------------------ */
/* draft-token sampling                                                      */

int sdvo_sample_rows(int n_rows, int V, long long row_stride, int dtype, double temperature,
                     const void* logits, int n_samples, const double* u, int* tokens, double* margin,
                     int* row_status)
{
    if (n_rows < 0 || V < 1 || row_stride < V || n_samples < 0 || (dtype != SDVO_F32 && dtype != SDVO_BF16) ||
        !(temperature >= 0.0) || isinf(temperature))
        return SDVO_ERR_INVALID;
    if (n_rows == 0 || n_samples == 0) return SDVO_OK;
    if (!logits || !tokens || (temperature > 0.0 && !u)) return SDVO_ERR_INVALID;
    /* the row helpers read V and dtype from a problem */
    sdvo_problem pb;
    memset(&pb, 0, sizeof pb);
    pb.V = V;
    pb.dtype = dtype;
    pb.row_stride = row_stride;
    double* P = (double*)malloc(sizeof(double) * (size_t)V);
    if (!P) return SDVO_ERR_NOMEM;
    for (int r = 0; r < n_rows; ++r) {
        const unsigned char* row = (const unsigned char*)logits + (size_t)r * (size_t)row_stride * elem_size(dtype);
        int* out = tokens + (size_t)r * n_samples;
        double* mg = margin ? margin + (size_t)r * n_samples : NULL;
        const int ok = row_usable(&pb, row);
        if (row_status) row_status[r] = ok ? 0 : SDVO_REQ_NONFINITE;
        if (!ok) {
            for (int s = 0; s < n_samples; ++s) {
                out[s] = -1;
                if (mg) mg[s] = INFINITY;
            }
            continue;
        }
        if (temperature == 0.0) {
            const int am = argmax_row(&pb, row);
            for (int s = 0; s < n_samples; ++s) {
                out[s] = am;
                if (mg) mg[s] = INFINITY;
            }
            continue;
        }
        softmax(&pb, row, temperature, P);
        double S = 0.0;
        for (int x = 0; x < V; ++x) S += P[x];
        for (int s = 0; s < n_samples; ++s) {
            /* the same inverse CDF as the correction draws of sdvo_verify */
            const double us = u[(size_t)r * n_samples + s];
            double cum = 0.0, lo = 0.0, hi = INFINITY, last_prev = 0.0;
            int chosen = -1, last = -1;
            for (int x = 0; x < V; ++x) {
                if (P[x] > 0.0) {
                    double prev = cum;
                    cum += P[x];
                    last = x;
                    last_prev = prev;
                    if (cum > us * S) {
                        chosen = x;
                        lo = prev / S;
                        hi = cum / S;
                        break;
                    }
                }
            }
            if (chosen < 0) {
                chosen = last;
                lo = last_prev / S;
                hi = INFINITY;
            }
            out[s] = chosen;
            if (mg) mg[s] = fmin(us - lo, hi - us);
        }
    }
    free(P);
    return SDVO_OK;
}


/* ------------------------------------------------------------------------ */
/* the target model's LM head                                                */

int sdvo_lm_head_logits(int M, int V, int d, const void* hidden, const void* lm_head, double* logits,
                        long long out_stride)
{
    if (M < 0 || V < 1 || d < 1 || out_stride < V) return SDVO_ERR_INVALID;
    if (M == 0) return SDVO_OK;
    if (!hidden || !lm_head || !logits) return SDVO_ERR_INVALID;
    const uint16_t* h = (const uint16_t*)hidden;
    const uint16_t* w = (const uint16_t*)lm_head;
    for (int r = 0; r < M; ++r) {
        const uint16_t* hr = h + (size_t)r * (size_t)d;
        for (int x = 0; x < V; ++x) {
            const uint16_t* wx = w + (size_t)x * (size_t)d;
            double s = 0.0;
            for (int i = 0; i < d; ++i) s += bf16_value(hr[i]) * bf16_value(wx[i]);
            logits[(size_t)r * (size_t)out_stride + x] = s;
        }
    }
    return SDVO_OK;
}
