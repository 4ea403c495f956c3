/*
 * exact.c -- exact output distributions of the oracle, for pinning it.
 * TEST INFRASTRUCTURE ONLY.
 *
 * The oracle's decisions compare each uniform with thresholds that depend
 * only on the logits and the drafted tokens, never on other uniforms.  So
 * the output is constant on any box of the uniform cube that no reported
 * threshold cuts.  The integrator runs the oracle at the centre of a box,
 * reads its comparison trace, and splits the box at the first threshold
 * that falls strictly inside it; a box with no such cut adds its volume to
 * the outcome it produced.  This treats the decision code as a black box:
 * it restates none of the method, so a mistake in the method shows up in
 * the integrated distribution instead of being copied into it.
 */
#include "sdv_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

#define TRACE_CAP 4096

typedef void (*sink_fn)(void* ctx, const int* tokens, int K, int L, int tau, int kstar, int token, double w);

typedef struct {
    int mode;
    sdvo_problem pb; /* B == 1; uniforms point at ua / us */
    double* ua;
    double* us;
    double* lo;
    double* hi;
    int n_acc, n_smp;
    sdvo_trace tr;
    sink_fn sink;
    void* ctx;
    int err;
    int accept_only; /* split at accept-test thresholds only (the draws' uniforms stay whole) */
} integ_t;

static void run_box(integ_t* g, double w);

static void split_at(integ_t* g, int c, double s, double w)
{
    double l = g->lo[c], h = g->hi[c], width = h - l;
    g->hi[c] = s;
    run_box(g, w * (s - l) / width);
    g->hi[c] = h;
    g->lo[c] = s;
    run_box(g, w * (h - s) / width);
    g->lo[c] = l;
}

static void run_box(integ_t* g, double w)
{
    int tau, ks, tk, st, rc;
    if (w <= 0.0 || g->err) return;
    for (int c = 0; c < g->n_acc; ++c) g->ua[c] = 0.5 * (g->lo[c] + g->hi[c]);
    for (int c = 0; c < g->n_smp; ++c) g->us[c] = 0.5 * (g->lo[g->n_acc + c] + g->hi[g->n_acc + c]);
    g->tr.n = 0;
    rc = sdvo_verify(g->mode, &g->pb, &tau, &ks, &tk, NULL, NULL, NULL, NULL, &st, &g->tr);
    if (rc != SDVO_OK || st != 0 || g->tr.n > g->tr.cap) {
        g->err = rc != SDVO_OK ? rc : SDVO_ERR_INVALID;
        return;
    }
    for (int i = 0; i < g->tr.n; ++i) {
        sdvo_trace_entry e = g->tr.e[i];
        int c = e.kind == 0 ? e.index : g->n_acc + e.index;
        if (e.kind == 1 && g->accept_only) continue;
        if (g->lo[c] < e.lo && e.lo < g->hi[c]) {
            split_at(g, c, e.lo, w);
            return;
        }
        if (e.kind == 1 && g->lo[c] < e.hi && e.hi < g->hi[c]) {
            split_at(g, c, e.hi, w);
            return;
        }
    }
    g->sink(g->ctx, g->pb.tokens, g->pb.K, g->pb.L, tau, ks, tk, w);
}

static int integ_init(integ_t* g, int mode, const sdvo_problem* pb)
{
    memset(g, 0, sizeof *g);
    g->mode = mode;
    g->pb = *pb;
    g->pb.B = 1;
    g->n_acc = pb->K * pb->L;
    g->n_smp = pb->K * (pb->L + 1);
    g->ua = (double*)calloc((size_t)g->n_acc + 1, sizeof(double));
    g->us = (double*)calloc((size_t)g->n_smp, sizeof(double));
    g->lo = (double*)calloc((size_t)(g->n_acc + g->n_smp), sizeof(double));
    g->hi = (double*)calloc((size_t)(g->n_acc + g->n_smp), sizeof(double));
    g->tr.e = (sdvo_trace_entry*)calloc(TRACE_CAP, sizeof(sdvo_trace_entry));
    g->tr.cap = TRACE_CAP;
    if (!g->ua || !g->us || !g->lo || !g->hi || !g->tr.e) return SDVO_ERR_NOMEM;
    g->pb.accept_u = g->ua;
    g->pb.sample_u = g->us;
    return SDVO_OK;
}

static void integ_reset_box(integ_t* g)
{
    for (int c = 0; c < g->n_acc + g->n_smp; ++c) {
        g->lo[c] = 0.0;
        g->hi[c] = 1.0;
    }
}

static void integ_free(integ_t* g)
{
    free(g->ua);
    free(g->us);
    free(g->lo);
    free(g->hi);
    free(g->tr.e);
}

/* ---- one fixed request -------------------------------------------------- */

typedef struct {
    double* out;
    int K, V;
} outcome_sink_t;

static void outcome_sink(void* ctx, const int* tokens, int K, int L, int tau, int kstar, int token, double w)
{
    outcome_sink_t* s = (outcome_sink_t*)ctx;
    (void)tokens;
    (void)K;
    (void)L;
    s->out[((size_t)tau * s->K + kstar) * s->V + token] += w;
}

int sdvo_exact_outcomes(int mode, const sdvo_problem* pb, double* out_prob)
{
    integ_t g;
    outcome_sink_t s;
    int rc;
    if (!pb || pb->B != 1 || !out_prob) return SDVO_ERR_INVALID;
    rc = integ_init(&g, mode, pb);
    if (rc == SDVO_OK) {
        memset(out_prob, 0, sizeof(double) * (size_t)(pb->L + 1) * pb->K * pb->V);
        s.out = out_prob;
        s.K = pb->K;
        s.V = pb->V;
        g.sink = outcome_sink;
        g.ctx = &s;
        integ_reset_box(&g);
        run_box(&g, 1.0);
        rc = g.err;
    }
    integ_free(&g);
    return rc;
}

/* ---- accepted length only ------------------------------------------------ */

/* The accepted length is settled by the accept tests alone: every rule
 * takes them all before it draws the correction.  Integrating over the
 * accept uniforms only, with the draws' uniforms left whole, gives
 * P(tau = i) exactly at the cost of one oracle run per decision path. */
static void tau_sink(void* ctx, const int* tokens, int K, int L, int tau, int kstar, int token, double w)
{
    double* out = (double*)ctx;
    (void)tokens;
    (void)K;
    (void)L;
    (void)kstar;
    (void)token;
    out[tau] += w;
}

int sdvo_exact_accept_len(int mode, const sdvo_problem* pb, double* tau_prob)
{
    integ_t g;
    int rc;
    if (!pb || pb->B != 1 || !tau_prob) return SDVO_ERR_INVALID;
    rc = integ_init(&g, mode, pb);
    if (rc == SDVO_OK) {
        memset(tau_prob, 0, sizeof(double) * (size_t)(pb->L + 1));
        g.sink = tau_sink;
        g.ctx = tau_prob;
        g.accept_only = 1;
        integ_reset_box(&g);
        run_box(&g, 1.0);
        rc = g.err;
    }
    integ_free(&g);
    return rc;
}

/* ---- toy model: all draft tuples ---------------------------------------- */

typedef struct {
    double* stream_prob;
    double* tau_prob;
    int V;
} stream_sink_t;

static void stream_sink(void* ctx, const int* tokens, int K, int L, int tau, int kstar, int token, double w)
{
    stream_sink_t* s = (stream_sink_t*)ctx;
    int st[SDVO_MAX_L + 1];
    (void)K;
    for (int i = 0; i < tau; ++i) st[i] = tokens[kstar * L + i];
    st[tau] = token;
    s->stream_prob[sdvo_prefix_index(st, tau + 1, s->V)] += w;
    s->tau_prob[tau] += w;
}

int sdvo_exact_streams(int mode, int V, int K, int L, double temperature, const float* tgt_tab,
                       const float* dft_tab, const double* q_tab, double* stream_prob, double* tau_prob)
{
    integ_t g;
    stream_sink_t s;
    sdvo_problem pb;
    int rc, n_digits = K * L;
    int* tokens;
    float *trows, *drows;
    long long n_stream;
    if (V < 1 || K < 1 || K > SDVO_MAX_K || L < 0 || L > SDVO_MAX_L || !tgt_tab || !dft_tab || !q_tab ||
        !stream_prob || !tau_prob)
        return SDVO_ERR_INVALID;
    {
        int full[SDVO_MAX_L + 1];
        for (int i = 0; i <= L; ++i) full[i] = V - 1;
        n_stream = sdvo_prefix_index(full, L + 1, V) + 1;
    }
    tokens = (int*)calloc((size_t)(n_digits + 1), sizeof(int));
    trows = (float*)calloc((size_t)K * (L + 1) * V, sizeof(float));
    drows = (float*)calloc((size_t)K * (L + 1) * V, sizeof(float));
    memset(&pb, 0, sizeof pb);
    pb.B = 1;
    pb.K = K;
    pb.L = L;
    pb.V = V;
    pb.row_stride = V;
    pb.dtype = SDVO_F32;
    pb.temperature = temperature;
    pb.target = trows;
    pb.draft = drows;
    pb.tokens = tokens;
    pb.lengths = NULL;
    rc = (tokens && trows && drows) ? integ_init(&g, mode, &pb) : SDVO_ERR_NOMEM;
    if (rc != SDVO_OK) {
        free(tokens);
        free(trows);
        free(drows);
        return rc;
    }
    memset(stream_prob, 0, sizeof(double) * (size_t)n_stream);
    memset(tau_prob, 0, sizeof(double) * (size_t)(L + 1));
    s.stream_prob = stream_prob;
    s.tau_prob = tau_prob;
    s.V = V;
    g.sink = stream_sink;
    g.ctx = &s;
    for (;;) {
        double w = 1.0;
        /* rows and weight of this tuple: draft k's token j was drawn from
           q(. | its first j tokens) */
        for (int k = 0; k < K && w > 0.0; ++k) {
            for (int j = 0; j <= L; ++j) {
                long long pi = sdvo_prefix_index(tokens + k * L, j, V);
                memcpy(trows + ((size_t)k * (L + 1) + j) * V, tgt_tab + (size_t)pi * V, sizeof(float) * V);
                if (j < L) {
                    memcpy(drows + ((size_t)k * L + j) * V, dft_tab + (size_t)pi * V, sizeof(float) * V);
                    w *= q_tab[(size_t)pi * V + tokens[k * L + j]];
                }
            }
        }
        if (w > 0.0) {
            integ_reset_box(&g);
            run_box(&g, w);
            if (g.err) break;
        }
        /* next tuple (odometer over K*L digits) */
        {
            int d = n_digits - 1;
            while (d >= 0 && tokens[d] == V - 1) tokens[d--] = 0;
            if (d < 0) break;
            tokens[d]++;
        }
    }
    rc = g.err;
    integ_free(&g);
    free(tokens);
    free(trows);
    free(drows);
    return rc;
}
