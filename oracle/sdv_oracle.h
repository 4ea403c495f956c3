/*
 * sdv_oracle.h -- plain CPU oracle for batched speculative-decoding
 * verification.
 *
 * TEST INFRASTRUCTURE ONLY.  This code exists to check the CUDA library
 * against a slow, obviously correct restatement of the method.  Only the
 * tests, the smoke check and the bench's CPU-baseline leg may load it; the
 * product path never calls it and shares no code, header or table with it.
 *
 * Arithmetic: IEEE double throughout; bf16 logits are decoded exactly.
 * Single-threaded.  No blocking, fusion or reordering beyond what each
 * definition states.
 *
 * Sources (web summaries of the papers; no formula is printed on them, so
 * the steps below are the published algorithms restated):
 *   [SD]   standard speculative sampling, as named in
 *          "SpecTr-GBV: Multi-Draft Block Verification Accelerating
 *          Speculative Decoding", section 1 (problem definition), and
 *          "MineDraft: A Framework for Batch Parallel Speculative Decoding",
 *          section 1 (het probleem).
 *   [GBV]  greedy block verification, named in the SpecTr-GBV page, section 1
 *          (the block-verification bullet).
 *   [SPECTR] per-position multi-draft verification, SpecTr-GBV page,
 *          section 1 (the multi-draft bullet).
 *   [ALG1] SpecTr-GBV, SpecTr-GBV page, section 2, "algorithmic procedure",
 *          steps 1-5 (Eq. 2, Eq. 4 and Algorithm 2 are referred to but not
 *          printed; the reading used here is the residual recursion
 *          documented in sdv_oracle.c).
 */
#ifndef SDV_ORACLE_H
#define SDV_ORACLE_H

#ifdef __cplusplus
extern "C" {
#endif

#define SDVO_MAX_K 16
#define SDVO_MAX_L 16

enum { SDVO_F32 = 0, SDVO_BF16 = 1, SDVO_F64 = 2 };
enum { SDVO_MODE_TOKEN = 0, SDVO_MODE_GREEDY = 1, SDVO_MODE_BLOCK = 2, SDVO_MODE_MULTIDRAFT = 3, SDVO_MODE_KSEQ = 4 };
enum { SDVO_OK = 0, SDVO_ERR_INVALID = 1, SDVO_ERR_UNSUPPORTED = 2, SDVO_ERR_NOMEM = 3 };
/* per-request data status bits (same meaning as the CUDA library's) */
enum { SDVO_REQ_BAD_LENGTH = 1, SDVO_REQ_BAD_TOKEN = 2, SDVO_REQ_NONFINITE = 4 };

/* One batch.  Layouts (row-major, all host memory):
 *   target   [B][K][L+1][row_stride]  f32, bf16 bits or f64 (the f64 form
 *                                     carries the LM head's exact logits)
 *   draft    [B][K][L][row_stride]
 *   tokens   [B][K][L]                int32, drafted token X^k_{j+1} at [b][k][j]
 *   lengths  [B] in 0..L, or NULL (= L for every request)
 *   accept_u [B][K][L]                uniforms in [0,1) (double)
 *   sample_u [B][K][L+1]              uniforms in [0,1) (double)
 * Row (b,k,j) holds the logits conditioned on draft k's first j tokens.
 * Row 0 is the request's context row; only draft 0's copy is read. */
typedef struct {
    int B, K, L, V;
    long long row_stride;
    int dtype;
    double temperature;
    const void* target;
    const void* draft;
    const int* tokens;
    const int* lengths;
    const double* accept_u;
    const double* sample_u;
} sdvo_problem;

/* Trace of every comparison between a uniform and a threshold, in the order
 * made.  kind 0: accept test "accept_u[index] <= lo".  kind 1: inverse-CDF
 * sample that mapped sample_u[index] into the interval [lo, hi). */
typedef struct { int kind; int index; double lo, hi; } sdvo_trace_entry;
typedef struct { sdvo_trace_entry* e; int cap; int n; } sdvo_trace;

/* Verify every request.  Outputs ([B] unless stated; optional ones may be
 * NULL):
 *   accept_len, accept_draft, out_token
 *   accept_prob    [B][K][L] float: threshold of each draft position
 *   residual_mass  [B]: mass of the unnormalised distribution out_token was
 *                  drawn from (1 for greedy)
 *   margin         [B]: smallest |u - threshold| (or distance of u to the
 *                  chosen CDF interval's ends) over the decisions taken
 *   residual_out   [B][V]: the normalised distribution out_token was drawn from
 *   req_status     [B]: SDVO_REQ_* bits (0 = valid request)
 *   trace          comparisons made (meaningful for B == 1)
 * Returns SDVO_OK or an SDVO_ERR_* code for invalid arguments. */
int sdvo_verify(int mode, const sdvo_problem* pb,
                int* accept_len, int* accept_draft, int* out_token,
                float* accept_prob, double* residual_mass, double* margin,
                double* residual_out, int* req_status, sdvo_trace* trace);

/* Exact output distribution of one request (B == 1) over its uniforms: the
 * uniform cube is split at every threshold the oracle reports until the
 * outcome is constant on each box.  out_prob has (L+1)*K*V entries indexed
 * [tau][k*][token].  Returns SDVO_OK or an error code. */
int sdvo_exact_outcomes(int mode, const sdvo_problem* pb, double* out_prob);

/* Exact P(tau = i), i = 0..L, of one request (B == 1) over its accept
 * uniforms: the integration of sdvo_exact_outcomes with the draws'
 * uniforms left whole (tau is settled before the correction is drawn).
 * E[tau] = sum_i i tau_prob[i] is the expected accepted length for the
 * request's fixed drafts.  Returns SDVO_OK or an error code. */
int sdvo_exact_accept_len(int mode, const sdvo_problem* pb, double* tau_prob);

/* Exact distribution of the emitted stream (accepted prefix + correction
 * token) of a prefix-consistent toy model, over all K-tuples of i.i.d.
 * drafts of length L and over the uniforms.
 *   tgt_tab, dft_tab  [n_prefix][V] f32 logits for every prefix of length
 *                     0..L (prefix index: see sdvo_prefix_index)
 *   q_tab             [n_prefix][V] double: draft sampling probabilities
 *   stream_prob       [n_prefix(L+1)] accumulated P(emitted stream == s),
 *                     indexed by sdvo_prefix_index over lengths 0..L+1
 *   tau_prob          [L+1] P(tau == i)
 * Returns SDVO_OK or an error code. */
int sdvo_exact_streams(int mode, int V, int K, int L, double temperature,
                       const float* tgt_tab, const float* dft_tab, const double* q_tab,
                       double* stream_prob, double* tau_prob);

/* Draft-token sampling: n_samples independent draws from each row's
 * distribution softmax(logits / T), the step before verification in which a
 * draft model proposes its tokens ("SpecTr-GBV: Multi-Draft Block
 * Verification Accelerating Speculative Decoding", section 1: every draft
 * token is drawn from the draft model's distribution).
 *   logits   [n_rows][row_stride]  f32 or bf16 bits; columns >= V unread
 *   u        [n_rows][n_samples]   uniforms in [0,1) (double)
 *   tokens   [n_rows][n_samples]   out: the inverse-CDF draw of each uniform:
 *            the first token in index order whose running sum exceeds u*S
 *            (S the row's total), else the last token of nonzero mass;
 *            T = 0: the row's argmax (lowest index on ties) for every sample
 *   margin   [n_rows][n_samples]   out, may be NULL: distance of u to the
 *            ends of the chosen token's CDF interval (infinite at T = 0)
 *   row_status [n_rows]            out, may be NULL: SDVO_REQ_NONFINITE for a
 *            row with NaN, +Inf or no finite logit (its tokens are -1)
 * Returns SDVO_OK, SDVO_ERR_INVALID or SDVO_ERR_NOMEM. */
int sdvo_sample_rows(int n_rows, int V, long long row_stride, int dtype, double temperature,
                     const void* logits, int n_samples, const double* u, int* tokens, double* margin,
                     int* row_status);

/* The target model's LM head, the last step of the target pass whose output
 * verification consumes ("Speculative Decoding: Performance or Illusion?",
 * section 3.2: verification is the target model's pass over the drafts):
 *   logits[r][x] = sum over i < d of hidden[r][i] * lm_head[x][i]
 * in double.  bf16 inputs are decoded exactly and each product of two bf16
 * values is exact in double; the sum runs in index order.
 *   hidden   [M][d]           bf16 bits
 *   lm_head  [V][d]           bf16 bits (one row per vocabulary entry)
 *   logits   [M][out_stride]  double; columns >= V are not written
 * Verification fused into the LM head is sdvo_verify on these logits, passed
 * as SDVO_F64 rows.  Returns SDVO_OK or SDVO_ERR_INVALID. */
int sdvo_lm_head_logits(int M, int V, int d, const void* hidden, const void* lm_head, double* logits,
                        long long out_stride);

/* Index of a prefix of length j: all prefixes of length < j come first,
 * then the base-V number of the tokens (first token most significant). */
long long sdvo_prefix_index(const int* tokens, int j, int V);

#ifdef __cplusplus
}
#endif
#endif
