/*
 * sdv.h -- batched speculative-decoding verification on GB300 (sm_103a).
 *
 * Given, for a batch of B requests, the target and draft logits of every
 * draft position, the drafted tokens and per-position uniforms, each call
 * returns per request the accepted prefix length tau, the index k* of the
 * draft whose prefix was accepted, and the correction (or bonus) token.
 *
 * The verification entry points are the rules named on the source pages:
 *   sdv_verify_token       standard token-level speculative sampling;
 *                          with K > 1 drafts, per-position multi-draft
 *                          verification (recursive rejection sampling over
 *                          the draft trie).  "SpecTr-GBV: Multi-Draft Block
 *                          Verification Accelerating Speculative Decoding",
 *                          section 1 (problem definition, the single-draft
 *                          and SpecTr-style multi-draft bullets);
 *                          "MineDraft: A Framework for Batch Parallel
 *                          Speculative Decoding", section 1.
 *   sdv_verify_greedy      temperature-0 argmax matching (the T = 0 limit
 *                          of every sampling rule).
 *   sdv_verify_block       greedy block verification (GBV) of one draft.
 *                          SpecTr-GBV page, section 1 (block verification
 *                          bullet).
 *   sdv_verify_multidraft  SpecTr-GBV: K i.i.d. drafts verified as blocks,
 *                          acceptance probabilities h_ik, rejected set H,
 *                          residual correction and target adjustment.
 *                          SpecTr-GBV page, section 2 (algorithmic
 *                          procedure, steps 1-5).
 *   sdv_verify_greedy_lm_head  greedy verification fused into the target
 *                          model's LM head: the logits are computed on the
 *                          tensor cores and reduced to argmaxes without
 *                          being stored (declared below).
 *   sdv_verify_kseq        SpecTr's K-SEQ per position, the rule whose
 *                          search for a scaling factor SpecTr-GBV avoids
 *                          (SpecTr-GBV page, sections 3-4); stated below.
 *
 * The pages print none of the formulas; the rules computed are:
 *   P_v = softmax(target_row / T), Q_v = softmax(draft_row / T) at a trie
 *   node v (drafts sharing a prefix share the node and the rows of the
 *   lowest-index draft through it).  At a node of weight p (p = 1 for
 *   sdv_verify_token, and at the root) with draws y_1..y_n (the next tokens
 *   of the drafts through v, in index order):
 *     R_0 = p P_v, D_0 = 1,
 *     a_j = min(R_{j-1}(y_j) / (D_{j-1} Q_v(y_j)), 1)     (1 if D Q = 0)
 *     R_j = max(R_{j-1} - D_{j-1} Q_v, 0), S_j = sum R_j, D_j = 1 - p + S_j
 *   A child first reached by draw j has weight a_j; h_v = S_n / D_n (1 if
 *   D_n = 0) is the block acceptance probability of the sub-block ending
 *   at v; the correction is drawn from R_n / S_n (P_v if S_n = 0).
 *   token:      walk from the root; at each node try the draws in order,
 *               draw j accepted iff accept_u[b][k_j][depth] <= a_j; the
 *               first accepted draw moves to its child; stop when all are
 *               rejected or at depth L_b.
 *   block/multidraft: depth-first over the trie (children in order of first
 *               appearance); a node v at depth d >= 1 is accepted iff
 *               accept_u[b][owner(v)][d-1] <= h_v, tried after its whole
 *               subtree failed; the first accepted node ends the search
 *               (the root if none).  K = 1 gives GBV exactly.
 *   greedy:     a draft position matches iff its token is the row's argmax
 *               (lowest index on ties); the longest matching draft wins
 *               (lowest k on ties); the correction is the argmax of the
 *               row after the accepted prefix.
 *   Sampling:   the correction is the first token x (index order) whose
 *               running sum of the distribution exceeds u * S with
 *               u = sample_u[b][k*][tau] (else the last token of nonzero
 *               mass).  T = 0 in any sampling rule gives the greedy result.
 *
 * Memory and ownership.  Every pointer argument is a device pointer (or
 * host memory registered with CUDA and mapped into the device's address
 * space) owned by the caller; the library allocates nothing and keeps no
 * pointer after the call returns.  Calls are asynchronous on cuda_stream
 * (a cudaStream_t; NULL = the legacy default stream); the caller must keep
 * every buffer alive until the stream has passed the call.  Two calls that
 * share a workspace must not overlap on the GPU.
 *
 * Errors.  The return value reports argument validation and launch errors
 * only (SDV_OK or an SDV_ERR_* code; nothing is launched on error).  Data
 * errors are found on the device: for each request whose length is outside
 * 0..L, whose used tokens are outside [0, V), or one of whose read rows
 * (see target_logits) holds NaN or +Inf or no finite value, the outputs are accept_len = 0,
 * accept_draft = 0, out_token = -1, residual_mass = 0 and accept_prob = 0,
 * and the request's SDV_REQ_* bit is OR-ed into *device_status.  Other
 * requests are unaffected.  Kernels never trap.
 */
#ifndef SDV_H
#define SDV_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SDV_MAX_K 16      /* drafts per request */
#define SDV_MAX_L 16      /* draft tokens per draft */
#define SDV_MAX_V 262144  /* vocabulary size */
#define SDV_MAX_SAMPLES 64 /* draws per row in sdv_sample_rows */

/* logit element types */
enum { SDV_F32 = 0, SDV_BF16 = 1 };

/* modes, for sdv_workspace_bytes */
enum { SDV_MODE_TOKEN = 0, SDV_MODE_GREEDY = 1, SDV_MODE_BLOCK = 2, SDV_MODE_MULTIDRAFT = 3, SDV_MODE_KSEQ = 4 };

/* return codes */
enum {
    SDV_OK = 0,
    SDV_ERR_INVALID = 1,     /* an argument is out of range, misaligned or not device memory */
    SDV_ERR_UNSUPPORTED = 2, /* valid, but this build or this GPU cannot run it */
    SDV_ERR_CUDA = 3,        /* a CUDA runtime call or launch failed */
    SDV_ERR_TIMEOUT = 4,     /* reserved: a device wait ran out (reported in device_status) */
    SDV_ERR_WORKSPACE = 5    /* workspace NULL, misaligned or smaller than sdv_workspace_bytes */
};

/* *device_status bits (OR of all requests) */
enum {
    SDV_REQ_BAD_LENGTH = 1, /* lengths[b] outside 0..L */
    SDV_REQ_BAD_TOKEN = 2,  /* a used draft token outside [0, V) */
    SDV_REQ_NONFINITE = 4,  /* a used row holds NaN or +Inf, or no finite value */
    SDV_DEV_TIMEOUT = 8     /* a bounded device wait gave up; outputs are not valid */
};

/*
 * Arguments shared by the sdv_verify_* entry points.
 *   B, K, L, V   batch size (>= 0), drafts per request (1..SDV_MAX_K), draft
 *                length (0..SDV_MAX_L), vocabulary size (1..SDV_MAX_V).
 *   row_stride   elements between consecutive rows; >= V and a multiple
 *                of 8.  Elements V..row_stride-1 of a row are never read.
 *   dtype        SDV_F32 or SDV_BF16 (both logit tensors).
 *   temperature  T >= 0 and finite; the same T applies to target and draft.
 *   target_logits [B][K][L+1][row_stride], 16-byte aligned.  Row (b,k,j) is
 *                conditioned on draft k's first j tokens.  Only the rows of
 *                trie nodes are read: row (b,k,j) with j <= lengths[b] and k
 *                the lowest-index draft with that prefix (row 0: k = 0).
 *                A leaf's row (j = lengths[b]) is read only if the decision
 *                ends at that leaf, for the token drawn there: a leaf has
 *                no draws (in the sampling rules its residual p P has mass
 *                p whatever P is; greedy matching uses the inner nodes'
 *                argmaxes, and the leaf's is the correction).
 *   draft_logits [B][K][L][row_stride], 16-byte aligned; same rule with
 *                j < lengths[b].  May be NULL when L = 0 or for greedy.
 *   draft_tokens [B][K][L] int32; positions j >= lengths[b] are ignored.
 *   lengths      [B] int32 in 0..L, or NULL for L everywhere.
 *   accept_u     [B][K][L] fp32 uniforms in [0,1); NULL for greedy.
 *   sample_u     [B][K][L+1] fp32 uniforms in [0,1); NULL for greedy.
 * Outputs:
 *   accept_len   [B] int32: tau in 0..lengths[b].
 *   accept_draft [B] int32: k*, the lowest-index draft whose first tau
 *                tokens were accepted (0 when tau = 0).
 *   out_token    [B] int32: correction token (bonus when tau = lengths[b]).
 *   accept_prob  [B][K][L] fp32 or NULL: the threshold each draft position
 *                was (or would have been) tested against -- token: a of
 *                draft k's draw at depth j; block/multidraft: h of the node
 *                ending draft k's first j+1 tokens; greedy: 1 if the token
 *                is its row's argmax else 0.  0 past lengths[b].
 *   residual_mass [B] fp32 or NULL: S_n of the end node, the mass of the
 *                unnormalised distribution the correction was drawn from
 *                (a leaf's is its weight p); 1 for greedy.
 *   device_status [1] int32 or NULL: cleared by the call, then OR of the
 *                SDV_REQ_* / SDV_DEV_* bits.
 *   workspace    device scratch of at least sdv_workspace_bytes(mode, B, K,
 *                L, V) bytes, 256-byte aligned; contents need no
 *                initialisation and are meaningless after the call.
 *   cuda_stream  cudaStream_t to launch on.
 */
#define SDV_VERIFY_ARGS                                                                              \
    int B, int K, int L, int V, long long row_stride, int dtype, float temperature,                  \
        const void *target_logits, const void *draft_logits, const int *draft_tokens,                \
        const int *lengths, const float *accept_u, const float *sample_u, int *accept_len,           \
        int *accept_draft, int *out_token, float *accept_prob, float *residual_mass,                 \
        int *device_status, void *workspace, size_t workspace_bytes, void *cuda_stream

/* Token-level speculative sampling; K > 1: per-position multi-draft. */
int sdv_verify_token(SDV_VERIFY_ARGS);

/* Temperature-0 argmax matching; temperature, draft_logits, accept_u and
 * sample_u are ignored and may be NULL. */
int sdv_verify_greedy(SDV_VERIFY_ARGS);

/* Greedy block verification; requires K == 1 (else SDV_ERR_INVALID). */
int sdv_verify_block(SDV_VERIFY_ARGS);

/* SpecTr-GBV multi-draft block verification. */
int sdv_verify_multidraft(SDV_VERIFY_ARGS);

/* SpecTr's K-SEQ, per position: the rule SpecTr-GBV is compared with, and
 * whose search for a scaling factor rho it avoids (SpecTr-GBV page, sections
 * 3-4; the rule follows SpecTr's published definition).  At a node with n
 * drafts through it (i.i.d. candidates from Q):
 *   beta(rho) = sum_x min(Q(x), P(x) / rho),
 *   gamma(rho) = (1 - (1 - beta)^n) / beta   (n when beta = 0);
 * candidate i (index order) is accepted iff accept_u[b][k_i][depth] <=
 * min(1, P(y_i) / (rho Q(y_i))), the first accepted moves to its child
 * (as in sdv_verify_token); when all are rejected the correction is drawn
 * from P - gamma min(Q, P / rho) (P where that has no mass).  rho: 1 if
 * gamma(1) <= 1, else 10 rounds starting from [lo, hi] = [1, n], each
 * testing lo + (hi - lo) i / 4 for i = 1, 2, 3 against gamma(rho) <= rho
 * and keeping the quarter that ends at the first one that passes (the
 * last quarter if none does); rho is the final hi.  Any such rho keeps the
 * emitted token distributed as P.  accept_prob holds each draw's
 * acceptance probability; residual_mass the end node's (1 - beta)^n.  The
 * search costs one vocabulary pass per round. */
int sdv_verify_kseq(SDV_VERIFY_ARGS);

/* Workspace bytes a call of `mode` with these sizes needs (0 if the sizes
 * are invalid). */
size_t sdv_workspace_bytes(int mode, int B, int K, int L, int V);

/* Static description of a return code (not of device status bits). */
const char *sdv_status_string(int status);

/* Draft-token sampling: the step before verification, in which a draft
 * model proposes its tokens, each drawn from the model's distribution
 * softmax(logits / T) ("SpecTr-GBV: Multi-Draft Block Verification
 * Accelerating Speculative Decoding", section 1).  n_samples independent
 * draws per row (K drafts sharing a prefix draw K tokens from one row).
 *   n_rows       rows (>= 0); V vocabulary size (1..SDV_MAX_V); row_stride
 *                elements between rows (>= V, a multiple of 8); dtype
 *                SDV_F32 or SDV_BF16; temperature T >= 0, finite.
 *   logits       [n_rows][row_stride] device, 16-byte aligned; columns >= V
 *                are never read.
 *   n_samples    draws per row, 1..SDV_MAX_SAMPLES.
 *   u            [n_rows][n_samples] device fp32 uniforms in [0, 1); may be
 *                NULL when T == 0.
 *   tokens       [n_rows][n_samples] device int32 out.  Each draw is the
 *                inverse CDF of its uniform: the first token in index order
 *                whose running sum of probabilities exceeds u * S (S the
 *                row's total), else the last token of nonzero probability.
 *                T == 0: the row's argmax, lowest index on ties.  A row
 *                holding NaN or +Inf, or no finite logit, gives -1.
 *   device_status [1] device int32 or NULL: zeroed, then SDV_REQ_NONFINITE
 *                if some row was unusable (other rows are unaffected).
 *   cuda_stream  the stream to run on (NULL: the default stream).
 * Asynchronous; allocates nothing.  Returns SDV_OK, SDV_ERR_INVALID or
 * SDV_ERR_CUDA.  Element masses are fp32, the row total and the running
 * sums over segments double; a draw whose uniform lies within about 1e-7
 * of a CDF boundary (the fp32 error of the largest masses) may fall on the
 * neighbouring token. */
int sdv_sample_rows(int n_rows, int V, long long row_stride, int dtype, float temperature, const void *logits,
                    int n_samples, const float *u, int *tokens, int *device_status, void *cuda_stream);

/* Launch shape of the node kernel (the one that reads vocabulary rows) for
 * rows of V elements of dtype: CTAs per SM (it is persistent: that many
 * CTAs per SM of the device), threads per CTA and dynamic shared memory per
 * CTA.  For callers that share the GPU with other work.
 * Needs no GPU.  Returns SDV_OK or SDV_ERR_INVALID (V or dtype out of
 * range). */
int sdv_launch_shape(int V, int dtype, int *ctas_per_sm, int *threads, int *smem_bytes);

/* Logits in host memory: verification reads only the rows of trie nodes
 * (see target_logits), so only those need to be on the device.
 * sdv_copy_read_rows copies, per request and draft, the one contiguous range
 * of rows it reads from each tensor: for draft k, target rows f..L_b and
 * draft rows f..L_b-1, where f is the first depth whose node draft k owns
 * (0 for k = 0; else one past the longest prefix it shares with a lower
 * draft).  A leaf's row is among them, since only the decision tells whether
 * its bonus draw needs it.  Requests whose length is outside 0..L get no
 * rows.
 *   host_target, host_draft  the full [B][K][L+1][row_stride] and
 *                [B][K][L][row_stride] tensors in host memory (pinned, for
 *                asynchronous copies); tokens [B][K][L] and lengths [B] (or
 *                NULL) in host memory, read on the host during the call.
 *   target, draft  device tensors of the same shapes; rows not copied keep
 *                whatever they held (they are never read).
 *   cuda_stream  the stream the copies are queued on, one cudaMemcpyAsync
 *                per range.
 *   bytes        out, may be NULL: the bytes queued.
 * Returns SDV_OK, SDV_ERR_INVALID or SDV_ERR_CUDA.  sdv_read_rows_bytes
 * returns the same byte count without copying (no GPU needed). */
int sdv_copy_read_rows(int B, int K, int L, int V, long long row_stride, int dtype, const void *host_target,
                       const void *host_draft, const int *tokens, const int *lengths, void *target, void *draft,
                       void *cuda_stream, long long *bytes);
int sdv_read_rows_bytes(int B, int K, int L, int V, long long row_stride, int dtype, const int *tokens,
                        const int *lengths, long long *bytes);

/* The same rows moved by the GPU itself: one kernel launch, one CTA per
 * (request, draft), reading host memory over the host link with many loads
 * in flight (no per-range copy calls).  host_target and host_draft must be
 * host memory mapped into the device's address space (pinned memory on a
 * UVA system); tokens and lengths (or NULL) device memory, as for the
 * verification calls; target and draft device tensors; all 16-byte
 * aligned.  Asynchronous on cuda_stream.  Returns SDV_OK, SDV_ERR_INVALID
 * (a pointer the device cannot address, misalignment, K > 256) or
 * SDV_ERR_CUDA. */
int sdv_gather_read_rows(int B, int K, int L, int V, long long row_stride, int dtype, const void *host_target,
                         const void *host_draft, const int *tokens, const int *lengths, void *target, void *draft,
                         void *cuda_stream);

/* As sdv_gather_read_rows, without the leaves' target rows: draft k brings
 * target rows [f_k, L_b - 1] and draft rows [f_k, L_b - 1], the rows every
 * decision reads.  A leaf's row (depth L_b) is read only where the decision
 * ends there; sdv_verify_leaves_apart can read those few rows from the host
 * tensor itself. */
int sdv_gather_inner_rows(int B, int K, int L, int V, long long row_stride, int dtype, const void *host_target,
                          const void *host_draft, const int *tokens, const int *lengths, void *target, void *draft,
                          void *cuda_stream);

/* The verification of `mode` (SDV_MODE_*), as its sdv_verify_* entry, with
 * the leaves' target rows (depth lengths[b]) read from leaf_target_logits
 * instead of target_logits.  leaf_target_logits has target_logits' layout
 * ([B][K][L+1][row_stride], same dtype), is 16-byte aligned, and may be
 * host memory mapped into the device's address space: only the leaf rows
 * the decisions end at are read from it (at most one per request), and
 * target_logits' rows at depth lengths[b] are never read.  With the inner
 * rows gathered by sdv_gather_inner_rows, a batch whose logits live in host
 * memory crosses the host link once, without its leaves.  Returns as the
 * sdv_verify_* calls; SDV_ERR_INVALID also for a mode out of range or a
 * leaf_target_logits the device cannot address. */
int sdv_verify_leaves_apart(int mode, SDV_VERIFY_ARGS, const void *leaf_target_logits);

/* The verification of `mode` (SDV_MODE_*), as its sdv_verify_* entry, that
 * also writes, per request, the normalised distribution its correction (or
 * bonus) token was drawn from: the residual of the end node after the
 * target adjustment, R_n / S_n (SpecTr-GBV page, section 2, steps 4-5: the
 * residual distribution of Eq. 4 and Algorithm 2's adjusted target); P_v at
 * a leaf or where S_n = 0; for K-SEQ, P - gamma min(Q, P / rho) normalised;
 * for greedy (or T = 0), the one-hot row of the correction token.  An
 * invalid request (see Errors above) gets a row of zeros.
 *   residual_out [B][V] fp32, device memory, 4-byte aligned, written in
 *                full (no other column); row b is each element's mass over
 *                the total mass the draw used, so it sums to 1 up to fp32
 *                rounding.
 * A debug and test output: it costs one more pass over the end node's rows
 * per request, after the draw.  Returns as the sdv_verify_* calls;
 * SDV_ERR_INVALID also for a mode out of range or a NULL residual_out with
 * B > 0. */
int sdv_verify_residual(int mode, SDV_VERIFY_ARGS, float *residual_out);

/* Fixed scratch of sdv_verify_multidraft_static: 4 MiB of device memory
 * that every GPU loading the library reserves until the process exits. */
#define SDV_STATIC_SCRATCH_BYTES (4u << 20)

/* SpecTr-GBV verification (as sdv_verify_multidraft) for callers that cannot
 * allocate device memory: a plugin whose host framework owns all device
 * memory and passes it only input and output buffers, code running inside a
 * device allocator's own hooks, or a serving loop that forbids cudaMalloc
 * because it can synchronise the device.  The source pages have no
 * counterpart: this is a library convenience.
 *   Arguments and outputs are those of sdv_verify_multidraft, without
 *   workspace and workspace_bytes: the scratch is a fixed device array of
 *   SDV_STATIC_SCRATCH_BYTES inside the library.  A problem whose
 *   sdv_workspace_bytes(SDV_MODE_MULTIDRAFT, B, K, L, V) exceeds that is
 *   rejected with SDV_ERR_WORKSPACE before anything is launched (e.g.
 *   B = 256, K = 8, L = 8 needs about 0.5 MiB).
 *   The first call on a device looks up the array's device address
 *   (cudaGetSymbolAddress) with that device current and keeps it; the first
 *   call after the device's context was destroyed and created again (e.g.
 *   by cudaDeviceReset) looks it up again.  Make those calls before any
 *   stream capture.  Nothing is allocated, then or later.
 *   Every call on a device shares the one array: two calls whose kernels
 *   overlap on the GPU (different streams without ordering, or different
 *   host threads) race and give wrong results.  Nothing in the array needs
 *   to start at zero; each call writes every record before reading it. */
int sdv_verify_multidraft_static(int B, int K, int L, int V, long long row_stride, int dtype, float temperature,
                                 const void *target_logits, const void *draft_logits, const int *draft_tokens,
                                 const int *lengths, const float *accept_u, const float *sample_u,
                                 int *accept_len, int *accept_draft, int *out_token, float *accept_prob,
                                 float *residual_mass, int *device_status, void *cuda_stream);

/* ---------------------------------------------------------------------------
 * The target model's LM head, and greedy verification fused into it.
 *
 * Verification consumes the target model's pass over the drafts
 * ("Speculative Decoding: Performance or Illusion?", section 3.2: that pass
 * is the verification step), and the pass ends in the LM head,
 *   logits[r][x] = sum over i < d of hidden[r][i] * lm_head[x][i],
 * a dense contraction over the hidden size d.  Both calls below compute it
 * on the tensor cores from bf16 inputs with fp32 accumulation; the order in
 * which the d products are summed is the hardware's, so a logit can differ
 * from the exact sum by a few fp32 rounding steps of the products' sizes.
 *
 * sdv_verify_greedy_lm_head applies the greedy rule (as sdv_verify_greedy)
 * to these logits without storing them: each inner trie node's row (one per
 * distinct draft prefix of length 0..L_b - 1) is computed once and reduced
 * in the tensor-core epilogue to its maximum and first index; after the
 * decision, the one leaf row a request ends at (if any) is computed the
 * same way for its correction token.
 *   B, K, L, V   as for sdv_verify_greedy; d hidden size, a multiple of 8 in
 *                8..65536.
 *   hidden       [B][K][L+1][d] bf16: row (b,k,j) is the target model's
 *                final hidden state after draft k's first j tokens (rows of
 *                drafts sharing those tokens are read from the lowest such
 *                draft; rows past L_b are never read).  16-byte aligned.
 *   lm_head      [V][d] bf16, one row per vocabulary entry; 16-byte aligned.
 *   draft_tokens, lengths, accept_len, accept_draft, out_token, accept_prob,
 *   device_status  as for sdv_verify_greedy.  A node whose logits hold NaN
 *                or +Inf marks its request SDV_REQ_NONFINITE.
 *   workspace    device scratch of at least sdv_lm_head_workspace_bytes(B,
 *                K, L, V, d) bytes, 256-byte aligned (it holds the nodes'
 *                hidden rows: about B*K*(L+1)*d*2 bytes).
 * Returns SDV_OK, SDV_ERR_INVALID, SDV_ERR_WORKSPACE, SDV_ERR_UNSUPPORTED (no
 * tensor-map encoder in the driver, or not enough shared memory) or
 * SDV_ERR_CUDA.  The profiling hook brackets the LM-head kernel. */
int sdv_verify_greedy_lm_head(int B, int K, int L, int V, int d, const void *hidden, const void *lm_head,
                              const int *draft_tokens, const int *lengths, int *accept_len, int *accept_draft,
                              int *out_token, float *accept_prob, int *device_status, void *workspace,
                              size_t workspace_bytes, void *cuda_stream);

/* The LM head for the sampling rules, which cannot be fused into it (each
 * residual sweep needs the row's normaliser first, and recomputing a row
 * costs far more than reading it back): every trie node's row, leaves
 * included, is computed once on the tensor cores and written, rounded to
 * bf16 (nearest even), into the verification layout, where any
 * sdv_verify_* call can read it.
 *   B, K, L, V, d, hidden, lm_head, draft_tokens, lengths  as for
 *                sdv_verify_greedy_lm_head.
 *   target_logits [B][K][L+1][row_stride] bf16, 16-byte aligned; row_stride
 *                >= V and a multiple of 8.  Row (b,k,j) is written for each
 *                trie node (j <= lengths[b], k the lowest draft with that
 *                prefix); every other row and the columns past V are left
 *                as they were.
 *   device_status [1] or NULL: zeroed, then SDV_REQ_* bits of requests
 *                with a bad length or token (their rows are not written),
 *                or SDV_DEV_TIMEOUT.
 *   workspace    as for sdv_verify_greedy_lm_head.
 * Returns SDV_OK, SDV_ERR_INVALID, SDV_ERR_WORKSPACE, SDV_ERR_UNSUPPORTED or
 * SDV_ERR_CUDA.  The profiling hook brackets the LM-head kernel. */
int sdv_lm_head_trie_logits(int B, int K, int L, int V, int d, const void *hidden, const void *lm_head,
                            const int *draft_tokens, const int *lengths, void *target_logits, long long row_stride,
                            int *device_status, void *workspace, size_t workspace_bytes, void *cuda_stream);

/* Workspace bytes of sdv_verify_greedy_lm_head and sdv_lm_head_trie_logits;
 * 0 for invalid sizes. */
size_t sdv_lm_head_workspace_bytes(int B, int K, int L, int V, int d);

/* The LM head alone: logits [M][logits_stride] fp32 (columns >= V are not
 * written) from hidden [M][d] and lm_head [V][d], both bf16 and 16-byte
 * aligned; logits_stride >= V and a multiple of 4, logits 16-byte aligned;
 * d as above; V in 1..SDV_MAX_V.  device_status (or NULL) is zeroed and
 * gets SDV_DEV_TIMEOUT if a device wait gave up.  Returns SDV_OK,
 * SDV_ERR_INVALID, SDV_ERR_UNSUPPORTED or SDV_ERR_CUDA. */
int sdv_lm_head_logits(int M, int V, int d, const void *hidden, const void *lm_head, float *logits,
                       long long logits_stride, int *device_status, void *cuda_stream);

/* Profiling hook.  With start and stop both cudaEvent_t handles, every
 * later call made from the calling host thread records `start` on its
 * stream just before its first vocabulary-row kernel (the node kernel, the
 * greedy argmax or the LM head) and `stop` just after it, so that
 * cudaEventElapsedTime gives the time of that kernel alone; NULL, NULL turns
 * it off.  Without the hook, the decision kernel of the sampling rules is
 * launched as the node kernel's programmatic dependent and overlaps its
 * last nodes; with the hook on, the two run one after the other.  The events stay owned by the
 * caller.  Returns SDV_OK, or SDV_ERR_INVALID if exactly one is NULL. */
int sdv_set_profile_events(void *start, void *stop);

#ifdef __cplusplus
}
#endif
#endif
