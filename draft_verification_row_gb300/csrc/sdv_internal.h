// sdv_internal.h -- declarations shared by the host API (sdv_api.cu) and
// the kernels (sdv_kernels.cu, sdv_stream.cu, sdv_sample.cu).  Not part of
// the public interface.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

#include "sdv.h"

namespace sdv {

// Per-call scratch, carved out of the caller's workspace.  Node and draw
// records are indexed by slot s = (b * (L + 1) + j) * K + k: the node of
// depth j owned by draft k (valid when k is the lowest draft with that
// prefix), and the draw of draft k at depth j.
struct Workspace {
    float* a;              // draw acceptance probability a (token / multidraft)
    float* h;              // node block acceptance probability h_v
    float* S;              // node residual mass S_n
    float2* wt;            // node weight {1 - p_v, p_v}, written together (one 8-byte store)
                           //   by the parent's draw; .x below 0 until then: the child's flag.
                           //   Both are kept so that neither loses its digits: 1 - p_v when
                           //   p_v is near 1, p_v when it is small
    float* prm;            // node residual for the correction draw: [slot][6] =
                           //   -(M_T c), -(M_D c), aT = p / Z_T, aD / aT, R_n(x*), floor
                           //   (the residual is aT max(e_T - (aD/aT) e_D, floor e_T))
    int* xs;               // node shared dominant token x* (or -1)
    int* am;               // node argmax (greedy)
    unsigned char* owner;  // lowest draft sharing draft k's first j tokens
    int* req;              // [B] request status bits
    int* left;             // [B] inner nodes the node kernel has still to finish (set by the prep kernel)
    int* nodes;            // [L+1][B*K] node slots by depth, listed by the prep kernel: nodes
                           //   with several draws from the front, one-draw nodes from the back
    int* ncount;           // [2][L+1] nodes per depth (several draws, one draw), then the
                           //   node kernel's work counter
};

struct Problem {
    int B, K, L, V;
    long long stride;
    int dtype;
    int mode;       // SDV_MODE_*; greedy when temperature == 0
    float c;        // log2(e) / T
    const void* target;
    const void* leaf_target;  // where leaf rows (depth L_b) are read from, if not target (may be mapped host memory)
    const void* draft;
    const int* tokens;
    const int* lengths;
    const float* accept_u;
    const float* sample_u;
    int* accept_len;
    int* accept_draft;
    int* out_token;
    float* accept_prob;
    float* residual_mass;
    int* device_status;
    int* leaf_pending;  // greedy with the LM head: [B] end leaf slot whose argmax is still to come, or -1
    float* residual_out;  // [B][V] or NULL: the normalised distribution each correction was drawn from
    unsigned long long wait_ns;  // limit of every bounded device wait, in nanoseconds
    Workspace ws;
};

__host__ __device__ inline size_t slot_count(int B, int K, int L) { return (size_t)B * (size_t)(L + 1) * (size_t)K; }

// Kernel launchers (sdv_kernels.cu, sdv_stream.cu); each returns a cudaError_t.
cudaError_t launch_prep(const Problem& pb, cudaStream_t st);
cudaError_t launch_argmax(const Problem& pb, cudaStream_t st);

// The rows verification reads, gathered from host memory the device can
// address (mapped, pinned) into device tensors (sdv_kernels.cu).
struct GatherArgs {
    int B, K, L;
    int leaves;  // 1: target rows down to depth L_b; 0: inner rows only (depth < L_b)
    long long row_bytes;
    const void* host_target;
    const void* host_draft;
    const int* tokens;   // device
    const int* lengths;  // device, or NULL
    void* target;
    void* draft;
};
cudaError_t launch_gather_rows(const GatherArgs& a, cudaStream_t st);
cudaError_t launch_stream(const Problem& pb, cudaStream_t st);

// Draft-token sampling (sdv_sample.cu): n_samples draws per row.
struct SampleArgs {
    int n_rows, V, n_samples, dtype;
    long long stride;
    float c;  // log2(e) / T; 0 means T = 0 (argmax)
    const void* logits;
    const float* u;  // [n_rows][n_samples], unread when c == 0
    int* tokens;     // [n_rows][n_samples]
    int* device_status;
};
cudaError_t launch_sample_rows(const SampleArgs& a, cudaStream_t st);
// Per request: the decision, then the correction (or bonus) draw at its end
// node (sdv_sample.cu).
// after_nodes: launched right after the node kernel, as its programmatic
// dependent; each CTA waits for its request's nodes (Workspace::left).
cudaError_t launch_finish(const Problem& pb, bool greedy, cudaStream_t st, bool after_nodes = false);

// The target model's LM head on the tensor cores (sdv_lmhead.cu):
// logits = hidden . W^T over the hidden size d, bf16 in, fp32 accumulate.
enum { LM_EPI_ARGMAX = 0, LM_EPI_LOGITS = 1, LM_EPI_ROWS_BF16 = 2 };
struct LmArgs {
    int rows;                  // rows of the A operand (used when rows_dev is NULL)
    const int* rows_dev;       // device row count, written by an earlier launch, or NULL
    int V, d;
    unsigned long long* keys;  // ARGMAX: [rows] (maximum, first index) keys, zeroed beforehand
    float* logits;             // LOGITS: [rows][out_stride] fp32
    void* out_bf16;            // ROWS_BF16: bf16 rows of out_stride elements; row r goes to row dest_row[r]
    const int* dest_row;
    long long out_stride;
    int* device_status;
};
// hidden: [hidden_rows][d] bf16 (the A operand); lm_head: [V][d] bf16.
cudaError_t launch_lm_head(const void* hidden, long long hidden_rows, const void* lm_head, const LmArgs& a,
                           int epi, cudaStream_t st);
size_t lm_head_smem_bytes();
// 1: the LM head runs as one CTA per tile even where CTA pairs fit (a test
// hook: the pair form is the default, the one-CTA form its fallback).
extern int g_lm_single_cta;

// Greedy verification fused into the LM head: the trie nodes' hidden rows,
// gathered into the A operand, and their argmax keys.
struct LmRows {
    int d;
    const void* hidden;        // [B][K][L+1][d] bf16
    void* rows;                // [slots][d] bf16: the nodes' hidden rows, contiguous
    int* compact;              // [slots]: node slot -> its row
    int* count;                // rows listed
    unsigned long long* keys;  // [slots]
    int leaves;                // 1: list the leaves (depth L_b) too
    int* row_of;               // [slots] or NULL: each listed row's index in [B][K][L+1]
    // the end leaves the decision reached, one per request at most
    void* leaf_rows;                // [B][d] bf16
    int* leaf_req;                  // [B]: request of each listed leaf
    int* leaf_count;
    unsigned long long* leaf_keys;  // [B]
};
cudaError_t launch_lm_rows(const Problem& pb, const LmRows& r, cudaStream_t st);
cudaError_t launch_lm_argmax(const Problem& pb, const LmRows& r, cudaStream_t st);
cudaError_t launch_lm_leaf_rows(const Problem& pb, const LmRows& r, cudaStream_t st);
cudaError_t launch_lm_leaf_token(const Problem& pb, const LmRows& r, cudaStream_t st);

// The node kernel's launch shape: persistent CTAs per SM, threads per CTA
// and dynamic shared memory.
int stream_ctas_per_sm();
int stream_threads();
size_t stream_smem_bytes();

}  // namespace sdv
