// sdv_api.cu -- the C-ABI of include/sdv.h: argument checks, workspace
// layout and the launch sequence of each verification rule.
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>

#include "sdv_internal.h"

namespace sdv {
namespace {

constexpr size_t kAlign = 256;

size_t align_up(size_t n) { return (n + kAlign - 1) / kAlign * kAlign; }

bool sizes_ok(int B, int K, int L, int V)
{
    // node slots are kept in 30 bits (the decision's end-node record)
    return B >= 0 && K >= 1 && K <= SDV_MAX_K && L >= 0 && L <= SDV_MAX_L && V >= 1 && V <= SDV_MAX_V &&
           slot_count(B, K, L) < ((size_t)1 << 30);
}

size_t workspace_size(int B, int K, int L)
{
    const size_t n = slot_count(B, K, L);
    return 5 * align_up(n * 4) + align_up(n * 8) + align_up(n * 6 * 4) + align_up(n) + 2 * align_up((size_t)B * 4) +
           align_up((size_t)(L + 1) * B * K * 4) + align_up((size_t)(2 * L + 3) * 4);
}

// The hidden size of the LM head: whole 16-byte units per row (TMA row pitch).
bool lm_d_ok(int d) { return d >= 8 && d % 8 == 0 && d <= (1 << 16); }

// LM-head calls: the verification workspace, then the node rows of the LM
// head (compact map, row count, argmax keys, hidden rows, row indices),
// then the end leaves (pending slot and request per leaf, count, keys,
// hidden rows).
size_t lm_workspace_size(int B, int K, int L, int d)
{
    const size_t n = slot_count(B, K, L);
    const size_t nb = (size_t)B;
    return workspace_size(B, K, L) + align_up(n * 4) + align_up(4) + align_up(n * 8) + align_up(n * (size_t)d * 2) +
           align_up(n * 4) + 2 * align_up(nb * 4) + align_up(4) + align_up(nb * 8) + align_up(nb * (size_t)d * 2);
}

Workspace carve(void* base, int B, int K, int L)
{
    const size_t n = slot_count(B, K, L);
    char* p = static_cast<char*>(base);
    Workspace w;
    w.a = reinterpret_cast<float*>(p);
    p += align_up(n * 4);
    w.h = reinterpret_cast<float*>(p);
    p += align_up(n * 4);
    w.S = reinterpret_cast<float*>(p);
    p += align_up(n * 4);
    w.wt = reinterpret_cast<float2*>(p);
    p += align_up(n * 8);
    w.prm = reinterpret_cast<float*>(p);
    p += align_up(n * 6 * 4);
    w.xs = reinterpret_cast<int*>(p);
    p += align_up(n * 4);
    w.am = reinterpret_cast<int*>(p);
    p += align_up(n * 4);
    w.owner = reinterpret_cast<unsigned char*>(p);
    p += align_up(n);
    w.req = reinterpret_cast<int*>(p);
    p += align_up((size_t)B * 4);
    w.left = reinterpret_cast<int*>(p);
    p += align_up((size_t)B * 4);
    w.nodes = reinterpret_cast<int*>(p);
    p += align_up((size_t)(L + 1) * B * K * 4);
    w.ncount = reinterpret_cast<int*>(p);
    return w;
}

// Device memory of the current device, managed memory, or host memory
// mapped into the device's address space.
bool device_accessible(const void* ptr)
{
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, ptr) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    if (a.type == cudaMemoryTypeDevice) return a.device == dev;
    if (a.type == cudaMemoryTypeManaged) return true;
    if (a.type == cudaMemoryTypeHost) return a.devicePointer == ptr;
    return false;
}

bool aligned(const void* p, size_t n) { return (reinterpret_cast<uintptr_t>(p) % n) == 0; }

// profiling hook (sdv_set_profile_events): per host thread
thread_local cudaEvent_t g_prof_start = nullptr;
thread_local cudaEvent_t g_prof_stop = nullptr;

// limit of the bounded device waits (sdv_testing_set_wait_limit): per host
// thread; 0 means the default of 2 s
constexpr unsigned long long kDefaultWaitNs = 2000000000ull;
thread_local unsigned long long g_wait_ns = 0;

bool prof_record(cudaEvent_t e, cudaStream_t st) { return !e || cudaEventRecord(e, st) == cudaSuccess; }

int verify(int mode, int B, int K, int L, int V, long long row_stride, int dtype, float temperature,
           const void* target_logits, const void* draft_logits, const int* draft_tokens, const int* lengths,
           const float* accept_u, const float* sample_u, int* accept_len, int* accept_draft, int* out_token,
           float* accept_prob, float* residual_mass, int* device_status, void* workspace,
           size_t workspace_bytes, void* cuda_stream, const void* leaf_target = nullptr,
           float* residual_out = nullptr, bool skip_roots = false)
{
    if (!sizes_ok(B, K, L, V)) return SDV_ERR_INVALID;
    if (row_stride < V || row_stride % 8 != 0) return SDV_ERR_INVALID;
    if (dtype != SDV_F32 && dtype != SDV_BF16) return SDV_ERR_INVALID;
    if (!(temperature >= 0.f) || std::isinf(temperature)) return SDV_ERR_INVALID;
    if (mode == SDV_MODE_BLOCK && K != 1) return SDV_ERR_INVALID;
    const bool greedy = mode == SDV_MODE_GREEDY || temperature == 0.f;
    const float c = greedy ? 0.f : (float)(1.4426950408889634 / (double)temperature);
    if (!greedy && !std::isfinite(c)) return SDV_ERR_INVALID;
    cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);

    if (device_status && !device_accessible(device_status)) return SDV_ERR_INVALID;
    if (B == 0) {
        if (device_status && cudaMemsetAsync(device_status, 0, sizeof(int), st) != cudaSuccess) return SDV_ERR_CUDA;
        return SDV_OK;
    }

    // required pointers
    const bool need_draft = !greedy && L > 0;
    if (!target_logits || (L > 0 && !draft_tokens) || !accept_len || !accept_draft || !out_token)
        return SDV_ERR_INVALID;
    if (need_draft && (!draft_logits || !accept_u)) return SDV_ERR_INVALID;
    if (!greedy && !sample_u) return SDV_ERR_INVALID;
    if (!aligned(target_logits, 16) || (need_draft && !aligned(draft_logits, 16))) return SDV_ERR_INVALID;
    const void* ptrs[] = {target_logits,  need_draft ? draft_logits : nullptr,
                          L > 0 ? draft_tokens : nullptr, lengths,
                          need_draft ? accept_u : nullptr, greedy ? nullptr : sample_u,
                          accept_len, accept_draft, out_token, accept_prob, residual_mass, residual_out};
    for (const void* q : ptrs)
        if (q && !device_accessible(q)) return SDV_ERR_INVALID;
    if (residual_out && !aligned(residual_out, 4)) return SDV_ERR_INVALID;
    if (leaf_target && (!aligned(leaf_target, 16) || !device_accessible(leaf_target))) return SDV_ERR_INVALID;
    if (!workspace || !aligned(workspace, kAlign) || workspace_bytes < workspace_size(B, K, L))
        return SDV_ERR_WORKSPACE;
    if (!device_accessible(workspace)) return SDV_ERR_WORKSPACE;

    Problem pb;
    std::memset(&pb, 0, sizeof pb);
    pb.B = B;
    pb.K = K;
    pb.L = L;
    pb.V = V;
    pb.stride = row_stride;
    pb.dtype = dtype;
    pb.mode = greedy ? SDV_MODE_GREEDY : mode;
    pb.c = c;
    pb.target = target_logits;
    pb.leaf_target = leaf_target;
    pb.draft = draft_logits;
    pb.tokens = draft_tokens;
    pb.lengths = lengths;
    pb.accept_u = accept_u;
    pb.sample_u = sample_u;
    pb.accept_len = accept_len;
    pb.accept_draft = accept_draft;
    pb.out_token = out_token;
    pb.accept_prob = accept_prob;
    pb.residual_mass = residual_mass;
    pb.device_status = device_status;
    pb.residual_out = residual_out;
    pb.wait_ns = g_wait_ns ? g_wait_ns : kDefaultWaitNs;
    pb.ws = carve(workspace, B, K, L);

    if (device_status && cudaMemsetAsync(device_status, 0, sizeof(int), st) != cudaSuccess) return SDV_ERR_CUDA;
    if (cudaMemsetAsync(pb.ws.ncount, 0, sizeof(int) * (2 * L + 3), st) != cudaSuccess) return SDV_ERR_CUDA;
    if (launch_prep(pb, st) != cudaSuccess) return SDV_ERR_CUDA;
    // test hook: take the roots (depth 0) out of the node kernel's work list,
    // so that nothing writes their children's weights nor finishes their
    // requests, and every wait on them runs out
    if (skip_roots && (cudaMemsetAsync(pb.ws.ncount, 0, sizeof(int), st) != cudaSuccess ||
                       cudaMemsetAsync(pb.ws.ncount + (L + 1), 0, sizeof(int), st) != cudaSuccess))
        return SDV_ERR_CUDA;
    if (!prof_record(g_prof_start, st)) return SDV_ERR_CUDA;
    if (greedy) {
        if (launch_argmax(pb, st) != cudaSuccess) return SDV_ERR_CUDA;
    } else {
        // every node of every depth in one persistent launch; a node's
        // weight comes from its parent through a flag
        const cudaError_t e = launch_stream(pb, st);
        if (e == cudaErrorInvalidValue || e == cudaErrorNoKernelImageForDevice) {
            cudaGetLastError();
            return SDV_ERR_UNSUPPORTED;  // e.g. not enough shared memory on this device
        }
        if (e != cudaSuccess) return SDV_ERR_CUDA;
    }
    if (!prof_record(g_prof_stop, st)) return SDV_ERR_CUDA;
    // per request: the decision, then the correction (or bonus) token drawn
    // at its end node only.  After the node kernel it is launched as that
    // kernel's programmatic dependent, each CTA waiting for its request's
    // nodes; a profiling event between the two would serialize them, so
    // with the hook on it is an ordinary launch.
    const bool overlap = !greedy && !g_prof_stop;
    if (launch_finish(pb, greedy, st, overlap) != cudaSuccess) return SDV_ERR_CUDA;
    return SDV_OK;
}

// The LM-head part of the workspace (after carve's), and pb.ws itself.
LmRows carve_lm(void* workspace, Problem& pb, int d, const void* hidden)
{
    const int B = pb.B, K = pb.K, L = pb.L;
    pb.ws = carve(workspace, B, K, L);
    const size_t n = slot_count(B, K, L);
    char* p = static_cast<char*>(workspace) + workspace_size(B, K, L);
    LmRows r;
    std::memset(&r, 0, sizeof r);
    r.d = d;
    r.hidden = hidden;
    r.compact = reinterpret_cast<int*>(p);
    p += align_up(n * 4);
    r.count = reinterpret_cast<int*>(p);
    p += align_up(4);
    r.keys = reinterpret_cast<unsigned long long*>(p);
    p += align_up(n * 8);
    r.rows = p;
    p += align_up(n * (size_t)d * 2);
    r.row_of = reinterpret_cast<int*>(p);
    p += align_up(n * 4);
    pb.leaf_pending = reinterpret_cast<int*>(p);
    p += align_up((size_t)B * 4);
    r.leaf_req = reinterpret_cast<int*>(p);
    p += align_up((size_t)B * 4);
    r.leaf_count = reinterpret_cast<int*>(p);
    p += align_up(4);
    r.leaf_keys = reinterpret_cast<unsigned long long*>(p);
    p += align_up((size_t)B * 8);
    r.leaf_rows = p;
    return r;
}

int verify_greedy_lm_head(int B, int K, int L, int V, int d, const void* hidden, const void* lm_head,
                          const int* draft_tokens, const int* lengths, int* accept_len, int* accept_draft,
                          int* out_token, float* accept_prob, int* device_status, void* workspace,
                          size_t workspace_bytes, void* cuda_stream)
{
    if (!sizes_ok(B, K, L, V) || !lm_d_ok(d)) return SDV_ERR_INVALID;
    cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
    if (device_status && !device_accessible(device_status)) return SDV_ERR_INVALID;
    if (B == 0) {
        if (device_status && cudaMemsetAsync(device_status, 0, sizeof(int), st) != cudaSuccess) return SDV_ERR_CUDA;
        return SDV_OK;
    }
    if (!hidden || !lm_head || (L > 0 && !draft_tokens) || !accept_len || !accept_draft || !out_token)
        return SDV_ERR_INVALID;
    if (!aligned(hidden, 16) || !aligned(lm_head, 16)) return SDV_ERR_INVALID;
    const void* ptrs[] = {hidden, lm_head, L > 0 ? draft_tokens : nullptr, lengths, accept_len, accept_draft,
                          out_token, accept_prob};
    for (const void* q : ptrs)
        if (q && !device_accessible(q)) return SDV_ERR_INVALID;
    if (!workspace || !aligned(workspace, kAlign) || workspace_bytes < lm_workspace_size(B, K, L, d))
        return SDV_ERR_WORKSPACE;
    if (!device_accessible(workspace)) return SDV_ERR_WORKSPACE;

    Problem pb;
    std::memset(&pb, 0, sizeof pb);
    pb.B = B;
    pb.K = K;
    pb.L = L;
    pb.V = V;
    pb.stride = V;
    pb.dtype = SDV_BF16;
    pb.mode = SDV_MODE_GREEDY;
    pb.tokens = draft_tokens;
    pb.lengths = lengths;
    pb.accept_len = accept_len;
    pb.accept_draft = accept_draft;
    pb.out_token = out_token;
    pb.accept_prob = accept_prob;
    pb.device_status = device_status;
    pb.wait_ns = g_wait_ns ? g_wait_ns : kDefaultWaitNs;
    const size_t n = slot_count(B, K, L);
    LmRows r = carve_lm(workspace, pb, d, hidden);
    r.leaves = 0;
    LmArgs a;
    std::memset(&a, 0, sizeof a);
    a.rows_dev = r.count;
    a.V = V;
    a.d = d;
    a.keys = r.keys;
    a.device_status = device_status;

    if (device_status && cudaMemsetAsync(device_status, 0, sizeof(int), st) != cudaSuccess) return SDV_ERR_CUDA;
    if (cudaMemsetAsync(pb.ws.ncount, 0, sizeof(int) * (2 * L + 3), st) != cudaSuccess) return SDV_ERR_CUDA;
    if (cudaMemsetAsync(r.count, 0, sizeof(int), st) != cudaSuccess) return SDV_ERR_CUDA;
    if (cudaMemsetAsync(r.leaf_count, 0, sizeof(int), st) != cudaSuccess) return SDV_ERR_CUDA;
    if (launch_prep(pb, st) != cudaSuccess) return SDV_ERR_CUDA;
    if (launch_lm_rows(pb, r, st) != cudaSuccess) return SDV_ERR_CUDA;
    if (!prof_record(g_prof_start, st)) return SDV_ERR_CUDA;
    const cudaError_t e = launch_lm_head(r.rows, (long long)n, lm_head, a, LM_EPI_ARGMAX, st);
    if (e == cudaErrorInvalidValue) {
        cudaGetLastError();
        return SDV_ERR_UNSUPPORTED;  // no tensor-map encoder, or not enough shared memory
    }
    if (e != cudaSuccess) return SDV_ERR_CUDA;
    if (!prof_record(g_prof_stop, st)) return SDV_ERR_CUDA;
    if (launch_lm_argmax(pb, r, st) != cudaSuccess) return SDV_ERR_CUDA;
    // the decision; where it ends at a leaf, that leaf's row is computed now
    if (launch_finish(pb, true, st) != cudaSuccess) return SDV_ERR_CUDA;
    if (launch_lm_leaf_rows(pb, r, st) != cudaSuccess) return SDV_ERR_CUDA;
    LmArgs la = a;
    la.rows_dev = r.leaf_count;
    la.keys = r.leaf_keys;
    if (launch_lm_head(r.leaf_rows, (long long)B, lm_head, la, LM_EPI_ARGMAX, st) != cudaSuccess) return SDV_ERR_CUDA;
    if (launch_lm_leaf_token(pb, r, st) != cudaSuccess) return SDV_ERR_CUDA;
    return SDV_OK;
}

}  // namespace

// The rows verification reads, as one contiguous range per (request, draft)
// and tensor: draft k owns its trie nodes from depth f_k on (f_0 = 0; for
// k > 0, one past the longest prefix it shares with a lower draft, since a
// node belongs to the lowest draft through it), so it brings target rows
// [f_k, L_b] and draft rows [f_k, L_b - 1].  Requests with a length outside
// 0..L get none (they are reported invalid).  Each range goes to fn(target?,
// offset in rows, rows).
template <class Fn>
void for_read_rows(int B, int K, int L, const int* tokens, const int* lengths, Fn fn)
{
    for (int b = 0; b < B; ++b) {
        const int Lb = lengths ? lengths[b] : L;
        if (Lb < 0 || Lb > L) continue;
        for (int k = 0; k < K; ++k) {
            int f = 0;
            const int* tk = tokens + ((size_t)b * K + k) * L;
            for (int k2 = 0; k2 < k && f <= Lb; ++k2) {
                const int* t2 = tokens + ((size_t)b * K + k2) * L;
                int m = 0;
                while (m < Lb && tk[m] == t2[m]) ++m;
                if (m + 1 > f) f = m + 1;
            }
            if (f <= Lb) fn(true, ((size_t)b * K + k) * (L + 1) + f, (size_t)(Lb - f + 1));
            if (f < Lb) fn(false, ((size_t)b * K + k) * L + f, (size_t)(Lb - f));
        }
    }
}

}  // namespace sdv

extern "C" {

#define SDV_FORWARD(mode)                                                                                    \
    sdv::verify(mode, B, K, L, V, row_stride, dtype, temperature, target_logits, draft_logits, draft_tokens, \
                lengths, accept_u, sample_u, accept_len, accept_draft, out_token, accept_prob, residual_mass, \
                device_status, workspace, workspace_bytes, cuda_stream)

int sdv_verify_token(SDV_VERIFY_ARGS) { return SDV_FORWARD(SDV_MODE_TOKEN); }
int sdv_verify_greedy(SDV_VERIFY_ARGS) { return SDV_FORWARD(SDV_MODE_GREEDY); }
int sdv_verify_block(SDV_VERIFY_ARGS) { return SDV_FORWARD(SDV_MODE_BLOCK); }
int sdv_verify_multidraft(SDV_VERIFY_ARGS) { return SDV_FORWARD(SDV_MODE_MULTIDRAFT); }
int sdv_verify_kseq(SDV_VERIFY_ARGS) { return SDV_FORWARD(SDV_MODE_KSEQ); }

int sdv_verify_leaves_apart(int mode, SDV_VERIFY_ARGS, const void* leaf_target_logits)
{
    if (mode < SDV_MODE_TOKEN || mode > SDV_MODE_KSEQ) return SDV_ERR_INVALID;
    return sdv::verify(mode, B, K, L, V, row_stride, dtype, temperature, target_logits, draft_logits, draft_tokens,
                       lengths, accept_u, sample_u, accept_len, accept_draft, out_token, accept_prob, residual_mass,
                       device_status, workspace, workspace_bytes, cuda_stream, leaf_target_logits);
}

int sdv_verify_residual(int mode, SDV_VERIFY_ARGS, float* residual_out)
{
    if (mode < SDV_MODE_TOKEN || mode > SDV_MODE_KSEQ) return SDV_ERR_INVALID;
    if (!residual_out && B > 0) return SDV_ERR_INVALID;
    return sdv::verify(mode, B, K, L, V, row_stride, dtype, temperature, target_logits, draft_logits, draft_tokens,
                       lengths, accept_u, sample_u, accept_len, accept_draft, out_token, accept_prob, residual_mass,
                       device_status, workspace, workspace_bytes, cuda_stream, nullptr, residual_out);
}

int sdv_testing_set_wait_limit(unsigned long long wait_ns)
{
    sdv::g_wait_ns = wait_ns;
    return SDV_OK;
}

int sdv_testing_set_lm_head_single_cta(int on)
{
    sdv::g_lm_single_cta = on ? 1 : 0;
    return SDV_OK;
}

int sdv_testing_verify_without_roots(int mode, SDV_VERIFY_ARGS)
{
    if (mode != SDV_MODE_BLOCK && mode != SDV_MODE_MULTIDRAFT) return SDV_ERR_INVALID;
    return sdv::verify(mode, B, K, L, V, row_stride, dtype, temperature, target_logits, draft_logits, draft_tokens,
                       lengths, accept_u, sample_u, accept_len, accept_draft, out_token, accept_prob, residual_mass,
                       device_status, workspace, workspace_bytes, cuda_stream, nullptr, nullptr, true);
}

size_t sdv_workspace_bytes(int mode, int B, int K, int L, int V)
{
    if (mode < SDV_MODE_TOKEN || mode > SDV_MODE_KSEQ || !sdv::sizes_ok(B, K, L, V)) return 0;
    if (mode == SDV_MODE_BLOCK && K != 1) return 0;
    return sdv::workspace_size(B, K, L);
}

int sdv_verify_greedy_lm_head(int B, int K, int L, int V, int d, const void* hidden, const void* lm_head,
                              const int* draft_tokens, const int* lengths, int* accept_len, int* accept_draft,
                              int* out_token, float* accept_prob, int* device_status, void* workspace,
                              size_t workspace_bytes, void* cuda_stream)
{
    return sdv::verify_greedy_lm_head(B, K, L, V, d, hidden, lm_head, draft_tokens, lengths, accept_len,
                                      accept_draft, out_token, accept_prob, device_status, workspace,
                                      workspace_bytes, cuda_stream);
}

int sdv_lm_head_trie_logits(int B, int K, int L, int V, int d, const void* hidden, const void* lm_head,
                            const int* draft_tokens, const int* lengths, void* target_logits, long long row_stride,
                            int* device_status, void* workspace, size_t workspace_bytes, void* cuda_stream)
{
    using namespace sdv;
    if (!sizes_ok(B, K, L, V) || !lm_d_ok(d) || row_stride < V || row_stride % 8) return SDV_ERR_INVALID;
    cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
    if (device_status && !device_accessible(device_status)) return SDV_ERR_INVALID;
    if (device_status && cudaMemsetAsync(device_status, 0, sizeof(int), st) != cudaSuccess) return SDV_ERR_CUDA;
    if (B == 0) return SDV_OK;
    if (!hidden || !lm_head || !target_logits || (L > 0 && !draft_tokens)) return SDV_ERR_INVALID;
    if (!aligned(hidden, 16) || !aligned(lm_head, 16) || !aligned(target_logits, 16)) return SDV_ERR_INVALID;
    const void* ptrs[] = {hidden, lm_head, target_logits, L > 0 ? draft_tokens : nullptr, lengths};
    for (const void* q : ptrs)
        if (q && !device_accessible(q)) return SDV_ERR_INVALID;
    if (!workspace || !aligned(workspace, kAlign) || workspace_bytes < lm_workspace_size(B, K, L, d))
        return SDV_ERR_WORKSPACE;
    if (!device_accessible(workspace)) return SDV_ERR_WORKSPACE;

    Problem pb;
    std::memset(&pb, 0, sizeof pb);
    pb.B = B;
    pb.K = K;
    pb.L = L;
    pb.V = V;
    pb.stride = row_stride;
    pb.dtype = SDV_BF16;
    pb.mode = SDV_MODE_MULTIDRAFT;
    pb.tokens = draft_tokens;
    pb.lengths = lengths;
    pb.device_status = device_status;
    pb.wait_ns = g_wait_ns ? g_wait_ns : kDefaultWaitNs;
    LmRows r = carve_lm(workspace, pb, d, hidden);
    r.leaves = 1;  // every trie node's row, leaves included
    LmArgs a;
    std::memset(&a, 0, sizeof a);
    a.rows_dev = r.count;
    a.V = V;
    a.d = d;
    a.out_bf16 = target_logits;
    a.dest_row = r.row_of;
    a.out_stride = row_stride;
    a.device_status = device_status;
    if (cudaMemsetAsync(pb.ws.ncount, 0, sizeof(int) * (2 * L + 3), st) != cudaSuccess) return SDV_ERR_CUDA;
    if (cudaMemsetAsync(r.count, 0, sizeof(int), st) != cudaSuccess) return SDV_ERR_CUDA;
    if (launch_prep(pb, st) != cudaSuccess) return SDV_ERR_CUDA;
    if (launch_lm_rows(pb, r, st) != cudaSuccess) return SDV_ERR_CUDA;
    if (!prof_record(g_prof_start, st)) return SDV_ERR_CUDA;
    const cudaError_t e = launch_lm_head(r.rows, (long long)slot_count(B, K, L), lm_head, a, LM_EPI_ROWS_BF16, st);
    if (e == cudaErrorInvalidValue) {
        cudaGetLastError();
        return SDV_ERR_UNSUPPORTED;
    }
    if (e != cudaSuccess) return SDV_ERR_CUDA;
    return prof_record(g_prof_stop, st) ? SDV_OK : SDV_ERR_CUDA;
}

size_t sdv_lm_head_workspace_bytes(int B, int K, int L, int V, int d)
{
    if (!sdv::sizes_ok(B, K, L, V) || !sdv::lm_d_ok(d)) return 0;
    return sdv::lm_workspace_size(B, K, L, d);
}

int sdv_lm_head_logits(int M, int V, int d, const void* hidden, const void* lm_head, float* logits,
                       long long logits_stride, int* device_status, void* cuda_stream)
{
    if (M < 0 || V < 1 || V > SDV_MAX_V || !sdv::lm_d_ok(d) || logits_stride < V || logits_stride % 4)
        return SDV_ERR_INVALID;
    cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
    if (device_status && !sdv::device_accessible(device_status)) return SDV_ERR_INVALID;
    if (device_status && cudaMemsetAsync(device_status, 0, sizeof(int), st) != cudaSuccess) return SDV_ERR_CUDA;
    if (M == 0) return SDV_OK;
    if (!hidden || !lm_head || !logits) return SDV_ERR_INVALID;
    if (!sdv::aligned(hidden, 16) || !sdv::aligned(lm_head, 16) || !sdv::aligned(logits, 16)) return SDV_ERR_INVALID;
    const void* ptrs[] = {hidden, lm_head, logits};
    for (const void* q : ptrs)
        if (!sdv::device_accessible(q)) return SDV_ERR_INVALID;
    sdv::LmArgs a;
    std::memset(&a, 0, sizeof a);
    a.rows = M;
    a.V = V;
    a.d = d;
    a.logits = logits;
    a.out_stride = logits_stride;
    a.device_status = device_status;
    if (!sdv::prof_record(sdv::g_prof_start, st)) return SDV_ERR_CUDA;
    const cudaError_t e = sdv::launch_lm_head(hidden, M, lm_head, a, sdv::LM_EPI_LOGITS, st);
    if (e == cudaErrorInvalidValue) {
        cudaGetLastError();
        return SDV_ERR_UNSUPPORTED;
    }
    if (e != cudaSuccess) return SDV_ERR_CUDA;
    return sdv::prof_record(sdv::g_prof_stop, st) ? SDV_OK : SDV_ERR_CUDA;
}

const char* sdv_status_string(int status)
{
    switch (status) {
    case SDV_OK: return "ok";
    case SDV_ERR_INVALID: return "invalid argument";
    case SDV_ERR_UNSUPPORTED: return "unsupported on this build or device";
    case SDV_ERR_CUDA: return "CUDA runtime or launch error";
    case SDV_ERR_TIMEOUT: return "device wait timed out";
    case SDV_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    default: return "unknown status";
    }
}

int sdv_set_profile_events(void* start, void* stop)
{
    if ((start == nullptr) != (stop == nullptr)) return SDV_ERR_INVALID;
    sdv::g_prof_start = static_cast<cudaEvent_t>(start);
    sdv::g_prof_stop = static_cast<cudaEvent_t>(stop);
    return SDV_OK;
}

int sdv_sample_rows(int n_rows, int V, long long row_stride, int dtype, float temperature, const void* logits,
                    int n_samples, const float* u, int* tokens, int* device_status, void* cuda_stream)
{
    if (n_rows < 0 || V < 1 || V > SDV_MAX_V || (dtype != SDV_F32 && dtype != SDV_BF16)) return SDV_ERR_INVALID;
    if (row_stride < V || row_stride % 8 != 0) return SDV_ERR_INVALID;
    if (n_samples < 1 || n_samples > SDV_MAX_SAMPLES) return SDV_ERR_INVALID;
    if (!(temperature >= 0.f) || std::isinf(temperature)) return SDV_ERR_INVALID;
    const bool greedy = temperature == 0.f;
    const float c = greedy ? 0.f : (float)(1.4426950408889634 / (double)temperature);
    if (!greedy && !std::isfinite(c)) return SDV_ERR_INVALID;
    cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
    if (device_status && !sdv::device_accessible(device_status)) return SDV_ERR_INVALID;
    if (device_status && cudaMemsetAsync(device_status, 0, sizeof(int), st) != cudaSuccess) return SDV_ERR_CUDA;
    if (n_rows == 0) return SDV_OK;
    if (!logits || !tokens || (!greedy && !u)) return SDV_ERR_INVALID;
    if (!sdv::aligned(logits, 16)) return SDV_ERR_INVALID;
    const void* ptrs[] = {logits, greedy ? nullptr : u, tokens};
    for (const void* q : ptrs)
        if (q && !sdv::device_accessible(q)) return SDV_ERR_INVALID;
    sdv::SampleArgs a;
    a.n_rows = n_rows;
    a.V = V;
    a.n_samples = n_samples;
    a.dtype = dtype;
    a.stride = row_stride;
    a.c = c;
    a.logits = logits;
    a.u = u;
    a.tokens = tokens;
    a.device_status = device_status;
    return sdv::launch_sample_rows(a, st) == cudaSuccess ? SDV_OK : SDV_ERR_CUDA;
}

int sdv_launch_shape(int V, int dtype, int* ctas_per_sm, int* threads, int* smem_bytes)
{
    if (V < 1 || V > SDV_MAX_V || (dtype != SDV_F32 && dtype != SDV_BF16)) return SDV_ERR_INVALID;
    if (ctas_per_sm) *ctas_per_sm = sdv::stream_ctas_per_sm();
    if (threads) *threads = sdv::stream_threads();
    if (smem_bytes) *smem_bytes = (int)sdv::stream_smem_bytes();
    return SDV_OK;
}

static int gather_rows(int B, int K, int L, int V, long long row_stride, int dtype, const void* host_target,
                       const void* host_draft, const int* tokens, const int* lengths, void* target, void* draft,
                       void* cuda_stream, int leaves)
{
    if (!sdv::sizes_ok(B, K, L, V) || row_stride < V || row_stride % 8 || (dtype != SDV_F32 && dtype != SDV_BF16) ||
        K > 256)
        return SDV_ERR_INVALID;
    if (B == 0) return SDV_OK;
    // every pointer must be one the device can address: device memory, or
    // host memory mapped into the device's address space
    if (!sdv::device_accessible(host_target) || !sdv::device_accessible(target) || !sdv::aligned(host_target, 16) ||
        !sdv::aligned(target, 16))
        return SDV_ERR_INVALID;
    if (L > 0 && (!tokens || !host_draft || !draft || !sdv::device_accessible(tokens) ||
                  !sdv::device_accessible(host_draft) || !sdv::device_accessible(draft) ||
                  !sdv::aligned(host_draft, 16) || !sdv::aligned(draft, 16)))
        return SDV_ERR_INVALID;
    if (lengths && !sdv::device_accessible(lengths)) return SDV_ERR_INVALID;
    sdv::GatherArgs a;
    a.B = B;
    a.K = K;
    a.L = L;
    a.leaves = leaves;
    a.row_bytes = row_stride * (dtype == SDV_BF16 ? 2 : 4);
    a.host_target = host_target;
    a.host_draft = host_draft;
    a.tokens = tokens;
    a.lengths = lengths;
    a.target = target;
    a.draft = draft;
    return sdv::launch_gather_rows(a, static_cast<cudaStream_t>(cuda_stream)) == cudaSuccess ? SDV_OK : SDV_ERR_CUDA;
}

int sdv_gather_read_rows(int B, int K, int L, int V, long long row_stride, int dtype, const void* host_target,
                         const void* host_draft, const int* tokens, const int* lengths, void* target, void* draft,
                         void* cuda_stream)
{
    return gather_rows(B, K, L, V, row_stride, dtype, host_target, host_draft, tokens, lengths, target, draft,
                       cuda_stream, 1);
}

int sdv_gather_inner_rows(int B, int K, int L, int V, long long row_stride, int dtype, const void* host_target,
                          const void* host_draft, const int* tokens, const int* lengths, void* target, void* draft,
                          void* cuda_stream)
{
    return gather_rows(B, K, L, V, row_stride, dtype, host_target, host_draft, tokens, lengths, target, draft,
                       cuda_stream, 0);
}

int sdv_read_rows_bytes(int B, int K, int L, int V, long long row_stride, int dtype, const int* tokens,
                        const int* lengths, long long* bytes)
{
    if (!sdv::sizes_ok(B, K, L, V) || row_stride < V || row_stride % 8 || (dtype != SDV_F32 && dtype != SDV_BF16) ||
        !bytes || (B > 0 && L > 0 && !tokens))
        return SDV_ERR_INVALID;
    const size_t row = (size_t)row_stride * (dtype == SDV_BF16 ? 2 : 4);
    size_t n = 0;
    sdv::for_read_rows(B, K, L, tokens, lengths, [&](bool, size_t, size_t rows) { n += rows * row; });
    *bytes = (long long)n;
    return SDV_OK;
}

int sdv_copy_read_rows(int B, int K, int L, int V, long long row_stride, int dtype, const void* host_target,
                       const void* host_draft, const int* tokens, const int* lengths, void* target, void* draft,
                       void* cuda_stream, long long* bytes)
{
    if (!sdv::sizes_ok(B, K, L, V) || row_stride < V || row_stride % 8 || (dtype != SDV_F32 && dtype != SDV_BF16) ||
        (B > 0 && (!host_target || !target || (L > 0 && (!tokens || !host_draft || !draft)))))
        return SDV_ERR_INVALID;
    const size_t row = (size_t)row_stride * (dtype == SDV_BF16 ? 2 : 4);
    const cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
    size_t n = 0;
    cudaError_t e = cudaSuccess;
    sdv::for_read_rows(B, K, L, tokens, lengths, [&](bool is_target, size_t first, size_t rows) {
        if (e != cudaSuccess) return;
        const size_t off = first * row, len = rows * row;
        if (is_target)
            e = cudaMemcpyAsync(static_cast<char*>(target) + off, static_cast<const char*>(host_target) + off, len,
                                cudaMemcpyHostToDevice, st);
        else
            e = cudaMemcpyAsync(static_cast<char*>(draft) + off, static_cast<const char*>(host_draft) + off, len,
                                cudaMemcpyHostToDevice, st);
        n += len;
    });
    if (bytes) *bytes = (long long)n;
    return e == cudaSuccess ? SDV_OK : SDV_ERR_CUDA;
}

}  // extern "C"
