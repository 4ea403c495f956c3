// sdv_kernels.cu -- the small kernels around the node kernel (which is in
// sdv_stream.cu).
//
// prep_kernel     one warp per request: length and token checks, the
//                 draft-trie owners, the depth-major list of trie nodes the
//                 node kernel works through.
// argmax_kernel   greedy: one CTA per node, streaming argmax of the target.
// decide_kernel   one warp per request: the token-level walk, the
//                 depth-first block search or greedy matching over the
//                 node records; writes the outputs.
//
// The rules (SpecTr-GBV: Multi-Draft Block Verification Accelerating
// Speculative Decoding, sections 1 and 2) are stated in include/sdv.h.
#include "sdv_internal.h"
#include "sdv_device.cuh"

namespace sdv {
namespace {

// ------------------------------------------------------------------------
// prep: one warp per request

__global__ void prep_kernel(Problem pb)
{
    const int lane = threadIdx.x & 31;
    const int b = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (b >= pb.B) return;
    const int K = pb.K, L = pb.L, V = pb.V;
    const int Lb = pb.lengths ? pb.lengths[b] : L;
    int st = 0;
    if (Lb < 0 || Lb > L) {
        st = SDV_REQ_BAD_LENGTH;
    } else {
        int bad = 0;
        for (int i = lane; i < K * Lb; i += 32) {
            const int t = pb.tokens[((size_t)b * K + i / Lb) * L + i % Lb];
            bad |= (t < 0 || t >= V);
        }
        if (__any_sync(0xffffffffu, bad)) st = SDV_REQ_BAD_TOKEN;
    }
    if (lane == 0) {
        pb.ws.req[b] = st;
        if (st && pb.device_status) atomicOr(pb.device_status, st);
    }
    if (st) return;
    // owner[j][k] = lowest k2 whose first j tokens equal draft k's: drafts
    // share a prefix of length j iff they share the one of length j-1 and
    // token j-1.  Lane k holds draft k.
    unsigned char* own = pb.ws.owner + (size_t)b * (L + 1) * K;
    int o = 0;
    if (lane < K) own[lane] = 0;
    for (int j = 1; j <= Lb; ++j) {
        const int tk = lane < K ? pb.tokens[((size_t)b * K + lane) * L + j - 1] : -1;
        int no = lane;
        for (int k2 = K - 1; k2 >= 0; --k2) {
            const int o2 = __shfl_sync(0xffffffffu, o, k2);
            const int t2 = __shfl_sync(0xffffffffu, tk, k2);
            if (k2 <= lane && o2 == o && t2 == tk) no = k2;
        }
        o = no;
        if (lane < K) own[j * K + lane] = (unsigned char)o;
    }
    if (lane == 0) pb.ws.pbar[(size_t)b * (L + 1) * K] = 0.f;  // root weight 1
    // list the request's nodes by depth (for the streaming kernel) and clear
    // the flags through which parents publish their children's weights
    const size_t BK = (size_t)pb.B * K;
    for (int j = 0; j <= Lb; ++j) {
        const bool node = lane < K && own[j * K + lane] == lane;
        const unsigned m = __ballot_sync(0xffffffffu, node);
        int base = 0;
        if (lane == 0) base = atomicAdd(&pb.ws.ncount[j], __popc(m));
        base = __shfl_sync(0xffffffffu, base, 0);
        const size_t slot = ((size_t)b * (L + 1) + j) * K + lane;
        if (node) pb.ws.nodes[j * BK + base + __popc(m & ((1u << lane) - 1))] = (int)slot;
        if (lane < K) pb.ws.ready[slot] = 0;
    }
}

// ------------------------------------------------------------------------
// greedy argmax: one CTA per node, streaming

template <int DT>
__global__ void __launch_bounds__(256) argmax_kernel(Problem pb)
{
    using E = Elem<DT>;
    constexpr int EPU = E::kPerUnit;
    const int K = pb.K, L = pb.L, V = pb.V;
    const int slot = blockIdx.x;  // (b * (L+1) + j) * K + k
    const int k = slot % K;
    const int j = (slot / K) % (L + 1);
    const int b = slot / (K * (L + 1));
    if (pb.ws.req[b] & (SDV_REQ_BAD_LENGTH | SDV_REQ_BAD_TOKEN)) return;
    const int Lb = pb.lengths ? pb.lengths[b] : L;
    if (j > Lb || pb.ws.owner[slot] != k) return;
    const size_t row = ((size_t)b * K + k) * (L + 1) + j;
    const uint4* g = reinterpret_cast<const uint4*>(static_cast<const char*>(pb.target) +
                                                    row * (size_t)pb.stride * E::kBytes);
    const int n_units = (V + EPU - 1) / EPU;
    float best = -INFINITY;
    int bidx = 0x7fffffff;
    bool bad = false;
    for (int uu = threadIdx.x; uu < n_units; uu += blockDim.x) {
        float v[EPU];
        unpack_masked<DT>(__ldg(g + uu), uu * EPU, V, v);
#pragma unroll
        for (int e = 0; e < EPU; ++e) {
            bad |= (v[e] != v[e]) || (v[e] == INFINITY);
            if (v[e] > best) {
                best = v[e];
                bidx = uu * EPU + e;
            }
        }
    }
    // larger value wins, then the lower index
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float ob = __shfl_xor_sync(0xffffffffu, best, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bidx, o);
        if (ob > best || (ob == best && oi < bidx)) {
            best = ob;
            bidx = oi;
        }
    }
    bad = __any_sync(0xffffffffu, bad);
    __shared__ float sb[8];
    __shared__ int si[8];
    __shared__ int sbad[8];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) {
        sb[warp] = best;
        si[warp] = bidx;
        sbad[warp] = bad;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int w = 1; w < (int)(blockDim.x >> 5); ++w) {
            if (sb[w] > best || (sb[w] == best && si[w] < bidx)) {
                best = sb[w];
                bidx = si[w];
            }
            bad |= sbad[w] != 0;
        }
        if (bad || best == -INFINITY) {
            atomicOr(&pb.ws.req[b], SDV_REQ_NONFINITE);
            if (pb.device_status) atomicOr(pb.device_status, SDV_REQ_NONFINITE);
            bidx = -1;
        }
        pb.ws.am[slot] = bidx;
    }
}

// ------------------------------------------------------------------------
// decision: one warp per request; the request's node records are copied to
// shared memory first, then lane 0 walks them

constexpr int kDecideWarps = 4;
constexpr int kSlotsMax = (SDV_MAX_L + 1) * SDV_MAX_K;

__global__ void __launch_bounds__(32 * kDecideWarps) decide_kernel(Problem pb, int greedy)
{
    __shared__ unsigned char s_own[kDecideWarps][kSlotsMax];
    __shared__ float s_val[kDecideWarps][kSlotsMax];  // a (token), h (block) or argmax bits (greedy)
    __shared__ float s_u[kDecideWarps][SDV_MAX_K * SDV_MAX_L];
    __shared__ int s_tok[kDecideWarps][SDV_MAX_K * SDV_MAX_L];
    __shared__ signed char s_sib[kDecideWarps][kSlotsMax];  // next sibling's draft, or -1
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int b = blockIdx.x * kDecideWarps + w;
    if (b >= pb.B) return;
    const int K = pb.K, L = pb.L;
    const int st = pb.ws.req[b];
    float* ap = pb.accept_prob ? pb.accept_prob + (size_t)b * K * L : nullptr;
    if (st) {
        if (ap)
            for (int i = lane; i < K * L; i += 32) ap[i] = 0.f;
        if (lane == 0) {
            pb.accept_len[b] = 0;
            pb.accept_draft[b] = 0;
            pb.out_token[b] = -1;
            pb.ws.endn[b] = -1;  // no correction draw
            if (pb.residual_mass) pb.residual_mass[b] = 0.f;
            if (pb.device_status) atomicOr(pb.device_status, st);
        }
        return;
    }
    const int Lb = pb.lengths ? pb.lengths[b] : L;
    const size_t s0 = (size_t)b * (L + 1) * K;
    const bool token = pb.mode == SDV_MODE_TOKEN;
    unsigned char* own = s_own[w];
    float* val = s_val[w];
    float* uu = s_u[w];
    int* tk = s_tok[w];
    for (int i = lane; i < (Lb + 1) * K; i += 32) {
        own[i] = pb.ws.owner[s0 + i];
        float v;
        if (greedy)
            v = __int_as_float(pb.ws.am[s0 + i]);
        else if (token)
            v = pb.ws.a[s0 + i];
        else  // a leaf's block acceptance is its weight p (the node kernel only checks leaves)
            v = i >= Lb * K ? (Lb == 0 ? 1.f : 1.f - pb.ws.pbar[s0 + i]) : pb.ws.h[s0 + i];
        val[i] = v;
    }
    for (int i = lane; i < K * L; i += 32) {
        tk[i] = pb.tokens[(size_t)b * K * L + i];
        uu[i] = greedy ? 0.f : pb.accept_u[(size_t)b * K * L + i];
    }
    __syncwarp();
    // accept_prob[k][d]: the threshold draft k's position d is tested against
    if (ap) {
        for (int i = lane; i < K * L; i += 32) {
            const int kk = i / L, d = i % L;
            float v = 0.f;
            if (d < Lb) {
                if (greedy)
                    v = tk[i] == __float_as_int(val[d * K + own[d * K + kk]]) ? 1.f : 0.f;
                else if (token)
                    v = val[d * K + kk];
                else
                    v = val[(d + 1) * K + own[(d + 1) * K + kk]];
            }
            ap[i] = v;
        }
    }
    int ej = 0, eo = 0;
    if (greedy) {
        if (lane != 0) return;
        int best = -1, bestk = 0;
        for (int kk = 0; kk < K; ++kk) {
            int m = 0;
            while (m < Lb && tk[kk * L + m] == __float_as_int(val[m * K + own[m * K + kk]])) ++m;
            if (m > best) {
                best = m;
                bestk = kk;
            }
        }
        ej = best;
        eo = own[best * K + bestk];
        pb.accept_len[b] = best;
        pb.accept_draft[b] = bestk;
        pb.out_token[b] = __float_as_int(val[ej * K + eo]);
        if (pb.residual_mass) pb.residual_mass[b] = 1.f;
        return;
    }
    if (token) {
        if (lane != 0) return;
        int j = 0, o = 0;
        while (j < Lb) {
            int acc = -1;
            for (int kk = 0; kk < K && acc < 0; ++kk)
                if (own[j * K + kk] == o && uu[kk * L + j] <= val[j * K + kk]) acc = kk;
            if (acc < 0) break;
            o = own[(j + 1) * K + acc];
            ++j;
        }
        ej = j;
        eo = o;
    } else {
        // Depth first, children in order of first appearance, each node
        // tested after its subtree: the end node is the first accepted
        // node in that post-order (the root always accepts).  A node
        // (j, o) is owned by draft o; its first child is (j + 1, o), its
        // parent (j - 1, own[j - 1][o]), and its next sibling the lowest
        // later draft through the parent that owns a node at depth j.
        signed char* sib = s_sib[w];
        for (int i = lane + K; i < (Lb + 1) * K; i += 32) {  // depths 1..Lb (owned nodes only)
            const int j = i / K, k = i % K;
            int nx = -1;
            if (own[i] == k) {
                const int par = own[(j - 1) * K + k];
                for (int k3 = k + 1; k3 < K; ++k3)
                    if (own[(j - 1) * K + k3] == par && own[j * K + k3] == k3) {
                        nx = k3;
                        break;
                    }
            }
            sib[i] = (signed char)nx;
        }
        __syncwarp();
        if (lane != 0) return;
        int jj = Lb, o = 0;  // the leftmost deepest node
        for (;;) {
            if (jj == 0) {
                ej = 0;
                eo = 0;
                break;
            }
            if (uu[o * L + jj - 1] <= val[jj * K + o]) {
                ej = jj;
                eo = o;
                break;
            }
            const int nx = sib[jj * K + o];
            if (nx >= 0) {
                o = nx;   // the next sibling's subtree, from its leftmost deepest node
                jj = Lb;  // (a draft's own nodes run down to depth Lb)
            } else {
                o = own[(jj - 1) * K + o];  // the parent
                --jj;
            }
        }
    }
    // the correction (or bonus) token is drawn at the end node afterwards;
    // a leaf's residual is p P (mass p; p = 1 in the token rule)
    const size_t se = s0 + (size_t)ej * K + eo;
    const bool leaf = ej == Lb;
    pb.accept_len[b] = ej;
    pb.accept_draft[b] = eo;
    pb.ws.endn[b] = (int)(se | (leaf ? (1u << 30) : 0u));
    if (pb.residual_mass)
        pb.residual_mass[b] = leaf ? (token || Lb == 0 ? 1.f : 1.f - pb.ws.pbar[se]) : pb.ws.S[se];
}

}  // namespace

// ------------------------------------------------------------------------
// launchers

cudaError_t launch_prep(const Problem& pb, cudaStream_t st)
{
    const int warps = 4;  // one warp per request
    prep_kernel<<<(pb.B + warps - 1) / warps, 32 * warps, 0, st>>>(pb);
    return cudaGetLastError();
}

cudaError_t launch_argmax(const Problem& pb, cudaStream_t st)
{
    const size_t n = slot_count(pb.B, pb.K, pb.L);
    if (n == 0) return cudaSuccess;
    if (pb.dtype == SDV_BF16)
        argmax_kernel<SDV_BF16><<<(unsigned)n, 256, 0, st>>>(pb);
    else
        argmax_kernel<SDV_F32><<<(unsigned)n, 256, 0, st>>>(pb);
    return cudaGetLastError();
}

cudaError_t launch_decide(const Problem& pb, bool greedy, cudaStream_t st)
{
    decide_kernel<<<(pb.B + kDecideWarps - 1) / kDecideWarps, 32 * kDecideWarps, 0, st>>>(pb, greedy ? 1 : 0);
    return cudaGetLastError();
}

}  // namespace sdv
