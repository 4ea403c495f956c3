// sdv_kernels.cu -- the small kernels around the node kernel (which is in
// sdv_stream.cu).
//
// prep_kernel     one warp per request: length and token checks, the
//                 draft-trie owners, the depth-major list of inner trie
//                 nodes the node kernel works through.
// argmax_kernel   greedy: one CTA per node, streaming argmax of the target.
// gather_rows_kernel  one CTA per (request, draft): the rows verification
//                 reads, from host memory mapped into the device's address
//                 space into device tensors.
// (The decision and the correction draw are in sdv_sample.cu.)
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
    // lane k < K holds draft k's tokens, all loaded at once (L <= 16)
    int tk[SDV_MAX_L];
    int st = 0;
    if (Lb < 0 || Lb > L) {
        st = SDV_REQ_BAD_LENGTH;
    } else {
        const int* row = pb.tokens + ((size_t)b * K + lane) * L;
#pragma unroll
        for (int j = 0; j < SDV_MAX_L; ++j) tk[j] = lane < K && j < Lb ? row[j] : 0;
        int bad = 0;
#pragma unroll
        for (int j = 0; j < SDV_MAX_L; ++j) bad |= j < Lb && lane < K && (tk[j] < 0 || tk[j] >= V);
        if (__any_sync(0xffffffffu, bad)) st = SDV_REQ_BAD_TOKEN;
    }
    if (lane == 0) {
        pb.ws.req[b] = st;
        pb.ws.left[b] = 0;  // the node count below, for a valid request
        if (st && pb.device_status) atomicOr(pb.device_status, st);
    }
    if (st) return;
    // owner[j][k] = lowest k2 whose first j tokens equal draft k's: drafts
    // share a prefix of length j iff they share the one of length j-1 and
    // token j-1.  Lane k holds draft k.
    unsigned char* own = pb.ws.owner + (size_t)b * (L + 1) * K;
    int o = 0;
    if (lane < K) own[lane] = 0;
#pragma unroll
    for (int j = 1; j <= SDV_MAX_L; ++j) {
        if (j > Lb) break;
        const int t = lane < K ? tk[j - 1] : -1;
        int no = lane;
        for (int k2 = K - 1; k2 >= 0; --k2) {
            const int o2 = __shfl_sync(0xffffffffu, o, k2);
            const int t2 = __shfl_sync(0xffffffffu, t, k2);
            if (k2 <= lane && o2 == o && t2 == t) no = k2;
        }
        o = no;
        if (lane < K) own[j * K + lane] = (unsigned char)o;
    }
    // list the request's inner nodes by depth (for the node kernel) and
    // mark every weight below the root unwritten (-1: a parent's draw
    // writes it, and the child waits for a value of 0 or more).  Within a
    // depth, nodes with several draws (several sweeps) fill the list from
    // the front and one-draw nodes from the back, so that the longest work
    // of a depth is handed out first.  Leaves are not listed: a leaf has no
    // draws, and its target row is read by the bonus draw alone, once the
    // decision ends there.
    const size_t BK = (size_t)pb.B * K;
    int* const front = pb.ws.ncount;
    int* const back = pb.ws.ncount + (L + 1);
    int listed = 0;  // the request's inner nodes: the node kernel counts them down
    for (int j = 0; j <= Lb; ++j) {
        const bool node = j < Lb && lane < K && own[j * K + lane] == lane;
        int draws = 0;  // drafts through the node
        if (node)
            for (int k2 = 0; k2 < K; ++k2) draws += own[j * K + k2] == lane;
        const unsigned mh = __ballot_sync(0xffffffffu, node && draws > 1);
        const unsigned ml = __ballot_sync(0xffffffffu, node && draws == 1);
        int fb = 0, bb = 0;
        if (lane == 0 && mh) fb = atomicAdd(&front[j], __popc(mh));
        if (lane == 0 && ml) bb = atomicAdd(&back[j], __popc(ml));
        fb = __shfl_sync(0xffffffffu, fb, 0);
        bb = __shfl_sync(0xffffffffu, bb, 0);
        const size_t slot = ((size_t)b * (L + 1) + j) * K + lane;
        const unsigned below = (1u << lane) - 1;
        if (node && draws > 1) pb.ws.nodes[j * BK + fb + __popc(mh & below)] = (int)slot;
        if (node && draws == 1) pb.ws.nodes[j * BK + BK - 1 - (bb + __popc(ml & below))] = (int)slot;
        if (lane < K) pb.ws.wt[slot] = j == 0 ? make_float2(0.f, 1.f) : make_float2(-1.f, 0.f);  // root: p = 1
        listed += __popc(mh) + __popc(ml);
    }
    if (lane == 0) pb.ws.left[b] = listed;
}

// ------------------------------------------------------------------------
// greedy argmax: one CTA per inner node, streaming

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
    // inner nodes only: a leaf's argmax is taken where the decision ends there
    if (j >= Lb || pb.ws.owner[slot] != k) return;
    const size_t row = ((size_t)b * K + k) * (L + 1) + j;
    const uint4* g = reinterpret_cast<const uint4*>(static_cast<const char*>(pb.target) +
                                                    row * (size_t)pb.stride * E::kBytes);
    const int n_units = (V + EPU - 1) / EPU;
    float best = -INFINITY;
    int bidx = 0x7fffffff;
    bool bad = false;
    // four 16-byte loads in flight per thread; a thread's units increase,
    // so the first maximum it sees is its lowest index
    constexpr int U = 4;
    for (int u0 = threadIdx.x; u0 < n_units; u0 += U * blockDim.x) {
        uint4 w[U];
#pragma unroll
        for (int q = 0; q < U; ++q) {
            const int uu = u0 + q * blockDim.x;
            w[q] = uu < n_units ? __ldg(g + uu) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int q = 0; q < U; ++q) {
            const int uu = u0 + q * blockDim.x;
            if (uu >= n_units) break;
            float v[EPU];
            unpack_masked<DT>(w[q], uu * EPU, V, v);
#pragma unroll
            for (int e = 0; e < EPU; ++e) {
                bad |= (v[e] != v[e]) || (v[e] == INFINITY);
                if (v[e] > best) {
                    best = v[e];
                    bidx = uu * EPU + e;
                }
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
// gather of the rows verification reads: draft k owns its trie nodes from
// depth f on (f = 0 for k = 0; else one past the longest prefix it shares
// with a lower draft), so it brings target rows [f, L_b] and draft rows
// [f, L_b - 1]; without leaves, target rows [f, L_b - 1].  The reads cross the host link; many 16-byte loads per
// thread are kept in flight to cover its latency.

__device__ __forceinline__ void copy_bytes(const void* src, void* dst, size_t n)
{
    const uint4* s = static_cast<const uint4*>(src);
    uint4* d = static_cast<uint4*>(dst);
    const size_t n16 = n / 16;
    constexpr int U = 8;
    size_t i = threadIdx.x;
    for (; i + (U - 1) * blockDim.x < n16; i += U * blockDim.x) {
        uint4 v[U];
#pragma unroll
        for (int u = 0; u < U; ++u) v[u] = s[i + u * blockDim.x];
#pragma unroll
        for (int u = 0; u < U; ++u) d[i + u * blockDim.x] = v[u];
    }
    for (; i < n16; i += blockDim.x) d[i] = s[i];
}

__global__ void __launch_bounds__(256) gather_rows_kernel(GatherArgs a)
{
    const int K = a.K, L = a.L;
    const int b = blockIdx.x / K, k = blockIdx.x % K;
    const int Lb = a.lengths ? a.lengths[b] : L;
    if (Lb < 0 || Lb > L) return;
    __shared__ int first;
    if (threadIdx.x == 0) first = 0;
    __syncthreads();
    if ((int)threadIdx.x < k) {  // the prefix shared with lower draft threadIdx.x
        const int* t1 = a.tokens + ((size_t)b * K + k) * L;
        const int* t2 = a.tokens + ((size_t)b * K + threadIdx.x) * L;
        int m = 0;
        while (m < Lb && t1[m] == t2[m]) ++m;
        atomicMax(&first, m + 1);
    }
    __syncthreads();
    const int f = first;
    const size_t rb = (size_t)a.row_bytes;
    const int last = a.leaves ? Lb : Lb - 1;  // the deepest target row brought
    if (f <= last) {
        const size_t off = (((size_t)b * K + k) * (L + 1) + f) * rb;
        copy_bytes(static_cast<const char*>(a.host_target) + off, static_cast<char*>(a.target) + off,
                   (size_t)(last - f + 1) * rb);
    }
    if (f < Lb) {
        const size_t off = (((size_t)b * K + k) * L + f) * rb;
        copy_bytes(static_cast<const char*>(a.host_draft) + off, static_cast<char*>(a.draft) + off,
                   (size_t)(Lb - f) * rb);
    }
}

}  // namespace

// ------------------------------------------------------------------------
// launchers

cudaError_t launch_gather_rows(const GatherArgs& a, cudaStream_t st)
{
    const long long n = (long long)a.B * a.K;
    if (n == 0) return cudaSuccess;
    gather_rows_kernel<<<(unsigned)n, 256, 0, st>>>(a);
    return cudaGetLastError();
}

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

}  // namespace sdv
