// sdv_kernels.cu -- sm_103a kernels for batched speculative-decoding
// verification.
//
// prep_kernel     per request: length and token checks, draft-trie owners.
// node_kernel     one thread-block cluster per trie node.  Each CTA holds a
//                 vocabulary slice of the node's target and draft rows in
//                 shared memory (1-D TMA bulk copies, mbarrier completion),
//                 so HBM is read once; every vocabulary-wide quantity is a
//                 sweep over shared memory plus a DSMEM exchange:
//                   row maxima and softmax normalisers,
//                   the residual recursion S_j = sum max(p P - C_j Q, 0),
//                   one inverse-CDF candidate sample per node.
//                 Rows: the target and draft rows of the node's owner draft
//                 (a leaf reads only its target row).
// argmax_kernel   greedy: one CTA per node, streaming argmax of the target.
// decide_kernel   one thread per request: the token-level walk, the
//                 depth-first block search or greedy matching over the
//                 node records; writes the outputs.
//
// The rules (SpecTr-GBV: Multi-Draft Block Verification Accelerating
// Speculative Decoding, sections 1 and 2) are stated in include/sdv.h.
#include <cooperative_groups.h>

#include "sdv_internal.h"

namespace cg = cooperative_groups;

namespace sdv {
namespace {

constexpr int kMaxThreads = 512;
constexpr int kMaxCluster = 16;
constexpr uint64_t kWaitNs = 2000000000ull;  // bounded waits: 2 s

// ------------------------------------------------------------------------
// PTX helpers

__device__ __forceinline__ float ex2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float max_nan(float a, float b)
{
    float r;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
    return r;
}

__device__ __forceinline__ uint32_t max_nan_bf16x2(uint32_t a, uint32_t b)
{
    uint32_t r;
    asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ uint64_t globaltimer()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_fence_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t phase)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(phase)
        : "memory");
    return ok != 0;
}

// Waits for phase `phase` of the barrier for at most kWaitNs.
__device__ bool mbar_wait_bounded(uint64_t* bar, uint32_t phase)
{
    const uint64_t t0 = globaltimer();
    while (!mbar_try_wait(bar, phase)) {
        if (globaltimer() - t0 > kWaitNs) return false;
    }
    return true;
}

// 1-D bulk copy global -> this CTA's shared memory, completing on `bar`.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// ------------------------------------------------------------------------
// element access: rows are held as 16-byte units (4 fp32 or 8 bf16)

template <int DT>
struct Elem;

template <>
struct Elem<SDV_F32> {
    static constexpr int kPerUnit = 4;
    static constexpr int kBytes = 4;
    __device__ static __forceinline__ void unpack(const uint4& u, float (&v)[4])
    {
        v[0] = __uint_as_float(u.x);
        v[1] = __uint_as_float(u.y);
        v[2] = __uint_as_float(u.z);
        v[3] = __uint_as_float(u.w);
    }
    __device__ static __forceinline__ float unit_max(const uint4& u, float m)
    {
        m = max_nan(m, __uint_as_float(u.x));
        m = max_nan(m, __uint_as_float(u.y));
        m = max_nan(m, __uint_as_float(u.z));
        return max_nan(m, __uint_as_float(u.w));
    }
    __device__ static __forceinline__ float load(const void* row, int x)
    {
        return __ldg(reinterpret_cast<const float*>(row) + x);
    }
};

template <>
struct Elem<SDV_BF16> {
    static constexpr int kPerUnit = 8;
    static constexpr int kBytes = 2;
    __device__ static __forceinline__ void unpack(const uint4& u, float (&v)[8])
    {
        v[0] = bf_lo(u.x);
        v[1] = bf_hi(u.x);
        v[2] = bf_lo(u.y);
        v[3] = bf_hi(u.y);
        v[4] = bf_lo(u.z);
        v[5] = bf_hi(u.z);
        v[6] = bf_lo(u.w);
        v[7] = bf_hi(u.w);
    }
    __device__ static __forceinline__ float unit_max(const uint4& u, float m)
    {
        uint32_t a = max_nan_bf16x2(max_nan_bf16x2(u.x, u.y), max_nan_bf16x2(u.z, u.w));
        return max_nan(m, max_nan(bf_lo(a), bf_hi(a)));
    }
    __device__ static __forceinline__ float load(const void* row, int x)
    {
        const unsigned short h = __ldg(reinterpret_cast<const unsigned short*>(row) + x);
        return __uint_as_float(static_cast<uint32_t>(h) << 16);
    }
};

// Elements of a unit at or past V read as -inf (no mass, never chosen).
template <int DT>
__device__ __forceinline__ void unpack_masked(const uint4& u, int x0, int V, float (&v)[Elem<DT>::kPerUnit])
{
    Elem<DT>::unpack(u, v);
    if (x0 + Elem<DT>::kPerUnit > V) {
#pragma unroll
        for (int e = 0; e < Elem<DT>::kPerUnit; ++e)
            if (x0 + e >= V) v[e] = -INFINITY;
    }
}

// ------------------------------------------------------------------------
// reductions

__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ float warp_max_nan(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = max_nan(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// Block-wide sum / max of two values; every thread gets the result.
// red must hold 64 floats; ends with a barrier so red can be reused.
__device__ void block_sum2(float& a, float& b, float* red)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    a = warp_sum(a);
    b = warp_sum(b);
    if (lane == 0) {
        red[warp] = a;
        red[32 + warp] = b;
    }
    __syncthreads();
    a = 0.f;
    b = 0.f;
    for (int w = 0; w < nw; ++w) {
        a += red[w];
        b += red[32 + w];
    }
    __syncthreads();
}

__device__ void block_max2(float& a, float& b, float* red)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    a = warp_max_nan(a);
    b = warp_max_nan(b);
    if (lane == 0) {
        red[warp] = a;
        red[32 + warp] = b;
    }
    __syncthreads();
    a = -INFINITY;
    b = -INFINITY;
    for (int w = 0; w < nw; ++w) {
        a = max_nan(a, red[w]);
        b = max_nan(b, red[32 + w]);
    }
    __syncthreads();
}

// Softmax of one row in fp64, from the fp32 sweep results.  The row
// maximum is excluded from `zrest`, so that P and 1 - P of a dominant
// token are both exact to fp64 rounding of fp32-accurate addends.
struct RowD {
    double z;      // sum of e(x) = 2^(x c - m c) over the row
    double zrest;  // the same without the elements equal to the maximum
    float emax;    // e at the maximum
    float neg;     // -(m c)
    int n;         // elements equal to the maximum
    int ux;        // index of the unique maximum, or -1
};

struct ProbD {
    double P, Pbar;
};

// Shared-memory layout of the node kernel (after the two row slices).
struct NodeSmem {
    float part[kMaxThreads];          // per-thread partial mass of the last residual sweep
    float partT[kMaxThreads];         // per-thread partial target mass (normaliser sweep)
    float xbuf[2][kMaxCluster][8];    // cluster exchange, double-buffered
    float red[64];                    // block reductions
    int ired[4][32];                  // block reductions of counts / indices
    uint64_t bar[2];                  // row-slice mbarriers
    // scalar state, written by thread 0 and read by every thread
    float aT, aD;                     // sweep weights p / Z_T and C_j / Z_D
    float tot[kMaxCluster];           // per-CTA mass of the sampled distribution
    float thr;                        // u * total mass
    int use_res;                      // sample the residual (else P)
    int rstar;                        // CTA holding the sample
    float base;                       // mass before CTA rstar
    int spec_x[2];                    // indices whose residual weight is exact (or -1)
    float spec_w[2];                  // their exact weights
    int bad;                          // a used row is not finite
    int pick;                         // sampling: chosen thread
    float pick_base;                  // sampling: mass before the chosen thread
    RowD rT, rD;                      // fp64 row state (thread 0)
    double S, D, cbar;                // residual recursion state (thread 0)
};

}  // namespace

size_t node_smem_bytes(int units_per_cta) { return (size_t)units_per_cta * 16 * 2 + sizeof(NodeSmem); }

namespace {

// ------------------------------------------------------------------------
// prep: one thread per request

__global__ void prep_kernel(Problem pb)
{
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= pb.B) return;
    const int K = pb.K, L = pb.L, V = pb.V;
    const int Lb = pb.lengths ? pb.lengths[b] : L;
    int st = 0;
    if (Lb < 0 || Lb > L) {
        st = SDV_REQ_BAD_LENGTH;
    } else {
        for (int k = 0; k < K; ++k)
            for (int j = 0; j < Lb; ++j) {
                const int t = pb.tokens[((size_t)b * K + k) * L + j];
                if (t < 0 || t >= V) st = SDV_REQ_BAD_TOKEN;
            }
    }
    pb.ws.req[b] = st;
    if (st) {
        if (pb.device_status) atomicOr(pb.device_status, st);
        return;
    }
    // owner[j][k]: lowest k2 whose first j tokens equal draft k's.  Drafts
    // share a prefix of length j iff they share the one of length j-1 and
    // token j-1.
    unsigned char* own = pb.ws.owner + (size_t)b * (L + 1) * K;
    for (int k = 0; k < K; ++k) own[k] = 0;
    for (int j = 1; j <= Lb; ++j) {
        for (int k = 0; k < K; ++k) {
            const int tk = pb.tokens[((size_t)b * K + k) * L + j - 1];
            int o = k;
            for (int k2 = 0; k2 < k; ++k2) {
                if (own[(j - 1) * K + k2] == own[(j - 1) * K + k] &&
                    pb.tokens[((size_t)b * K + k2) * L + j - 1] == tk) {
                    o = k2;
                    break;
                }
            }
            own[j * K + k] = (unsigned char)o;
        }
    }
    pb.ws.pbar[(size_t)b * (L + 1) * K] = 0.f;  // root weight 1
}

// ------------------------------------------------------------------------
// node kernel

// Cluster-wide exchange: thread 0 of every CTA publishes n (<= 8) words
// into slot [rank] of buffer `par` of every CTA; after the cluster barrier
// each CTA reads all slots locally.
__device__ __forceinline__ void cluster_publish(cg::cluster_group& cl, NodeSmem* sm, int par, int rank, int C,
                                                const float* v, int n)
{
    if (threadIdx.x == 0) {
        for (int r = 0; r < C; ++r) {
            float* dst = cl.map_shared_rank(&sm->xbuf[par][rank][0], r);
            for (int i = 0; i < n; ++i) dst[i] = v[i];
        }
    }
    cl.sync();
}

// Block-wide sum of two ints and minimum of two ints (thread 0's result).
__device__ void block_int4(int& s0, int& s1, int& m0, int& m1, int (*ired)[32])
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        s0 += __shfl_xor_sync(0xffffffffu, s0, o);
        s1 += __shfl_xor_sync(0xffffffffu, s1, o);
        m0 = min(m0, __shfl_xor_sync(0xffffffffu, m0, o));
        m1 = min(m1, __shfl_xor_sync(0xffffffffu, m1, o));
    }
    if (lane == 0) {
        ired[0][warp] = s0;
        ired[1][warp] = s1;
        ired[2][warp] = m0;
        ired[3][warp] = m1;
    }
    __syncthreads();
    s0 = s1 = 0;
    m0 = m1 = 0x7fffffff;
    for (int w = 0; w < nw; ++w) {
        s0 += ired[0][w];
        s1 += ired[1][w];
        m0 = min(m0, ired[2][w]);
        m1 = min(m1, ired[3][w]);
    }
    __syncthreads();
}

// The residual term of one element as every sweep computes it, in fp32.
__device__ __forceinline__ float res_term(float eT, float eD, float aT, float aD)
{
    return fmaxf(__fmaf_rn(eT, aT, -__fmul_rn(eD, aD)), 0.f);
}

template <int DT>
__device__ ProbD row_prob(const RowD& r, const char* g, int x, float c)
{
    ProbD o;
    if (x == r.ux) {
        o.P = (double)r.emax / r.z;
        o.Pbar = r.zrest / r.z;
    } else {
        const float e = ex2(fmaf(Elem<DT>::load(g, x), c, r.neg));
        o.P = (double)e / r.z;
        o.Pbar = 1.0 - o.P;
    }
    return o;
}

// alpha P(x) - beta Q(x) with alpha = 1 - pbar and beta = 1 + cbar, written
// with complements so that nothing of order one cancels when P and Q are
// both close to 1.
__device__ __forceinline__ double g_diff(const ProbD& P, const ProbD& Q, double pbar, double cbar)
{
    return Q.Pbar - P.Pbar + pbar * P.Pbar + cbar * Q.Pbar - pbar - cbar;
}

template <int DT>
__global__ void __launch_bounds__(kMaxThreads) node_kernel(Problem pb, Shape sh, int j_lo)
{
    using E = Elem<DT>;
    constexpr int EPU = E::kPerUnit;
    cg::cluster_group cl = cg::this_cluster();
    const int C = sh.cluster;
    const int rank = (int)cl.block_rank();
    const int tid = threadIdx.x;
    const int K = pb.K, L = pb.L, V = pb.V;
    const int BK = pb.B * K;
    const int slot_id = blockIdx.x / C;
    const int j = j_lo + slot_id / BK;
    const int b = (slot_id % BK) / K;
    const int k = slot_id % K;

    // Uniform over the cluster: only the prep kernel's bits are read here.
    if (pb.ws.req[b] & (SDV_REQ_BAD_LENGTH | SDV_REQ_BAD_TOKEN)) return;
    const int Lb = pb.lengths ? pb.lengths[b] : L;
    if (j > Lb) return;
    const size_t s = ((size_t)b * (L + 1) + j) * K + k;
    if (pb.ws.owner[s] != k) return;
    const bool leaf = j == Lb;

    extern __shared__ __align__(128) unsigned char smem_raw[];
    uint4* smT = reinterpret_cast<uint4*>(smem_raw);
    uint4* smD = smT + sh.units_per_cta;
    NodeSmem* sm = reinterpret_cast<NodeSmem*>(smD + sh.units_per_cta);

    const int n_units = (V + EPU - 1) / EPU;
    const int u_base = rank * sh.units_per_cta;
    const int nU = max(0, min(sh.units_per_cta, n_units - u_base));
    const int cu0 = min(tid * sh.units_per_thr, nU);
    const int cu1 = min(cu0 + sh.units_per_thr, nU);

    const size_t rowT = ((size_t)b * K + k) * (L + 1) + j;
    const size_t rowD = ((size_t)b * K + k) * L + j;
    const char* gT = static_cast<const char*>(pb.target) + rowT * (size_t)pb.stride * E::kBytes;
    const char* gD = leaf ? nullptr : static_cast<const char*>(pb.draft) + rowD * (size_t)pb.stride * E::kBytes;

    // ---- stage the slices of the node's rows into shared memory ----
    if (tid == 0) {
        mbar_init(&sm->bar[0], 1);
        mbar_init(&sm->bar[1], 1);
        mbar_fence_init();
    }
    __syncthreads();
    if (tid == 0 && nU > 0) {
        const uint32_t bytes = (uint32_t)nU * 16u;
        constexpr uint32_t kPiece = 32768;
        mbar_expect_tx(&sm->bar[0], bytes);
        for (uint32_t off = 0; off < bytes; off += kPiece)
            bulk_g2s(reinterpret_cast<char*>(smT) + off, gT + (size_t)u_base * 16 + off, min(kPiece, bytes - off),
                     &sm->bar[0]);
        if (!leaf) {
            mbar_expect_tx(&sm->bar[1], bytes);
            for (uint32_t off = 0; off < bytes; off += kPiece)
                bulk_g2s(reinterpret_cast<char*>(smD) + off, gD + (size_t)u_base * 16 + off,
                         min(kPiece, bytes - off), &sm->bar[1]);
        }
    }
    if (rank == 0 && tid == 0) pb.ws.tok[s] = -1;

    bool timed_out = false;
    // ---- row maxima (NaN-propagating) ----
    float mlT = -INFINITY, mlD = -INFINITY;
    if (nU > 0) {
        if (!mbar_wait_bounded(&sm->bar[0], 0)) timed_out = true;
        for (int u = cu0; u < cu1; ++u) {
            if ((u_base + u + 1) * EPU > V) {
                float v[EPU];
                unpack_masked<DT>(smT[u], (u_base + u) * EPU, V, v);
                for (int e = 0; e < EPU; ++e) mlT = max_nan(mlT, v[e]);
            } else {
                mlT = E::unit_max(smT[u], mlT);
            }
        }
        if (!leaf) {
            if (!mbar_wait_bounded(&sm->bar[1], 0)) timed_out = true;
            for (int u = cu0; u < cu1; ++u) {
                if ((u_base + u + 1) * EPU > V) {
                    float v[EPU];
                    unpack_masked<DT>(smD[u], (u_base + u) * EPU, V, v);
                    for (int e = 0; e < EPU; ++e) mlD = max_nan(mlD, v[e]);
                } else {
                    mlD = E::unit_max(smD[u], mlD);
                }
            }
        }
    }
    float mT = mlT, mD = mlD;
    block_max2(mT, mD, sm->red);
    {
        float v[2] = {mT, mD};
        cluster_publish(cl, sm, 0, rank, C, v, 2);
    }
    mT = -INFINITY;
    mD = -INFINITY;
    for (int r = 0; r < C; ++r) {
        mT = max_nan(mT, sm->xbuf[0][r][0]);
        mD = max_nan(mD, sm->xbuf[0][r][1]);
    }
    const float c = pb.c;
    // e(x) = 2^(x c - m c): the shift by the rounded m c is common to the
    // whole row and cancels in e(x) / sum e.
    const float negT = -(mT * c);
    const float negD = -(mD * c);
    const float emaxT = ex2(fmaf(mT, c, negT));
    const float emaxD = ex2(fmaf(mD, c, negD));

    // ---- softmax normalisers, the maxima counted apart ----
    float zT = 0.f, zD = 0.f;
    int cntT = 0, cntD = 0, firstT = 0x7fffffff, firstD = 0x7fffffff;
    if (mlT == mT) {  // this thread holds the target maximum
        for (int u = cu0; u < cu1; ++u) {
            float t[EPU];
            unpack_masked<DT>(smT[u], (u_base + u) * EPU, V, t);
            for (int e = 0; e < EPU; ++e) {
                if (t[e] == mT) {
                    ++cntT;
                    firstT = min(firstT, (u_base + u) * EPU + e);
                } else {
                    zT += ex2(fmaf(t[e], c, negT));
                }
            }
        }
    } else {
        for (int u = cu0; u < cu1; ++u) {
            float t[EPU];
            unpack_masked<DT>(smT[u], (u_base + u) * EPU, V, t);
#pragma unroll
            for (int e = 0; e < EPU; ++e) zT += ex2(fmaf(t[e], c, negT));
        }
    }
    if (!leaf) {
        if (mlD == mD) {
            for (int u = cu0; u < cu1; ++u) {
                float d[EPU];
                unpack_masked<DT>(smD[u], (u_base + u) * EPU, V, d);
                for (int e = 0; e < EPU; ++e) {
                    if (d[e] == mD) {
                        ++cntD;
                        firstD = min(firstD, (u_base + u) * EPU + e);
                    } else {
                        zD += ex2(fmaf(d[e], c, negD));
                    }
                }
            }
        } else {
            for (int u = cu0; u < cu1; ++u) {
                float d[EPU];
                unpack_masked<DT>(smD[u], (u_base + u) * EPU, V, d);
#pragma unroll
                for (int e = 0; e < EPU; ++e) zD += ex2(fmaf(d[e], c, negD));
            }
        }
    }
    sm->partT[tid] = zT + (float)cntT * emaxT;
    block_sum2(zT, zD, sm->red);
    block_int4(cntT, cntD, firstT, firstD, sm->ired);
    {
        float v[6] = {zT, zD, __int_as_float(cntT), __int_as_float(cntD), __int_as_float(firstT),
                      __int_as_float(firstD)};
        cluster_publish(cl, sm, 1, rank, C, v, 6);
    }

    // ---- scalar state (thread 0, fp64, kept in shared memory) ----
    RowD& rT = sm->rT;
    RowD& rD = sm->rD;
    const double p_in = (j == 0 || pb.mode == SDV_MODE_TOKEN) ? 0.0 : (double)pb.ws.pbar[s];
    const double pbar = p_in;
    const double p = 1.0 - pbar;
    if (tid == 0) {
        rT.zrest = rD.zrest = 0.0;
        rT.n = rD.n = 0;
        int fT = 0x7fffffff, fD = 0x7fffffff;
        for (int r = 0; r < C; ++r) {
            rT.zrest += (double)sm->xbuf[1][r][0];
            rD.zrest += (double)sm->xbuf[1][r][1];
            rT.n += __float_as_int(sm->xbuf[1][r][2]);
            rD.n += __float_as_int(sm->xbuf[1][r][3]);
            fT = min(fT, __float_as_int(sm->xbuf[1][r][4]));
            fD = min(fD, __float_as_int(sm->xbuf[1][r][5]));
        }
        rT.emax = emaxT;
        rD.emax = emaxD;
        rT.neg = negT;
        rD.neg = negD;
        rT.z = rT.n * (double)emaxT + rT.zrest;
        rD.z = rD.n * (double)emaxD + rD.zrest;
        rT.ux = rT.n == 1 ? fT : -1;
        rD.ux = rD.n == 1 ? fD : -1;
        const bool bad = !(isfinite(mT) && isfinite(rT.z) && rT.z > 0.0) ||
                         (!leaf && !(isfinite(mD) && isfinite(rD.z) && rD.z > 0.0));
        sm->bad = bad;
        if (bad && rank == 0) {
            atomicOr(&pb.ws.req[b], SDV_REQ_NONFINITE);
            if (pb.device_status) atomicOr(pb.device_status, SDV_REQ_NONFINITE);
        }
        sm->spec_x[0] = leaf ? -1 : rT.ux;
        sm->spec_x[1] = (leaf || rD.ux == rT.ux) ? -1 : rD.ux;
        sm->spec_w[0] = sm->spec_w[1] = 0.f;
        for (int r = 0; r < C; ++r)
            sm->tot[r] = sm->xbuf[1][r][0] + (float)__float_as_int(sm->xbuf[1][r][2]) * emaxT;
        sm->use_res = 0;
    }

    // ---- residual recursion over the draws of the drafts through the node ----
    // R_j = max(p P - C_j Q, 0), S_j = sum R_j, D_j = 1 - p + S_j,
    // C_1 = 1, C_{j+1} = C_j + D_j.  Thread 0 keeps the scalars in fp64 as
    // pbar = 1 - p and cbar = C_j - 1.
    double& S = sm->S;
    double& D = sm->D;
    double& cbar = sm->cbar;
    if (tid == 0) {
        S = p;
        D = 1.0;
        cbar = 0.0;
    }
    int par = 1;
    bool first = true;
    if (!leaf) {
        for (int k2 = k; k2 < K; ++k2) {
            if (pb.ws.owner[((size_t)b * (L + 1) + j) * K + k2] != k) continue;
            if (tid == 0) {
                const int y = pb.tokens[((size_t)b * K + k2) * L + j];
                const ProbD Py = row_prob<DT>(rT, gT, y, c);
                const ProbD Qy = row_prob<DT>(rD, gD, y, c);
                // R_{j-1}(y): C_0 = 0 for the first draw
                const double R = first ? p * Py.P : fmax(g_diff(Py, Qy, pbar, cbar), 0.0);
                const double cnew = first ? 0.0 : cbar + D;
                const double denom = D * Qy.P;
                double a, abar;
                if (!(denom > 0.0) || R >= denom) {
                    a = 1.0;
                    abar = 0.0;
                } else if (!(R > 0.0)) {
                    a = 0.0;
                    abar = 1.0;
                } else {
                    a = R / denom;
                    // 1 - a = (C_j Q(y) - p P(y)) / (D Q(y))
                    abar = fmin(fmax(-g_diff(Py, Qy, pbar, cnew), 0.0) / denom, 1.0);
                }
                cbar = cnew;
                if (rank == 0) {
                    pb.ws.a[((size_t)b * (L + 1) + j) * K + k2] = (float)a;
                    if (pb.mode != SDV_MODE_TOKEN) {
                        const size_t sc = ((size_t)b * (L + 1) + j + 1) * K + k2;
                        if (pb.ws.owner[sc] == k2) pb.ws.pbar[sc] = (float)abar;  // child first reached here
                    }
                }
                sm->aT = (float)(p / rT.z);
                sm->aD = (float)((1.0 + cbar) / rD.z);
            }
            __syncthreads();
            const float aT = sm->aT, aD = sm->aD;
            float w = 0.f;
            for (int u = cu0; u < cu1; ++u) {
                float t[EPU], d[EPU];
                unpack_masked<DT>(smT[u], (u_base + u) * EPU, V, t);
                unpack_masked<DT>(smD[u], (u_base + u) * EPU, V, d);
#pragma unroll
                for (int e = 0; e < EPU; ++e)
                    w += res_term(ex2(fmaf(t[e], c, negT)), ex2(fmaf(d[e], c, negD)), aT, aD);
            }
            sm->part[tid] = w;
            float dummy = 0.f;
            block_sum2(w, dummy, sm->red);
            par ^= 1;
            cluster_publish(cl, sm, par, rank, C, &w, 1);
            if (tid == 0) {
                // fp32 sweep sums, with the dominant tokens' terms replaced
                // by their exact values
                double Sj = 0.0;
                for (int r = 0; r < C; ++r) {
                    Sj += (double)sm->xbuf[par][r][0];
                    sm->tot[r] = sm->xbuf[par][r][0];
                }
                for (int i = 0; i < 2; ++i) {
                    const int x = sm->spec_x[i];
                    if (x < 0) continue;
                    const ProbD Px = row_prob<DT>(rT, gT, x, c);
                    const ProbD Qx = row_prob<DT>(rD, gD, x, c);
                    const double exact = fmax(g_diff(Px, Qx, pbar, cbar), 0.0);
                    const float f32 = res_term(ex2(fmaf(E::load(gT, x), c, negT)),
                                               ex2(fmaf(E::load(gD, x), c, negD)), aT, aD);
                    Sj += exact - (double)f32;
                    sm->spec_w[i] = (float)exact;
                    const int rx = (x / EPU) / sh.units_per_cta;
                    sm->tot[rx] += (float)exact - f32;
                    if (rx == rank) {
                        const int tx = ((x / EPU) - u_base) / sh.units_per_thr;
                        sm->part[tx] += (float)exact - f32;
                    }
                }
                S = fmax(Sj, 0.0);
                D = pbar + S;
                sm->use_res = S > 0.0;
            }
            first = false;
        }
    }

    // ---- node outputs and the candidate correction ----
    if (tid == 0) {
        const double h = leaf ? p : (D > 0.0 ? S / D : 1.0);
        if (rank == 0) {
            pb.ws.h[s] = (float)h;
            pb.ws.S[s] = (float)S;
        }
        if (!sm->use_res) {
            // sample P: per-CTA target mass
            for (int r = 0; r < C; ++r)
                sm->tot[r] = sm->xbuf[1][r][0] + (float)__float_as_int(sm->xbuf[1][r][2]) * emaxT;
        }
        float Stot = 0.f;
        for (int r = 0; r < C; ++r) Stot += sm->tot[r];
        const float u = pb.sample_u[((size_t)b * K + k) * (L + 1) + j];
        const float thr = u * Stot;
        int rstar = -1, last = -1;
        float run = 0.f, base = 0.f, last_base = 0.f;
        for (int r = 0; r < C; ++r) {
            if (sm->tot[r] > 0.f) {
                last = r;
                last_base = run;
                if (run + sm->tot[r] > thr) {
                    rstar = r;
                    base = run;
                    break;
                }
            }
            run += sm->tot[r];
        }
        if (rstar < 0) {
            rstar = last;
            base = last_base;
        }
        sm->rstar = sm->bad ? -1 : rstar;
        sm->base = base;
        sm->thr = thr;
    }
    __syncthreads();
    const bool use_res = sm->use_res != 0;
    const int rstar = sm->rstar;
    if (rank == rstar) {
        const float* parts = use_res ? sm->part : sm->partT;
        const float local = sm->thr - sm->base;
        // warp 0 finds the first thread whose running mass exceeds `local`
        if (tid < 32) {
            const int nthr = blockDim.x;
            const int per = (nthr + 31) / 32;
            const int t0 = tid * per, t1 = min(t0 + per, nthr);
            float lane_sum = 0.f;
            for (int t = t0; t < t1; ++t) lane_sum += parts[t];
            float incl = lane_sum;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float n = __shfl_up_sync(0xffffffffu, incl, o);
                if (tid >= o) incl += n;
            }
            const float excl = incl - lane_sum;
            const unsigned cm = __ballot_sync(0xffffffffu, lane_sum > 0.f && incl > local);
            const unsigned nz = __ballot_sync(0xffffffffu, lane_sum > 0.f);
            // the first crossing lane, else (rounding) the last lane of nonzero mass
            const int l = cm ? __ffs(cm) - 1 : (nz ? 31 - __clz(nz) : -1);
            int tsel = -1;
            float tbase = 0.f;
            if (tid == l) {
                float run = excl;
                for (int t = t0; t < t1; ++t) {
                    if (parts[t] > 0.f) {
                        const bool hit = run + parts[t] > local;
                        tsel = t;
                        tbase = run;
                        if (hit && cm) break;
                    }
                    run += parts[t];
                }
            }
            if (l >= 0) {
                tsel = __shfl_sync(0xffffffffu, tsel, l);
                tbase = __shfl_sync(0xffffffffu, tbase, l);
            }
            if (tid == 0) {
                sm->pick = tsel;
                sm->pick_base = tbase;
            }
        }
        __syncthreads();
        if (tid == sm->pick) {
            const float aT = sm->aT, aD = sm->aD;
            float run = sm->pick_base;
            int chosen = -1, last = -1;
            for (int uu = cu0; uu < cu1 && chosen < 0; ++uu) {
                float t[EPU], d[EPU];
                unpack_masked<DT>(smT[uu], (u_base + uu) * EPU, V, t);
                if (use_res) unpack_masked<DT>(smD[uu], (u_base + uu) * EPU, V, d);
                for (int e = 0; e < EPU; ++e) {
                    const int x = (u_base + uu) * EPU + e;
                    const float eT = ex2(fmaf(t[e], c, negT));
                    float wx = use_res ? res_term(eT, ex2(fmaf(d[e], c, negD)), aT, aD) : eT;
                    if (use_res && x == sm->spec_x[0]) wx = sm->spec_w[0];
                    if (use_res && x == sm->spec_x[1]) wx = sm->spec_w[1];
                    if (wx > 0.f) {
                        run += wx;
                        last = x;
                        if (run > local) {
                            chosen = x;
                            break;
                        }
                    }
                }
            }
            pb.ws.tok[s] = chosen >= 0 ? chosen : last;
        }
    }

    if (timed_out) {
        // give the copies in flight a second bounded chance before this
        // CTA's shared memory is released, then flag the request
        if (nU > 0) {
            mbar_wait_bounded(&sm->bar[0], 0);
            if (!leaf) mbar_wait_bounded(&sm->bar[1], 0);
        }
        if (tid == 0) {
            atomicOr(&pb.ws.req[b], SDV_DEV_TIMEOUT);
            if (pb.device_status) atomicOr(pb.device_status, SDV_DEV_TIMEOUT);
        }
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
// decision: one thread per request

__global__ void decide_kernel(Problem pb, int greedy)
{
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= pb.B) return;
    const int K = pb.K, L = pb.L;
    const int st = pb.ws.req[b];
    float* ap = pb.accept_prob ? pb.accept_prob + (size_t)b * K * L : nullptr;
    if (ap)
        for (int i = 0; i < K * L; ++i) ap[i] = 0.f;
    if (st) {
        pb.accept_len[b] = 0;
        pb.accept_draft[b] = 0;
        pb.out_token[b] = -1;
        if (pb.residual_mass) pb.residual_mass[b] = 0.f;
        if (pb.device_status) atomicOr(pb.device_status, st);
        return;
    }
    const int Lb = pb.lengths ? pb.lengths[b] : L;
    const unsigned char* own = pb.ws.owner + (size_t)b * (L + 1) * K;
    auto S = [&](int j, int k) { return ((size_t)b * (L + 1) + j) * K + k; };
    int ej = 0, eo = 0;
    if (greedy) {
        int best = -1, bestk = 0;
        for (int k = 0; k < K; ++k) {
            int m = 0;
            while (m < Lb && pb.tokens[((size_t)b * K + k) * L + m] == pb.ws.am[S(m, own[m * K + k])]) ++m;
            if (m > best) {
                best = m;
                bestk = k;
            }
            if (ap)
                for (int d = 0; d < Lb; ++d)
                    ap[k * L + d] =
                        pb.tokens[((size_t)b * K + k) * L + d] == pb.ws.am[S(d, own[d * K + k])] ? 1.f : 0.f;
        }
        ej = best;
        eo = own[best * K + bestk];
        pb.accept_len[b] = best;
        pb.accept_draft[b] = bestk;
        pb.out_token[b] = pb.ws.am[S(ej, eo)];
        if (pb.residual_mass) pb.residual_mass[b] = 1.f;
        return;
    }
    if (pb.mode == SDV_MODE_TOKEN) {
        if (ap)
            for (int k = 0; k < K; ++k)
                for (int d = 0; d < Lb; ++d) ap[k * L + d] = pb.ws.a[S(d, k)];
        int j = 0, o = 0;
        while (j < Lb) {
            int acc = -1;
            for (int k = 0; k < K && acc < 0; ++k)
                if (own[j * K + k] == o && pb.accept_u[((size_t)b * K + k) * L + j] <= pb.ws.a[S(j, k)]) acc = k;
            if (acc < 0) break;
            o = own[(j + 1) * K + acc];
            ++j;
        }
        ej = j;
        eo = o;
    } else {
        if (ap)
            for (int k = 0; k < K; ++k)
                for (int d = 0; d < Lb; ++d) ap[k * L + d] = pb.ws.h[S(d + 1, own[(d + 1) * K + k])];
        // depth-first: children in order of first appearance, then the
        // node's own test; the first accepted node ends the search
        int stk_o[SDV_MAX_L + 1], stk_next[SDV_MAX_L + 1];
        int top = 0;
        stk_o[0] = 0;
        stk_next[0] = 0;
        bool done = false;
        while (!done) {
            const int jj = top, o = stk_o[top];
            int child = -1;
            if (jj < Lb) {
                for (int k2 = stk_next[top]; k2 < K; ++k2) {
                    if (own[jj * K + k2] == o && own[(jj + 1) * K + k2] == k2) {
                        child = k2;
                        break;
                    }
                }
            }
            if (child >= 0) {
                stk_next[top] = child + 1;
                ++top;
                stk_o[top] = child;
                stk_next[top] = 0;
                continue;
            }
            if (jj == 0) {
                ej = 0;
                eo = 0;
                done = true;
            } else if (pb.accept_u[((size_t)b * K + o) * L + jj - 1] <= pb.ws.h[S(jj, o)]) {
                ej = jj;
                eo = o;
                done = true;
            } else {
                --top;
            }
        }
    }
    pb.accept_len[b] = ej;
    pb.accept_draft[b] = eo;
    pb.out_token[b] = pb.ws.tok[S(ej, eo)];
    if (pb.residual_mass) pb.residual_mass[b] = pb.ws.S[S(ej, eo)];
}

}  // namespace

// ------------------------------------------------------------------------
// launchers

cudaError_t launch_prep(const Problem& pb, cudaStream_t st)
{
    const int threads = 128;
    prep_kernel<<<(pb.B + threads - 1) / threads, threads, 0, st>>>(pb);
    return cudaGetLastError();
}

template <int DT>
static cudaError_t launch_nodes_t(const Problem& pb, const Shape& sh, int j_lo, int j_hi, cudaStream_t st)
{
    const long long n_slots = (long long)(j_hi - j_lo + 1) * pb.B * pb.K;
    if (n_slots <= 0) return cudaSuccess;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(n_slots * sh.cluster), 1, 1);
    cfg.blockDim = dim3(sh.threads, 1, 1);
    cfg.dynamicSmemBytes = (size_t)sh.smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = sh.cluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, node_kernel<DT>, pb, sh, j_lo);
}

cudaError_t launch_nodes(const Problem& pb, const Shape& sh, int j_lo, int j_hi, cudaStream_t st)
{
    return pb.dtype == SDV_BF16 ? launch_nodes_t<SDV_BF16>(pb, sh, j_lo, j_hi, st)
                                : launch_nodes_t<SDV_F32>(pb, sh, j_lo, j_hi, st);
}

cudaError_t prepare_node_kernel(const Shape& sh, int dtype)
{
    const void* fn = dtype == SDV_BF16 ? reinterpret_cast<const void*>(node_kernel<SDV_BF16>)
                                       : reinterpret_cast<const void*>(node_kernel<SDV_F32>);
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, sh.smem);
    if (e != cudaSuccess) return e;
    if (sh.cluster > 8) e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    return e;
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
    const int threads = 128;
    decide_kernel<<<(pb.B + threads - 1) / threads, threads, 0, st>>>(pb, greedy ? 1 : 0);
    return cudaGetLastError();
}

}  // namespace sdv
