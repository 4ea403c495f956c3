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
#include "sdv_device.cuh"

namespace cg = cooperative_groups;

namespace sdv {
namespace {

// Cluster exchange words published by each CTA after the normaliser sweep.
enum { X_MT, X_MD, X_ZT, X_ZD, X_NT, X_ND, X_FT, X_FD, X_PT, X_PD, X_WORDS };

// Shared-memory layout of the node kernel (after the two row slices).
struct NodeSmem {
    float part[kMaxThreads];          // per-thread partial mass of the last residual sweep
    float partT[kMaxThreads];         // per-thread partial target mass, in this CTA's units
    float xbuf[2][kMaxCluster][12];   // cluster exchange, double-buffered
    float red[64];                    // block sums
    float redm[64];                   // block maxima
    int ired[2][32];                  // block sums of counts
    unsigned long long firstT, firstD;  // (first index of the CTA maximum << 32) | partner logit bits
    uint64_t bar[2];                  // row-slice mbarriers
    float gT[SDV_MAX_K], gD[SDV_MAX_K];  // target / draft logits at each draft's drawn token
    // scalar state of thread 0
    float zT, zD;                     // normalisers, in units of the row's global reference
    float zrestT, zrestD;             // the same without the unique maximum
    float sclT[kMaxCluster], sclD[kMaxCluster];  // CTA r's unit 2^(x c - m_r c) in global units
    float negT[kMaxCluster], negD[kMaxCluster];   // CTA references -(m_r c)
    float gnegT, gnegD;               // global references -(m c)
    float MT, MD;                     // row maxima
    float emaxT, emaxD;               // e of the unique maxima (global units)
    int uT, uD;                       // unique maxima, or -1
    float duT, tuD;                   // draft logit at uT, target logit at uD
    float S, D, cbar;                 // residual recursion
    float Pbs, Qbs;                   // 1 - P and 1 - Q at the shared dominant token x*
    float Rs, Ts, Rj;                 // R_j(x*), residual mass elsewhere, R_j(x*) before clamping
    float aT, aD;                     // this CTA's sweep weights
    float tot[kMaxCluster];           // per-CTA mass of the sampled distribution (global units)
    float thr, base, unit;            // sampling threshold, mass before CTA rstar, its unit
    int use_res, rstar, bad, pick;
    int spec_x[2];                    // indices whose residual weight is exact, or -1
    float spec_w[2];                  // their exact weights
    float pick_base;
};

}  // namespace

size_t node_smem_bytes(int units_per_cta) { return (size_t)units_per_cta * 16 * 2 + sizeof(NodeSmem); }

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
// node kernel

// Cluster-wide exchange: thread 0's n words are written, by the lanes of
// warp 0 in parallel, into slot [rank] of buffer `par` of every CTA; after
// the cluster barrier each CTA reads all slots locally.
__device__ __forceinline__ void cluster_publish(cg::cluster_group& cl, NodeSmem* sm, int par, int rank, int C,
                                                const float* v, int n)
{
    if (threadIdx.x < 32) {  // lane r writes to CTA r; the values are thread 0's
        const int lane = threadIdx.x;
        float* dst = lane < C ? cl.map_shared_rank(&sm->xbuf[par][rank][0], lane) : nullptr;
        for (int i = 0; i < n; ++i) {
            const float x = __shfl_sync(0xffffffffu, v[i], 0);
            if (lane < C) dst[i] = x;
        }
    }
    cl.sync();
}

// The residual term of one element as every sweep computes it, in fp32.
__device__ __forceinline__ float res_term(float eT, float eD, float aT, float aD)
{
    return fmaxf(__fmaf_rn(eT, aT, -__fmul_rn(eD, aD)), 0.f);
}

struct ProbD {
    float P, Pbar;
};

// alpha P(x) - beta Q(x) with alpha = 1 - pbar and beta = 1 + cbar.  For a
// row's dominant token it is written with complements, so that nothing of
// order one cancels when P and Q are both close to 1; the complements are
// small and fp32 keeps their relative precision.  Elsewhere P and Q are at
// most 1/2 and the direct form is the accurate one.
__device__ __forceinline__ float g_diff(const ProbD& P, const ProbD& Q, float pbar, float cbar, bool dominant)
{
    if (dominant) return (((Q.Pbar - P.Pbar) + pbar * P.Pbar) + cbar * Q.Pbar) - (pbar + cbar);
    return (1.f - pbar) * P.P - (1.f + cbar) * Q.P;
}

// P(x) of the target row (is_t) or Q(x) of the draft row, in fp64, from the
// logit at x.  The unique maximum uses the sum without it, so 1 - P is exact.
__device__ __forceinline__ ProbD prob_at(const NodeSmem* sm, bool is_t, int x, float logit, float c)
{
    ProbD o;
    const int u = is_t ? sm->uT : sm->uD;
    const float z = is_t ? sm->zT : sm->zD;
    if (x == u) {
        o.P = (is_t ? sm->emaxT : sm->emaxD) / z;
        o.Pbar = (is_t ? sm->zrestT : sm->zrestD) / z;
    } else {
        o.P = ex2(fmaf(logit, c, is_t ? sm->gnegT : sm->gnegD)) / z;
        o.Pbar = 1.f - o.P;
    }
    return o;
}

// Sweep weights of CTA r: P(x) = e_r(x) sclT_r / zT, Q likewise.
__device__ __forceinline__ void sweep_weights(const NodeSmem* sm, int r, float p, float cbar, float& aT, float& aD)
{
    aT = p * sm->sclT[r] / sm->zT;
    aD = (1.f + cbar) * sm->sclD[r] / sm->zD;
}

// Per-row state from the exchanged per-CTA statistics, computed by warp 0
// with lane r holding CTA r.  Every sum is of nonnegative terms, so fp32
// keeps its relative precision.
__device__ void row_state_warp(NodeSmem* sm, const float (*xb)[12], int C, bool is_t, float c)
{
    const int lane = threadIdx.x & 31;
    const bool act = lane < C;
    const int iM = is_t ? X_MT : X_MD, iZ = is_t ? X_ZT : X_ZD, iN = is_t ? X_NT : X_ND;
    const int iF = is_t ? X_FT : X_FD, iP = is_t ? X_PT : X_PD;
    const float m = act ? xb[lane][iM] : -INFINITY;
    const int n = act ? __float_as_int(xb[lane][iN]) : 0;
    const float zr = act ? xb[lane][iZ] : 0.f;
    const float M = warp_max_nan(m);
    const float gneg = -(M * c);
    const float neg = -(m * c);
    // shift between the CTA's reference and the row's (gneg - neg is exact
    // when the two maxima are close, which is when the CTA's mass matters)
    const float scl = (n > 0 || zr > 0.f) ? ex2(gneg - neg) : 0.f;
    const float em = n > 0 ? ex2(fmaf(m, c, neg)) : 0.f;
    const float contrib = n > 0 ? scl * zr + scl * (float)n * em : scl * zr;
    const bool ismax = act && m == M && n > 0;
    const float z = warp_sum(contrib);
    const float zrest = warp_sum(ismax ? scl * zr : contrib);  // without the maximum's own mass
    int nmax = ismax ? n : 0;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) nmax += __shfl_xor_sync(0xffffffffu, nmax, o);
    const unsigned bm = __ballot_sync(0xffffffffu, ismax);
    const int rs = bm ? __ffs(bm) - 1 : 0;
    const float em_s = __shfl_sync(0xffffffffu, em, rs);
    const int f_s = __shfl_sync(0xffffffffu, act ? __float_as_int(xb[lane][iF]) : -1, rs);
    const float p_s = __shfl_sync(0xffffffffu, act ? xb[lane][iP] : 0.f, rs);
    if (act) {
        if (is_t) {
            sm->sclT[lane] = scl;
            sm->negT[lane] = neg;
        } else {
            sm->sclD[lane] = scl;
            sm->negD[lane] = neg;
        }
    }
    if (lane == 0) {
        const bool uniq = nmax == 1;
        if (is_t) {
            sm->MT = M;
            sm->gnegT = gneg;
            sm->zT = z;
            sm->zrestT = zrest;
            sm->emaxT = em_s;
            sm->uT = uniq ? f_s : -1;
            sm->duT = uniq ? p_s : 0.f;
        } else {
            sm->MD = M;
            sm->gnegD = gneg;
            sm->zD = z;
            sm->zrestD = zrest;
            sm->emaxD = em_s;
            sm->uD = uniq ? f_s : -1;
            sm->tuD = uniq ? p_s : 0.f;
        }
    }
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
    const size_t sbase = ((size_t)b * (L + 1) + j) * K;
    const size_t s = sbase + k;
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
        sm->firstT = sm->firstD = ~0ull;
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
    // logits at the drawn tokens, fetched while the slices land
    if (!leaf && tid >= k && tid < K && pb.ws.owner[sbase + tid] == k) {
        const int y = pb.tokens[((size_t)b * K + tid) * L + j];
        sm->gT[tid] = E::load(gT, y);
        sm->gD[tid] = E::load(gD, y);
    }

    bool timed_out = false;
    // ---- maxima of this CTA's slices (NaN-propagating) ----
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
    block_max2(mT, mD, sm->redm);
    const float c = pb.c;
    // this CTA's reference: e_r(x) = 2^(x c - m_r c)
    const float nTr = -(mT * c);
    const float nDr = -(mD * c);
    const float emT = ex2(fmaf(mT, c, nTr));

    // ---- normalisers: the CTA maxima are counted apart ----
    float zT = 0.f, zD = 0.f;
    int cntT = 0, cntD = 0;
    if (mlT == mT) {  // this thread holds the CTA's target maximum
        int first = -1;
        for (int u = cu0; u < cu1; ++u) {
            float t[EPU];
            unpack_masked<DT>(smT[u], (u_base + u) * EPU, V, t);
            for (int e = 0; e < EPU; ++e) {
                if (t[e] == mT) {
                    if (cntT++ == 0) first = u * EPU + e;
                } else {
                    zT += ex2(fmaf(t[e], c, nTr));
                }
            }
        }
        if (first >= 0) {
            const float partner = leaf ? 0.f : [&] {
                float d[EPU];
                Elem<DT>::unpack(smD[first / EPU], d);
                return d[first % EPU];
            }();
            atomicMin(&sm->firstT,
                      ((unsigned long long)(u_base * EPU + first) << 32) | __float_as_uint(partner));
        }
    } else {
        for (int u = cu0; u < cu1; ++u) {
            float t[EPU];
            unpack_masked<DT>(smT[u], (u_base + u) * EPU, V, t);
#pragma unroll
            for (int e = 0; e < EPU; ++e) zT += ex2(fmaf(t[e], c, nTr));
        }
    }
    if (!leaf) {
        if (mlD == mD) {
            int first = -1;
            for (int u = cu0; u < cu1; ++u) {
                float d[EPU];
                unpack_masked<DT>(smD[u], (u_base + u) * EPU, V, d);
                for (int e = 0; e < EPU; ++e) {
                    if (d[e] == mD) {
                        if (cntD++ == 0) first = u * EPU + e;
                    } else {
                        zD += ex2(fmaf(d[e], c, nDr));
                    }
                }
            }
            if (first >= 0) {
                float t[EPU];
                Elem<DT>::unpack(smT[first / EPU], t);
                atomicMin(&sm->firstD,
                          ((unsigned long long)(u_base * EPU + first) << 32) | __float_as_uint(t[first % EPU]));
            }
        } else {
            for (int u = cu0; u < cu1; ++u) {
                float d[EPU];
                unpack_masked<DT>(smD[u], (u_base + u) * EPU, V, d);
#pragma unroll
                for (int e = 0; e < EPU; ++e) zD += ex2(fmaf(d[e], c, nDr));
            }
        }
    }
    sm->partT[tid] = zT + (float)cntT * emT;
    block_sum_f2i2_t0(zT, zD, cntT, cntD, sm->red, sm->ired);
    {
        const unsigned long long fT = sm->firstT, fD = sm->firstD;
        float v[X_WORDS];
        v[X_MT] = mT;
        v[X_MD] = mD;
        v[X_ZT] = zT;
        v[X_ZD] = zD;
        v[X_NT] = __int_as_float(cntT);
        v[X_ND] = __int_as_float(cntD);
        v[X_FT] = __int_as_float((int)(fT >> 32));
        v[X_FD] = __int_as_float((int)(fD >> 32));
        v[X_PT] = __uint_as_float((unsigned)(fT & 0xffffffffu));
        v[X_PD] = __uint_as_float((unsigned)(fD & 0xffffffffu));
        cluster_publish(cl, sm, 1, rank, C, v, X_WORDS);
    }

    // ---- scalar state (warp 0 / thread 0, kept in shared memory) ----
    const float pbar = (j == 0 || pb.mode == SDV_MODE_TOKEN) ? 0.f : pb.ws.pbar[s];
    const float p = 1.f - pbar;
    if (tid < 32) {
        row_state_warp(sm, sm->xbuf[1], C, true, c);
        if (!leaf) row_state_warp(sm, sm->xbuf[1], C, false, c);
        __syncwarp();
    }
    if (tid == 0) {
        const bool bad = !(isfinite(sm->MT) && isfinite(sm->zT) && sm->zT > 0.f) ||
                         (!leaf && !(isfinite(sm->MD) && isfinite(sm->zD) && sm->zD > 0.f));
        sm->bad = bad;
        if (bad && rank == 0) {
            atomicOr(&pb.ws.req[b], SDV_REQ_NONFINITE);
            if (pb.device_status) atomicOr(pb.device_status, SDV_REQ_NONFINITE);
        }
        // The token that is the unique maximum of both rows: its residual
        // term shrinks geometrically through the recursion (p P and C_j Q
        // both near 1), so it is carried apart, in a form with small terms.
        const int xs = (!leaf && sm->uT >= 0 && sm->uT == sm->uD) ? sm->uT : -1;
        sm->spec_x[0] = xs;
        sm->spec_x[1] = -1;
        sm->spec_w[0] = sm->spec_w[1] = 0.f;
        sm->Pbs = xs >= 0 ? sm->zrestT / sm->zT : 0.f;  // 1 - P(x*)
        sm->Qbs = xs >= 0 ? sm->zrestD / sm->zD : 0.f;  // 1 - Q(x*)
        sm->Rs = 0.f;
        sm->Ts = 0.f;
        sm->use_res = 0;
        sm->S = p;
        sm->D = 1.f;
        sm->cbar = 0.f;
    }

    // ---- residual recursion over the draws of the drafts through the node ----
    // R_j = max(p P - C_j Q, 0), S_j = sum R_j, D_j = 1 - p + S_j,
    // C_1 = 1, C_{j+1} = C_j + D_j; thread 0 keeps pbar = 1 - p and
    // cbar = C_j - 1, which stay accurate where p -> 1 and C -> 1.
    // At the shared dominant token x*, with T_j the residual mass elsewhere:
    //   R_1(x*) = p P(x*) - Q(x*) = Qbar - Pbar - pbar + pbar Pbar,
    //   R_j(x*) = R_{j-1}(x*) Qbar - (pbar + T_{j-1}) (1 - Qbar).
    int par = 1;
    bool first_draw = true;
    if (!leaf) {
        for (int k2 = k; k2 < K; ++k2) {
            if (pb.ws.owner[sbase + k2] != k) continue;
            if (tid == 0) {
                const int y = pb.tokens[((size_t)b * K + k2) * L + j];
                const int xs = sm->spec_x[0];
                const float D = sm->D;
                const float cnew = first_draw ? 0.f : sm->cbar + D;
                const float Pbs = sm->Pbs, Qbs = sm->Qbs;
                // R_j(x*) before clamping, for this draw's sweep
                const float Rj = first_draw ? ((Qbs - Pbs) - pbar) + pbar * Pbs
                                            : sm->Rs * Qbs - (pbar + sm->Ts) * (1.f - Qbs);
                sm->Rj = Rj;
                float R, Qy, abar_num;
                if (y == xs) {
                    Qy = 1.f - Qbs;
                    R = first_draw ? (1.f - pbar) * (1.f - Pbs) : sm->Rs;  // R_{j-1}(x*)
                    abar_num = fmaxf(-Rj, 0.f);                              // D Q - R
                } else {
                    const ProbD Py = prob_at(sm, true, y, sm->gT[k2], c);
                    const ProbD Qp = prob_at(sm, false, y, sm->gD[k2], c);
                    Qy = Qp.P;
                    // R_{j-1}(y); C_0 = 0 for the first draw
                    R = first_draw ? p * Py.P : fmaxf(g_diff(Py, Qp, pbar, sm->cbar, false), 0.f);
                    abar_num = fmaxf(-g_diff(Py, Qp, pbar, cnew, false), 0.f);  // C_j Q - p P
                }
                // a = min(R / (D Q(y)), 1).  D and Q(y) can both be ~1e-30 at
                // low temperature: divide twice instead of forming D Q(y),
                // which would underflow fp32.
                float a, abar;
                const float ratio = (D > 0.f && Qy > 0.f) ? (R / D) / Qy : INFINITY;
                if (ratio >= 1.f) {
                    a = 1.f;
                    abar = 0.f;
                } else if (!(R > 0.f)) {
                    a = 0.f;
                    abar = 1.f;
                } else {
                    a = ratio;
                    abar = fminf((abar_num / D) / Qy, 1.f);
                }
                sm->cbar = cnew;
                if (rank == 0) {
                    pb.ws.a[sbase + k2] = a;
                    if (pb.mode != SDV_MODE_TOKEN) {
                        const size_t sc = sbase + K + k2;
                        if (pb.ws.owner[sc] == k2) pb.ws.pbar[sc] = abar;  // child first reached here
                    }
                }
                float wT, wD;
                sweep_weights(sm, rank, p, cnew, wT, wD);
                sm->aT = wT;
                sm->aD = wD;
            }
            __syncthreads();
            const float aT = sm->aT, aD = sm->aD;
            const int xs = sm->spec_x[0];
            float w = 0.f;
            if (xs >= (u_base + cu0) * EPU && xs < (u_base + cu1) * EPU) {
                // this thread holds x*: leave it out, its term is carried apart
                for (int u = cu0; u < cu1; ++u) {
                    float t[EPU], d[EPU];
                    unpack_masked<DT>(smT[u], (u_base + u) * EPU, V, t);
                    unpack_masked<DT>(smD[u], (u_base + u) * EPU, V, d);
                    for (int e = 0; e < EPU; ++e)
                        if ((u_base + u) * EPU + e != xs)
                            w += res_term(ex2(fmaf(t[e], c, nTr)), ex2(fmaf(d[e], c, nDr)), aT, aD);
                }
            } else {
                for (int u = cu0; u < cu1; ++u) {
                    float t[EPU], d[EPU];
                    unpack_masked<DT>(smT[u], (u_base + u) * EPU, V, t);
                    unpack_masked<DT>(smD[u], (u_base + u) * EPU, V, d);
#pragma unroll
                    for (int e = 0; e < EPU; ++e) w += res_term(ex2(fmaf(t[e], c, nTr)), ex2(fmaf(d[e], c, nDr)), aT, aD);
                }
            }
            sm->part[tid] = w;
            w = block_sum_t0(w, sm->red);
            par ^= 1;
            cluster_publish(cl, sm, par, rank, C, &w, 1);
            if (tid == 0) {
                float Sj = 0.f;
                for (int r = 0; r < C; ++r) {
                    Sj += sm->xbuf[par][r][0];
                    sm->tot[r] = sm->xbuf[par][r][0];
                }
                const int xs = sm->spec_x[0];
                if (xs >= 0) {
                    // the sweeps left x* out: their sum is the mass elsewhere
                    const int rx = (xs / EPU) / sh.units_per_cta;
                    const float Rs = fmaxf(sm->Rj, 0.f);
                    sm->Ts = Sj;
                    sm->Rs = Rs;
                    Sj += Rs;
                    sm->spec_w[0] = Rs;
                    sm->tot[rx] += Rs;
                    if (rx == rank) sm->part[((xs / EPU) - u_base) / sh.units_per_thr] += Rs;
                }
                sm->S = fmaxf(Sj, 0.f);
                sm->D = pbar + sm->S;
                sm->use_res = sm->S > 0.f;
            }
            first_draw = false;
        }
    }

    // ---- node outputs and the candidate correction ----
    if (tid == 0) {
        const float S = sm->S, D = sm->D;
        const float h = leaf ? p : (D > 0.f ? S / D : 1.f);
        if (rank == 0) {
            pb.ws.h[s] = h;
            pb.ws.S[s] = S;
        }
    }
    if (tid < 32) {
        // lane r holds CTA r's mass of the sampled distribution
        __syncwarp();
        const int lane = tid;
        const bool act = lane < C;
        const bool ures = sm->use_res != 0;
        float tr = 0.f;
        if (act) {
            if (ures) {
                tr = sm->tot[lane];
            } else {  // sample P: per-CTA target mass in global units
                const int n = __float_as_int(sm->xbuf[1][lane][X_NT]);
                const float m = sm->xbuf[1][lane][X_MT];
                const float em = n > 0 ? ex2(fmaf(m, c, sm->negT[lane])) : 0.f;
                tr = sm->sclT[lane] * (sm->xbuf[1][lane][X_ZT] + (float)n * em);
            }
        }
        float incl = tr;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += v;
        }
        const float Stot = __shfl_sync(0xffffffffu, incl, 31);
        const float u = pb.sample_u[((size_t)b * K + k) * (L + 1) + j];
        const float thr = u * Stot;
        const unsigned cross = __ballot_sync(0xffffffffu, act && tr > 0.f && incl > thr);
        const unsigned nz = __ballot_sync(0xffffffffu, act && tr > 0.f);
        // the first CTA whose running mass exceeds u * S, else (rounding) the
        // last CTA of nonzero mass
        const int rs = cross ? __ffs(cross) - 1 : (nz ? 31 - __clz(nz) : -1);
        const float base = __shfl_sync(0xffffffffu, incl - tr, rs < 0 ? 0 : rs);
        if (lane == 0) {
            sm->rstar = (sm->bad || rs < 0) ? -1 : rs;
            sm->thr = thr;
            sm->base = base;
            // the residual partials are in probability units; the target
            // partials in units of CTA rstar's reference
            sm->unit = (ures || rs < 0) ? 1.f : sm->sclT[rs];
        }
    }
    __syncthreads();
    const bool use_res = sm->use_res != 0;
    const int rstar = sm->rstar;
    if (rank == rstar) {
        const float* parts = use_res ? sm->part : sm->partT;
        const float local = (sm->thr - sm->base) / sm->unit;
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
                float acc = excl;
                for (int t = t0; t < t1; ++t) {
                    if (parts[t] > 0.f) {
                        const bool hit = acc + parts[t] > local;
                        tsel = t;
                        tbase = acc;
                        if (hit && cm) break;
                    }
                    acc += parts[t];
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
            float acc = sm->pick_base;
            int chosen = -1, last = -1;
            for (int uu = cu0; uu < cu1 && chosen < 0; ++uu) {
                float t[EPU], d[EPU];
                unpack_masked<DT>(smT[uu], (u_base + uu) * EPU, V, t);
                if (use_res) unpack_masked<DT>(smD[uu], (u_base + uu) * EPU, V, d);
                for (int e = 0; e < EPU; ++e) {
                    const int x = (u_base + uu) * EPU + e;
                    const float eT = ex2(fmaf(t[e], c, nTr));
                    float wx = use_res ? res_term(eT, ex2(fmaf(d[e], c, nDr)), aT, aD) : eT;
                    if (use_res && x == sm->spec_x[0]) wx = sm->spec_w[0];
                    if (use_res && x == sm->spec_x[1]) wx = sm->spec_w[1];
                    if (wx > 0.f) {
                        acc += wx;
                        last = x;
                        if (acc > local) {
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
        val[i] = greedy ? __int_as_float(pb.ws.am[s0 + i]) : (token ? pb.ws.a[s0 + i] : pb.ws.h[s0 + i]);
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
    if (lane != 0) return;
    int ej = 0, eo = 0;
    if (greedy) {
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
        // depth first: children in order of first appearance, then the
        // node's own test; the first accepted node ends the search
        int stk_o[SDV_MAX_L + 1], stk_next[SDV_MAX_L + 1];
        int top = 0;
        stk_o[0] = 0;
        stk_next[0] = 0;
        for (;;) {
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
                break;
            }
            if (uu[o * L + jj - 1] <= val[jj * K + o]) {
                ej = jj;
                eo = o;
                break;
            }
            --top;
        }
    }
    pb.accept_len[b] = ej;
    pb.accept_draft[b] = eo;
    pb.out_token[b] = pb.ws.tok[s0 + (size_t)ej * K + eo];
    if (pb.residual_mass) pb.residual_mass[b] = pb.ws.S[s0 + (size_t)ej * K + eo];
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
    decide_kernel<<<(pb.B + kDecideWarps - 1) / kDecideWarps, 32 * kDecideWarps, 0, st>>>(pb, greedy ? 1 : 0);
    return cudaGetLastError();
}

}  // namespace sdv
