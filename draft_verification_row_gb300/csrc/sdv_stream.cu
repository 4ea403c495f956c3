// sdv_stream.cu -- the node kernel: every vocabulary-row computation of a
// verification call, in one persistent launch.
//
// Two CTAs per SM, each verifying one draft-trie node at a time; the
// node's target and draft rows stream through shared memory:
//   pass 1 (from HBM): online maxima and softmax normalisers of both rows,
//           in a warp-uniform reference, the row maxima counted apart so
//           that 1 - P of a dominant token stays exact;
//   pass 2 (from L2, once per draw): the residual sweep
//           S_j = sum_x max(p P(x) - C_j Q(x), 0).  A node keeps its final
//           residual's description for the correction draw, which the
//           decision kernel takes (sdv_sample.cu) in a pass of its own.
// Only inner nodes are visited: a leaf has no draws (its residual is p P,
// of mass p), and its target row is read by the bonus draw alone, after
// the decision and only if the decision ends there.
// Warp 0 (metadata) takes nodes from the depth-major list the prep kernel
// built and fills a descriptor queue: draws, their tokens and logits.
// Warp 1 (copy) streams each node's rows in 12 KB-per-row chunks through a
// 3-stage ring with 1-D TMA bulk copies (mbarrier full/empty handshake),
// marked evict_last in L2 until the node's last pass, which is evict_first
// (so is the pass before a last sweep that may not be asked for).
// Warps 2..13 consume: a warp owns 64 contiguous 16-byte units of each
// chunk.  A node's weight p comes from its parent's write of it (a value
// below 0 means not yet written); waiting happens only before pass 2.  Every wait is
// bounded and a timeout is reported, never a hang or a trap.
//
// The rules computed are stated in include/sdv.h (SpecTr-GBV:
// Multi-Draft Block Verification Accelerating Speculative Decoding,
// sections 1 and 2).
#include <algorithm>

#include "sdv_device.cuh"
#include "sdv_internal.h"

namespace sdv {
namespace {

constexpr int kCtasPerSm = 2;            // two nodes in flight per SM
constexpr int kSW = 12;                  // consumer warps
constexpr int kCT = 32 * kSW;            // consumer threads
constexpr int kSThreads = kCT + 64;      // plus the metadata warp and the copy warp
constexpr int kUPT = 2;                  // 16-byte units per consumer thread per row per chunk
constexpr int kWU = 32 * kUPT;           // units per warp per chunk, contiguous
constexpr int kChunk = kCT * kUPT;       // units per row per chunk (12 KB)
constexpr int kStages = 3;               // 3 x 24 KB in flight per CTA
constexpr int kStash = 1;                // set-aside chunks a lane can hold (at most 2: d0, d1)
static_assert(kStash >= 1 && kStash <= 2, "a lane keeps at most two set-aside chunk indices");
constexpr int kQ = 4;                    // node descriptor queue depth
constexpr int kKseqRounds = 10;          // K-SEQ: search passes of a node with two draws or more

__device__ __forceinline__ void cbar_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kCT) : "memory"); }

__device__ __forceinline__ void mbar_arrive(uint64_t* bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_last()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t policy_evict_first()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ void bulk_g2s_hint(void* dst, const void* src, uint32_t bytes, uint64_t* bar, uint64_t pol)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(pol)
        : "memory");
}

// A node's weight is its own flag: the parent's draw writes the pair
// {1 - p, p} (the first 0 or more) in one 8-byte access and the child
// reads nothing else, so relaxed accesses suffice.
__device__ __forceinline__ float2 ld_weight(const float2* p)
{
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return make_float2(__uint_as_float((unsigned)v), __uint_as_float((unsigned)(v >> 32)));
}

__device__ __forceinline__ void st_weight(float2* p, float pbar, float pw)
{
    const unsigned long long v = (unsigned long long)__float_as_uint(pbar) |
                                 ((unsigned long long)__float_as_uint(pw) << 32);
    asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// What the metadata warp prepares for each node, ahead of its rows.
struct NodeDesc {
    int slot, b, j, k, nd;
    int dk[SDV_MAX_K];            // drafts of the draws, in index order
    int y[SDV_MAX_K];             // their tokens
    float gT[SDV_MAX_K], gD[SDV_MAX_K];  // target / draft logits at those tokens
};

struct StreamSmem {
    uint4 ring[kStages][2][kChunk];  // [stage][target, draft][units]
    uint64_t full[kStages], empty[kStages];
    uint64_t qfull[kQ], qempty[kQ];
    uint64_t lastdec;                // the consumers' word on a node's last sweep (block rules)
    NodeDesc qd[kQ];
    NodeDesc cur;                    // the consumers' copy of the current node
    float redf[5][kSW];
    int redi[4][kSW];
    int firstT, firstD;              // lowest index of each row's maximum
    uint4 stash[2][kCT][kStash][kUPT];  // set-aside units: [row][consumer thread][slot][unit]
    int abort;
    // scalar state (consumer thread 0)
    float MT, MD, gnegT, gnegD, zT, zD, zrestT, zrestD, emaxT, emaxD;
    int uT, uD;
    float S, D, cbar, pbar, pw, Pbs, Qbs, Rs, Ts, Rj, aT, aD, rD;  // pbar = 1 - p, pw = p
    int xs, bad;
    int skip_last, last_go;          // the node's last sweep: skipped here / issued by the copy warp
    // K-SEQ search (consumer thread 0): bracket [klo, khi] of rho, beta at
    // khi, this pass's points and their factors Z_D / (Z_T rho)
    float klo, khi, kbhi, krho[5], kf[5];
    int kdone, knp;
};

// Online statistics of one row, per thread, in a reference shared by the
// warp: e(x) = 2^(x c - m c) with m the largest logit the warp has seen in
// earlier chunks.  z sums the thread's elements below the row maximum; cnt
// counts its elements equal to it (first: the lowest such index).
//
// A chunk is summed against the reference of the chunks before it, and
// the reference moves after the chunk (one redux.sync, its latency hidden
// behind the chunk's exponentials).  A lane whose chunk reaches the
// reference (a new maximum, or a tie) does not add that chunk: it copies
// the chunk's units to its stash in shared memory (chunk indices d0, d1)
// and, after the pass, sums them against the final maximum, counting the
// elements equal to it apart.  Such chunks are rare (a handful per row
// per warp); a lane with more than kStash takes a synchronous, exact path.
struct Online {
    float m = -INFINITY;
    float neg = INFINITY;
    float z = 0.f;
    int cnt = 0;
    int first = 0x7fffffff;
    int nd = 0;
    int d0 = 0, d1 = 0;
};

// Unit maximum; the last unit of a row may extend past V.
template <int DT>
__device__ __forceinline__ float unit_max_masked(const uint4& u, int x0, int V)
{
    using E = Elem<DT>;
    if (x0 + E::kPerUnit <= V) return E::unit_max(u, -INFINITY);
    float v[E::kPerUnit];
    unpack_masked<DT>(u, x0, V, v);
    float um = -INFINITY;
#pragma unroll
    for (int e = 0; e < E::kPerUnit; ++e) um = max_nan(um, v[e]);
    return um;
}

// Move the warp's reference to wm (warp-uniform) if it is larger (or NaN).
__device__ __forceinline__ void online_rebase(Online& s, float wm, float c)
{
    if (wm > s.m || wm != wm) {
        // the offset is the rounded product, as every exponent argument
        // takes it: written so that it cannot fuse into the subtraction
        const float nneg = -__fmul_rn(wm, c);
        s.z = s.z * ex2(__fsub_rn(nneg, s.neg)) + (s.cnt > 0 ? (float)s.cnt * ex2(fmaf(s.m, c, nneg)) : 0.f);
        s.cnt = 0;
        s.first = 0x7fffffff;
        s.m = wm;
        s.neg = nneg;
    }
}

// Pairwise sum of a unit's 4 or 8 terms with packed adds: a dependency
// chain of depth log2(N) instead of N (the exponentials of a unit are
// independent).
template <int N>
__device__ __forceinline__ float tree_sum2(const float (&a)[N])
{
    static_assert(N == 4 || N == 8, "a unit holds 4 or 8 elements");
    float2 s = fadd2(make_float2(a[0], a[1]), make_float2(a[2], a[3]));
    if constexpr (N == 8) s = fadd2(s, fadd2(make_float2(a[4], a[5]), make_float2(a[6], a[7])));
    return s.x + s.y;
}

// Sum of one unit's elements below the reference, counting those equal to
// it apart (cnt, first).
template <int DT>
__device__ __forceinline__ float careful_unit(Online& s, const uint4 u, int x0, int V, float c)
{
    constexpr int EPU = Elem<DT>::kPerUnit;
    float v[EPU];
    unpack_masked<DT>(u, x0, V, v);
    float z = 0.f;
#pragma unroll
    for (int e = 0; e < EPU; ++e) {
        if (v[e] == s.m) {
            ++s.cnt;
            s.first = min(s.first, x0 + e);
        } else {
            z += ex2(fmaf(v[e], c, s.neg));
        }
    }
    return z;
}

template <int DT>
__device__ __forceinline__ float unit_sum(const uint4& u, int x0, int V, float c, float neg)
{
    constexpr int EPU = Elem<DT>::kPerUnit;
    float v[EPU];
    unpack_masked<DT>(u, x0, V, v);
    const float2 c2 = make_float2(c, c), n2 = make_float2(neg, neg);
#pragma unroll
    for (int e = 0; e < EPU; e += 2) {
        const float2 x = ffma2(make_float2(v[e], v[e + 1]), c2, n2);
        v[e] = ex2(x.x);
        v[e + 1] = ex2(x.y);
    }
    return tree_sum2(v);
}

// The same over a whole unit (every element below V: any chunk but the
// last), without the masking test.
template <int DT>
__device__ __forceinline__ float unit_sum_full(const uint4& u, float c, float neg)
{
    constexpr int EPU = Elem<DT>::kPerUnit;
    float v[EPU];
    Elem<DT>::unpack(u, v);
    const float2 c2 = make_float2(c, c), n2 = make_float2(neg, neg);
#pragma unroll
    for (int e = 0; e < EPU; e += 2) {
        const float2 x = ffma2(make_float2(v[e], v[e + 1]), c2, n2);
        v[e] = ex2(x.x);
        v[e + 1] = ex2(x.y);
    }
    return tree_sum2(v);
}

// Unit index of (chunk, warp, sub-unit, lane): a warp's units of a chunk
// are contiguous, consecutive lanes on consecutive units.
__device__ __forceinline__ int unit_local(int cw, int i, int lane) { return cw * kWU + i * 32 + lane; }

// Maximum of a thread's units of one row in one chunk.  Only the last
// chunk of a row holds units past V (masked) or no unit at all.
template <int DT>
__device__ __forceinline__ float chunk_max(const uint4 (&u)[kUPT], int ug0, int n_units, int V, bool tail)
{
    static_assert(kUPT == 2, "pair_max covers two units");
    if (!tail) return Elem<DT>::pair_max(u[0], u[1]);
    float m = -INFINITY;
#pragma unroll
    for (int i = 0; i < kUPT; ++i) {
        const int ug = ug0 + i * 32;
        if (ug < n_units) m = max_nan(m, unit_max_masked<DT>(u[i], ug * Elem<DT>::kPerUnit, V));
    }
    return m;
}

// A lane whose chunk reaches the reference sets the chunk aside: its units
// go to the lane's stash (slot nd) and the chunk index to d0 or d1.  With no
// room left it flags the chunk for the exact path.
__device__ __forceinline__ bool set_aside(Online& s, bool sp, int ch, uint4 (*stash)[kUPT], const uint4 (&u)[kUPT])
{
    if (!sp) return false;
    if (s.nd < kStash) {
#pragma unroll
        for (int i = 0; i < kUPT; ++i) stash[s.nd][i] = u[i];
        if (s.nd == 0)
            s.d0 = ch;
        else
            s.d1 = ch;
        ++s.nd;
        return false;
    }
    return true;
}

// After the pass: the set-aside chunks of this lane, from its stash,
// summed against the final maximum.
template <int DT>
__device__ __forceinline__ void online_finish(Online& s, const uint4 (*stash)[kUPT], int cw, int lane, int n_units,
                                              int V, float c)
{
    constexpr int EPU = Elem<DT>::kPerUnit;
    if (!(s.m > -INFINITY)) return;
    const int n = s.nd;
    s.nd = 0;
#pragma unroll
    for (int k = 0; k < kStash; ++k) {
        if (k < n) {
            const int ug0 = (k == 0 ? s.d0 : s.d1) * kChunk + unit_local(cw, 0, lane);
#pragma unroll
            for (int i = 0; i < kUPT; ++i) {
                const int ug = ug0 + i * 32;
                if (ug < n_units) s.z += careful_unit<DT>(s, stash[k][i], ug * EPU, V, c);
            }
        }
    }
}

// Pass 1 over one node's target and draft rows.
// Both rows' exponentials sit in one branch-free block.  A chunk can reach
// the reference only where one of its terms e = 2^(x c - m c) is at least
// 1, so a lane whose chunk sum is below 1/2 holds no maximum: the chunk
// maxima, the warp reduction and the reference moves run only when some
// lane's sum is not (in practice a few chunks per row and warp).
template <int DT>
__device__ __forceinline__ void pass1(StreamSmem* sm, Online& sT, Online& sD, uint32_t& g, bool& timed_out,
                                      int nc, int n_units, int V, float c, int cw, int lane, uint64_t lim)
{
    uint4(*const stashT)[kUPT] = sm->stash[0][cw * 32 + lane];
    uint4(*const stashD)[kUPT] = sm->stash[1][cw * 32 + lane];
    constexpr int EPU = Elem<DT>::kPerUnit;
#pragma unroll 1
    for (int ch = 0; ch < nc; ++ch, ++g) {
        const int s = g % kStages;
        if (!mbar_wait_bounded(&sm->full[s], (g / kStages) & 1, lim, timed_out)) timed_out = true;
        const bool tail = ch == nc - 1;
        const int ug0 = ch * kChunk + unit_local(cw, 0, lane);
        // (only the last chunk has units past V, or none: the others take no
        // test per unit; this loop and the sums below are the hot path)
        uint4 t[kUPT], d[kUPT];
        if (!tail) {
#pragma unroll
            for (int i = 0; i < kUPT; ++i) {
                const int ul = unit_local(cw, i, lane);
                t[i] = sm->ring[s][0][ul];
                d[i] = sm->ring[s][1][ul];
            }
        } else {
#pragma unroll
            for (int i = 0; i < kUPT; ++i) {
                const int ul = unit_local(cw, i, lane);
                t[i] = d[i] = make_uint4(0u, 0u, 0u, 0u);
                if (ug0 + i * 32 < n_units) {
                    t[i] = sm->ring[s][0][ul];
                    d[i] = sm->ring[s][1][ul];
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm->empty[s]);  // the units are in registers now
        // nothing finite seen yet: set the reference first (the first chunk,
        // in practice)
        if (!(sT.m > -INFINITY) || !(sD.m > -INFINITY)) {
            if (!(sT.m > -INFINITY)) online_rebase(sT, warp_max_redux(chunk_max<DT>(t, ug0, n_units, V, tail)), c);
            if (!(sD.m > -INFINITY)) online_rebase(sD, warp_max_redux(chunk_max<DT>(d, ug0, n_units, V, tail)), c);
        }
        const bool liveT = sT.m > -INFINITY, liveD = sD.m > -INFINITY;
        // (a row with nothing finite yet sums against 0: never added)
        const float negT = liveT ? sT.neg : 0.f, negD = liveD ? sD.neg : 0.f;
        float zt = 0.f, zd = 0.f;
        if (!tail) {
#pragma unroll
            for (int i = 0; i < kUPT; ++i) {
                zt += unit_sum_full<DT>(t[i], c, negT);
                zd += unit_sum_full<DT>(d[i], c, negD);
            }
        } else {
#pragma unroll
            for (int i = 0; i < kUPT; ++i) {
                const int ug = ug0 + i * 32;
                if (ug < n_units) {
                    zt += unit_sum<DT>(t[i], ug * EPU, V, c, negT);
                    zd += unit_sum<DT>(d[i], ug * EPU, V, c, negD);
                }
            }
        }
        // a sum of 1/2 or more (or NaN) may hold the maximum
        const bool hotT = liveT && !(zt < 0.5f), hotD = liveD && !(zd < 0.5f);
        if (__any_sync(0xffffffffu, hotT || hotD)) {
            const float cmT = hotT ? chunk_max<DT>(t, ug0, n_units, V, tail) : -INFINITY;
            const float cmD = hotD ? chunk_max<DT>(d, ug0, n_units, V, tail) : -INFINITY;
            const float wmT = warp_max_redux(cmT);
            const float wmD = warp_max_redux(cmD);
            // a chunk that reaches the reference is not added here
            const bool spT = hotT && cmT >= sT.m, spD = hotD && cmD >= sD.m;
            if (liveT) sT.z += spT ? 0.f : zt;
            if (liveD) sD.z += spD ? 0.f : zd;
            const bool ovT = set_aside(sT, spT, ch, stashT, t), ovD = set_aside(sD, spD, ch, stashD, d);
            // the chunk's sums are in the old reference: move it now
            online_rebase(sT, wmT, c);
            online_rebase(sD, wmD, c);
            if (__any_sync(0xffffffffu, ovT || ovD)) {
                // lanes with no room left: their units, exactly, against
                // the moved reference (which is at least their maximum)
#pragma unroll
                for (int i = 0; i < kUPT; ++i) {
                    const int ug = ug0 + i * 32;
                    if (!tail || ug < n_units) {
                        if (ovT) sT.z += careful_unit<DT>(sT, t[i], ug * EPU, V, c);
                        if (ovD) sD.z += careful_unit<DT>(sD, d[i], ug * EPU, V, c);
                    }
                }
            }
        } else {
            if (liveT) sT.z += zt;
            if (liveD) sD.z += zd;
        }
    }
}

// One residual sweep over a node's rows (from the ring): returns this
// thread's share of S_j = sum over x != x* of max(aT e_T(x) - aD e_D(x), 0).
// Each token's term is taken divided by aT = p / Z_T:
// max(aT e_T - aD e_D, 0) / aT = max(e_T - r e_D, 0), r = aD / aT, one FMA
// per token (two tokens per packed FMA); the sums are scaled by aT once.
// (With p = 0, aT = 0 and r is the largest float: every term is finite and
// scaled to 0.)  `back`: the chunks come last to first (the copy warp's
// order).
template <int DT>
__device__ __forceinline__ float sweep(StreamSmem* sm, uint32_t& g, bool& timed_out, int nc, int n_units, int V,
                                       float c, float gnegT, float gnegD, float aT, float r, int xs, int cw,
                                       int lane, bool back, uint64_t lim)
{
    constexpr int EPU = Elem<DT>::kPerUnit;
    const int xs_ch = xs >= 0 ? xs / EPU / kChunk : -1;  // x* is carried apart: its chunk skips it
    float tot = 0.f;
#pragma unroll 1
    for (int it = 0; it < nc; ++it, ++g) {
        const int ch = back ? nc - 1 - it : it;
        const int s = g % kStages;
        if (!mbar_wait_bounded(&sm->full[s], (g / kStages) & 1, lim, timed_out)) timed_out = true;
        const bool tail = ch == nc - 1;
        float w = 0.f;
        if (!tail && ch != xs_ch) {
            // the hot path: whole units, no x* (no test per unit or element)
            const float2 c2 = make_float2(c, c), nT = make_float2(gnegT, gnegT), nD = make_float2(gnegD, gnegD);
            const float2 mr = make_float2(-r, -r);
#pragma unroll
            for (int i = 0; i < kUPT; ++i) {
                const int ul = unit_local(cw, i, lane);
                float t[EPU], d[EPU];
                Elem<DT>::unpack(sm->ring[s][0][ul], t);
                Elem<DT>::unpack(sm->ring[s][1][ul], d);
#pragma unroll
                for (int e = 0; e < EPU; e += 2) {
                    const float2 xt = ffma2(make_float2(t[e], t[e + 1]), c2, nT);
                    const float2 xd = ffma2(make_float2(d[e], d[e + 1]), c2, nD);
                    const float2 v = ffma2(mr, make_float2(ex2(xd.x), ex2(xd.y)), make_float2(ex2(xt.x), ex2(xt.y)));
                    d[e] = fmaxf(v.x, 0.f);
                    d[e + 1] = fmaxf(v.y, 0.f);
                }
                w += tree_sum2(d);
            }
        } else
#pragma unroll
        for (int i = 0; i < kUPT; ++i) {
            const int ul = unit_local(cw, i, lane), ug = ch * kChunk + ul;
            if (!tail || ug < n_units) {
                float t[EPU], d[EPU];
                if (tail) {
                    unpack_masked<DT>(sm->ring[s][0][ul], ug * EPU, V, t);
                    unpack_masked<DT>(sm->ring[s][1][ul], ug * EPU, V, d);
                } else {
                    Elem<DT>::unpack(sm->ring[s][0][ul], t);
                    Elem<DT>::unpack(sm->ring[s][1][ul], d);
                }
                const float2 c2 = make_float2(c, c), nT = make_float2(gnegT, gnegT), nD = make_float2(gnegD, gnegD);
                const float2 mr = make_float2(-r, -r);
#pragma unroll
                for (int e = 0; e < EPU; e += 2) {
                    const float2 xt = ffma2(make_float2(t[e], t[e + 1]), c2, nT);
                    const float2 xd = ffma2(make_float2(d[e], d[e + 1]), c2, nD);
                    const float2 v = ffma2(mr, make_float2(ex2(xd.x), ex2(xd.y)), make_float2(ex2(xt.x), ex2(xt.y)));
                    d[e] = fmaxf(v.x, 0.f);
                    d[e + 1] = fmaxf(v.y, 0.f);
                }
                if (ch == xs_ch) {
#pragma unroll
                    for (int e = 0; e < EPU; ++e)
                        if (ug * EPU + e == xs) d[e] = 0.f;
                }
                w += tree_sum2(d);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm->empty[s]);
        tot += w;
    }
    return aT * tot;
}

// One K-SEQ search pass over a node's rows (from the ring): this thread's
// shares of Z_D beta(rho_k) = sum_x min(e_D(x), e_T(x) Z_D / (Z_T rho_k)),
// f[k] = Z_D / (Z_T rho_k), for NP points at once.  `back`: the chunks come
// last to first (the copy warp's order).
template <int DT, int NP>
__device__ __forceinline__ void kseq_sweep(StreamSmem* sm, uint32_t& g, bool& timed_out, int nc, int n_units, int V,
                                           float c, float gnegT, float gnegD, const float (&f)[5], float (&acc)[5],
                                           int cw, int lane, bool back, uint64_t lim)
{
    constexpr int EPU = Elem<DT>::kPerUnit;
#pragma unroll
    for (int k = 0; k < 5; ++k) acc[k] = 0.f;
#pragma unroll 1
    for (int it = 0; it < nc; ++it, ++g) {
        const int ch = back ? nc - 1 - it : it;
        const int s = g % kStages;
        if (!mbar_wait_bounded(&sm->full[s], (g / kStages) & 1, lim, timed_out)) timed_out = true;
        const bool tail = ch == nc - 1;
#pragma unroll
        for (int i = 0; i < kUPT; ++i) {
            const int ul = unit_local(cw, i, lane), ug = ch * kChunk + ul;
            if (!tail || ug < n_units) {
                float t[EPU], d[EPU];
                if (tail) {
                    unpack_masked<DT>(sm->ring[s][0][ul], ug * EPU, V, t);
                    unpack_masked<DT>(sm->ring[s][1][ul], ug * EPU, V, d);
                } else {  // (whole units: no masking test)
                    Elem<DT>::unpack(sm->ring[s][0][ul], t);
                    Elem<DT>::unpack(sm->ring[s][1][ul], d);
                }
                float2 u[NP];
#pragma unroll
                for (int k = 0; k < NP; ++k) u[k] = make_float2(0.f, 0.f);
                const float2 c2 = make_float2(c, c), nT = make_float2(gnegT, gnegT), nD = make_float2(gnegD, gnegD);
#pragma unroll
                for (int e = 0; e < EPU; e += 2) {
                    const float2 xt = ffma2(make_float2(t[e], t[e + 1]), c2, nT);
                    const float2 xd = ffma2(make_float2(d[e], d[e + 1]), c2, nD);
                    const float2 eT = make_float2(ex2(xt.x), ex2(xt.y)), eD = make_float2(ex2(xd.x), ex2(xd.y));
#pragma unroll
                    for (int k = 0; k < NP; ++k) {
                        const float2 m = fmul2(eT, make_float2(f[k], f[k]));
                        u[k] = fadd2(u[k], make_float2(fminf(eD.x, m.x), fminf(eD.y, m.y)));
                    }
                }
#pragma unroll
                for (int k = 0; k < NP; ++k) acc[k] += u[k].x + u[k].y;
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm->empty[s]);
    }
}

// K-SEQ's gamma = (1 - (1 - beta)^n) / beta (n when beta = 0) over n
// candidates, a rho qualifying when gamma(beta(rho)) <= rho.  The power is
// taken as -expm1(n log1p(-beta)): the same value without the
// cancellation of the plain form, which at small beta (nearly disjoint P
// and Q) costs fp32 several digits of gamma and turns the search.
__device__ __forceinline__ float kseq_gamma(float beta, int n)
{
    beta = fminf(fmaxf(beta, 0.f), 1.f);
    return beta > 0.f ? -expm1f((float)n * log1pf(-beta)) / beta : (float)n;
}

// Combine the consumers' online statistics of both rows (all consumer
// threads call it; results in shared memory from consumer thread 0): row
// maximum M, reference -(M c), Z_rest (the sum below M), the count n of
// maxima, Z = n e(M) + Z_rest, and the index of a unique maximum.
__device__ __forceinline__ void combine_rows(StreamSmem* sm, const Online& sT, const Online& sD, float c, int ct)
{
    const int lane = ct & 31, w = ct >> 5;
    float MT = warp_max_redux(sT.m), MD = warp_max_redux(sD.m);
    if (lane == 0) {
        sm->redf[0][w] = MT;
        sm->redf[1][w] = MD;
    }
    if (ct == 0) sm->firstT = sm->firstD = 0x7fffffff;  // read by thread 0 after the next barrier
    cbar_sync();
    MT = MD = -INFINITY;
    for (int i = 0; i < kSW; ++i) {
        MT = max_nan(MT, sm->redf[0][i]);
        MD = max_nan(MD, sm->redf[1][i]);
    }
    // rounded products (no FMA into the rescale differences below): each
    // partial sum was taken against -fl(m c), and moves to -fl(M c)
    const float gnegT = -__fmul_rn(MT, c), gnegD = -__fmul_rn(MD, c);
    // a thread whose reference is the row's adds its sums as they are;
    // another rescales them (its maxima are then ordinary elements)
    float cT, cD;
    int nT = 0, nD = 0;
    if (sT.m == MT) {
        cT = sT.z;
        nT = sT.cnt;
        if (nT > 0) atomicMin(&sm->firstT, sT.first);
    } else {
        const float scl = (sT.cnt > 0 || sT.z > 0.f) ? ex2(__fsub_rn(gnegT, sT.neg)) : 0.f;
        cT = sT.cnt > 0 ? scl * (sT.z + (float)sT.cnt * ex2(fmaf(sT.m, c, sT.neg))) : scl * sT.z;
    }
    if (sD.m == MD) {
        cD = sD.z;
        nD = sD.cnt;
        if (nD > 0) atomicMin(&sm->firstD, sD.first);
    } else {
        const float scl = (sD.cnt > 0 || sD.z > 0.f) ? ex2(__fsub_rn(gnegD, sD.neg)) : 0.f;
        cD = sD.cnt > 0 ? scl * (sD.z + (float)sD.cnt * ex2(fmaf(sD.m, c, sD.neg))) : scl * sD.z;
    }
    cT = warp_sum(cT);
    cD = warp_sum(cD);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        nT += __shfl_xor_sync(0xffffffffu, nT, o);
        nD += __shfl_xor_sync(0xffffffffu, nD, o);
    }
    if (lane == 0) {
        sm->redf[2][w] = cT;
        sm->redf[3][w] = cD;
        sm->redi[0][w] = nT;
        sm->redi[1][w] = nD;
    }
    cbar_sync();
    if (ct == 0) {
        float zT = 0.f, zD = 0.f;
        int n1 = 0, n2 = 0;
        for (int i = 0; i < kSW; ++i) {
            zT += sm->redf[2][i];
            zD += sm->redf[3][i];
            n1 += sm->redi[0][i];
            n2 += sm->redi[1][i];
        }
        const float emT = ex2(fmaf(MT, c, gnegT));
        sm->MT = MT;
        sm->gnegT = gnegT;
        sm->zrestT = zT;
        sm->zT = (float)n1 * emT + zT;
        sm->emaxT = emT;
        sm->uT = n1 == 1 ? sm->firstT : -1;
        const float emD = ex2(fmaf(MD, c, gnegD));
        sm->MD = MD;
        sm->gnegD = gnegD;
        sm->zrestD = zD;
        sm->zD = (float)n2 * emD + zD;
        sm->emaxD = emD;
        sm->uD = n2 == 1 ? sm->firstD : -1;
    }
}

struct ProbS {
    float P, Pbar;
};

// 2^(logit c + gneg) for one gathered token.  For a tail token the
// argument is 20 to 30 in size, where rounding it to fp32 alone moves the
// result by up to 7e-7 relative; in a row sum such errors average out,
// but a draw's own P(y) and Q(y) meet in R = P - C Q, whose cancellation
// multiplies it.  The product of two floats is exact in double, so the
// argument is formed there, split into a float and its remainder, and
// raised with the accurate exp2f and a first-order term for the remainder.
__device__ __forceinline__ float exp2_gathered(float logit, float c, float gneg)
{
    const double a = fma((double)logit, (double)c, (double)gneg);
    const float hi = (float)a;
    const float lo = (float)(a - (double)hi);
    return exp2f(hi) * fmaf(lo, 0.693147180559945309f, 1.f);
}

__device__ __forceinline__ ProbS prob_s(const StreamSmem* sm, bool is_t, int x, float logit, float c)
{
    ProbS o;
    if (x == (is_t ? sm->uT : sm->uD)) {
        const float z = is_t ? sm->zT : sm->zD;
        o.P = (is_t ? sm->emaxT : sm->emaxD) / z;
        o.Pbar = (is_t ? sm->zrestT : sm->zrestD) / z;
    } else {
        o.P = exp2_gathered(logit, c, is_t ? sm->gnegT : sm->gnegD) / (is_t ? sm->zT : sm->zD);
        o.Pbar = 1.f - o.P;
    }
    return o;
}

// KSEQ: the K-SEQ rule's search passes instead of the residual sweeps (a
// separate instantiation, so that the other rules' code is not affected)
template <int DT, bool KSEQ>
__global__ void __launch_bounds__(kSThreads, kCtasPerSm) stream_kernel(Problem pb)
{
    using E = Elem<DT>;
    constexpr int EPU = E::kPerUnit;
    extern __shared__ __align__(128) unsigned char smem_raw[];
    StreamSmem* sm = reinterpret_cast<StreamSmem*>(smem_raw);
    const int tid = threadIdx.x;
    // the finish kernel may be scheduled now: its CTAs take SMs only as this
    // kernel's CTAs leave them, and each waits for its own request's nodes
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int K = pb.K, L = pb.L, V = pb.V;
    const int BK = pb.B * K;
    const int n_units = (V + EPU - 1) / EPU;
    const int nc = (n_units + kChunk - 1) / kChunk;
    const float c = pb.c;
    const uint64_t lim = pb.wait_ns;
    int* const counter = pb.ws.ncount + 2 * (L + 1);
    // token rule: a node's last draw needs no sweep here (its S_n enters only
    // the end node's residual, summed by the decision kernel's draw pass)
    const bool lazy_last = !KSEQ && pb.mode == SDV_MODE_TOKEN;
    // block rules, when the caller does not ask for every node's h (accept_prob):
    // a node's last sweep gives S_n, which enters only h_v = S_n / D_n, read
    // when the decision tests v (accepted iff u_v <= h_v), and the residual
    // of the end node.  The root is never tested, and its residual is summed
    // by the decision kernel's draw pass; another node is skipped when its
    // test must fail: S_n <= S_{n-1}, so h_v <= S_{n-1} / D_{n-1} (p for one
    // draw), and u_v above that bound rejects v whatever S_n is.
    const bool lazy_block =
        !KSEQ && (pb.mode == SDV_MODE_BLOCK || pb.mode == SDV_MODE_MULTIDRAFT) && pb.accept_prob == nullptr;

    if (tid == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&sm->full[i], 1);
            mbar_init(&sm->empty[i], kSW);
        }
        for (int i = 0; i < kQ; ++i) {
            mbar_init(&sm->qfull[i], 1);
            mbar_init(&sm->qempty[i], 2);  // read by the copy warp and by the consumers
        }
        mbar_init(&sm->lastdec, 1);
        mbar_fence_init();
        sm->abort = 0;
    }
    __syncthreads();

    // ---------------------------------------------------------------- metadata warp
    // Takes nodes from the prep kernel's depth-major list (every parent
    // before its children) and fills the descriptor queue up to kQ nodes
    // ahead: draws, their tokens and logits, the sample uniform.
    if (tid < 32) {
        const int lane = tid;
        // lane j holds the node counts of depth j: several-draw nodes (from
        // the front of the depth's list) and one-draw nodes (from its back)
        const int cntf = lane <= L ? pb.ws.ncount[lane] : 0;
        const int cnt = lane <= L ? cntf + pb.ws.ncount[L + 1 + lane] : 0;
        int n_items = cnt;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) n_items += __shfl_xor_sync(0xffffffffu, n_items, o);
        for (uint32_t it = 0;; ++it) {
            const int q = it % kQ;
            int w = 0;
            if (lane == 0) w = atomicAdd(counter, 1);
            w = __shfl_sync(0xffffffffu, w, 0);
            int slot = -1;
            if (w < n_items) {
                // depth j: the first whose inclusive prefix of counts passes w
                int incl = cnt;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const int n = __shfl_up_sync(0xffffffffu, incl, o);
                    if (lane >= o) incl += n;
                }
                const int j = __ffs(__ballot_sync(0xffffffffu, incl > w)) - 1;
                const int before = __shfl_sync(0xffffffffu, incl - cnt, j);
                const int nf = __shfl_sync(0xffffffffu, cntf, j);
                const int i = w - before;
                slot = pb.ws.nodes[(size_t)j * BK + (i < nf ? i : BK - 1 - (i - nf))];
            }
            bool ok = true;
            if (lane == 0 && it >= kQ) ok = mbar_wait_bounded(&sm->qempty[q], (it / kQ - 1) & 1, lim);
            if (!__shfl_sync(0xffffffffu, (int)ok, 0)) {
                sm->abort = 1;
                break;
            }
            NodeDesc& d = sm->qd[q];
            if (slot >= 0) {
                const int k = slot % K, j = (slot / K) % (L + 1), b = slot / (K * (L + 1));
                const size_t sbase = (size_t)slot - k;
                const bool draw = lane < K && lane >= k && pb.ws.owner[sbase + lane] == k;
                const unsigned m = __ballot_sync(0xffffffffu, draw);
                if (draw) {
                    const int pos = __popc(m & ((1u << lane) - 1));
                    const int y = pb.tokens[((size_t)b * K + lane) * L + j];
                    const char* gT = static_cast<const char*>(pb.target) +
                                     (((size_t)b * K + k) * (L + 1) + j) * (size_t)pb.stride * E::kBytes;
                    const char* gD = static_cast<const char*>(pb.draft) +
                                     (((size_t)b * K + k) * L + j) * (size_t)pb.stride * E::kBytes;
                    d.dk[pos] = lane;
                    d.y[pos] = y;
                    d.gT[pos] = E::load(gT, y);
                    d.gD[pos] = E::load(gD, y);
                }
                if (lane == 0) {
                    d.slot = slot;
                    d.b = b;
                    d.j = j;
                    d.k = k;
                    d.nd = __popc(m);
                }
            } else if (lane == 0) {
                d.slot = -1;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm->qfull[q]);
            if (slot < 0) break;
        }
        return;
    }

    // ---------------------------------------------------------------- copy warp
    // Streams each node's rows: pass 1, then one pass per draw; evict_last
    // until the last pass, which is evict_first (as is the one before a
    // last sweep that waits for the consumers' word).
    if (tid < 64) {
        if (tid != 32) return;
        const uint64_t pol_last = policy_evict_last();
        const uint64_t pol_first = policy_evict_first();
        uint32_t g = 0;
        uint32_t dec_par = 0;  // parity of the next last-sweep decision
        for (uint32_t it = 0;; ++it) {
            const int q = it % kQ;
            if (!mbar_wait_bounded(&sm->qfull[q], (it / kQ) & 1, lim)) {
                sm->abort = 1;
                break;
            }
            const NodeDesc& d = sm->qd[q];
            const int slot = d.slot, b = d.b, j = d.j, k = d.k, nd = d.nd;
            mbar_arrive(&sm->qempty[q]);
            if (slot < 0) break;
            const char* gT = static_cast<const char*>(pb.target) +
                             (((size_t)b * K + k) * (L + 1) + j) * (size_t)pb.stride * E::kBytes;
            const char* gD = static_cast<const char*>(pb.draft) +
                             (((size_t)b * K + k) * L + j) * (size_t)pb.stride * E::kBytes;
            // the token rule's last sweep of a node only feeds the residual
            // the walk may end at: the decision kernel takes it then; so does
            // a root's under the block rules; another node's last sweep under
            // the block rules is issued only if the consumers ask for it
            const bool root_skip = lazy_block && j == 0;
            const bool ask_last = lazy_block && j > 0;
            const int passes = 1 + (KSEQ ? (nd > 1 ? kKseqRounds : 1) : nd - (lazy_last || root_skip ? 1 : 0));
            bool ok = true;
            for (int ps = 0; ps < passes && ok; ++ps) {
                if (ask_last && ps == passes - 1) {
                    ok = mbar_wait_bounded(&sm->lastdec, dec_par, lim);
                    dec_par ^= 1u;
                    if (!ok || !*static_cast<volatile int*>(&sm->last_go)) break;
                }
                // keep the rows in L2 until the node's last pass over them;
                // where that last pass is a sweep the consumers may not ask
                // for (most are not asked for), the pass before it is
                // already evict_first: L2 space is kept for the rows that
                // are surely read again
                const bool final_pass = ps == passes - 1 || (ask_last && ps == passes - 2);
                const uint64_t pol = final_pass ? pol_first : pol_last;
                // passes alternate direction (pass 1 forward, the first
                // sweep backward, ...): each pass starts on the chunks the
                // one before just brought into L2
                const bool back = (ps & 1) != 0;
                for (int i = 0; i < nc; ++i, ++g) {
                    const int ch = back ? nc - 1 - i : i;
                    const int s = g % kStages;
                    const uint32_t use = g / kStages;
                    if (use > 0 && !mbar_wait_bounded(&sm->empty[s], (use - 1) & 1, lim)) {
                        ok = false;
                        break;
                    }
                    const int u0 = ch * kChunk;
                    const uint32_t bytes = (uint32_t)min(kChunk, n_units - u0) * 16u;
                    mbar_expect_tx(&sm->full[s], 2 * bytes);
                    bulk_g2s_hint(&sm->ring[s][0][0], gT + (size_t)u0 * 16, bytes, &sm->full[s], pol);
                    bulk_g2s_hint(&sm->ring[s][1][0], gD + (size_t)u0 * 16, bytes, &sm->full[s], pol);
                }
            }
            if (!ok) {
                sm->abort = 1;
                break;
            }
        }
        // before the CTA may exit: every copy this warp issued has landed
        // (at once in a normal run, where the consumers waited for each;
        // after an abort they may not have)
        for (int s = 0; s < kStages; ++s) {
            if (g > (uint32_t)s) {
                const uint32_t last_use = (g - 1 - (uint32_t)s) / kStages;
                mbar_wait_bounded(&sm->full[s], last_use & 1, lim);
            }
        }
        return;
    }

    // ---------------------------------------------------------------- consumers
    const int ct = tid - 64, lane = ct & 31, cw = ct >> 5;
    uint32_t g = 0;
    bool timed_out = false;
    for (uint32_t it = 0;; ++it) {
        const int q = it % kQ;
        // copy the descriptor, then hand the queue slot back
        const bool got = mbar_wait_bounded(&sm->qfull[q], (it / kQ) & 1, lim);
        if (!got) atomicExch(&sm->abort, 1);
        cbar_sync();  // the previous node's readers of sm->cur are done
        if (ct < (int)(sizeof(NodeDesc) / 4))
            reinterpret_cast<int*>(&sm->cur)[ct] = reinterpret_cast<const int*>(&sm->qd[q])[ct];
        cbar_sync();
        if (ct == 0) mbar_arrive(&sm->qempty[q]);
        const int slot = *static_cast<volatile int*>(&sm->abort) ? -1 : sm->cur.slot;
        if (slot < 0) break;

        const int k = sm->cur.k, j = sm->cur.j, b = sm->cur.b;
        const size_t sbase = (size_t)slot - k;
        const int nd = sm->cur.nd;

        // ---- pass 1: online statistics ----
        Online sT, sD;
        pass1<DT>(sm, sT, sD, g, timed_out, nc, n_units, V, c, cw, lane, lim);
        online_finish<DT>(sT, sm->stash[0][ct], cw, lane, n_units, V, c);
        online_finish<DT>(sD, sm->stash[1][ct], cw, lane, n_units, V, c);
        combine_rows(sm, sT, sD, c, ct);

        // ---- scalar state ----
        if (ct == 0) {
            const bool bad = !(isfinite(sm->MT) && isfinite(sm->zT) && sm->zT > 0.f) ||
                             !(isfinite(sm->MD) && isfinite(sm->zD) && sm->zD > 0.f);
            sm->bad = bad;
            if (bad) {
                atomicOr(&pb.ws.req[b], SDV_REQ_NONFINITE);
                if (pb.device_status) atomicOr(pb.device_status, SDV_REQ_NONFINITE);
            }
            // the node weight {1 - p, p}, written by the parent (.x below 0
            // until then)
            float2 wt = make_float2(0.f, 1.f);
            if (!KSEQ && j > 0 && pb.mode != SDV_MODE_TOKEN) {
                const float2* f = pb.ws.wt + slot;
                wt = ld_weight(f);
                if (!(wt.x >= 0.f)) {
                    const uint64_t t0 = globaltimer();
                    while (!((wt = ld_weight(f)).x >= 0.f)) {
                        if (globaltimer() - t0 > lim) {
                            sm->abort = 1;
                            wt = make_float2(0.f, 1.f);
                            break;
                        }
                    }
                }
            }
            sm->pbar = wt.x;
            sm->pw = wt.y;
            const int xs = (sm->uT >= 0 && sm->uT == sm->uD) ? sm->uT : -1;
            sm->xs = xs;
            sm->Pbs = xs >= 0 ? sm->zrestT / sm->zT : 0.f;
            sm->Qbs = xs >= 0 ? sm->zrestD / sm->zD : 0.f;
            sm->Rs = sm->Ts = 0.f;
            sm->S = wt.y;
            sm->D = 1.f;
            sm->cbar = 0.f;
            if constexpr (KSEQ) {
                // the first pass tests rho = 1, the first round's quarter
                // points of [1, n], and n (a node with one draw: rho = 1)
                const float n = (float)nd;
                sm->klo = 1.f;
                sm->khi = n;
                sm->kdone = nd == 1;
                sm->knp = nd == 1 ? 1 : 5;
                for (int t = 0; t < 5; ++t) {
                    const float rho = t == 0 ? 1.f : (t == 4 ? n : 1.f + (n - 1.f) * (float)t / 4.f);
                    sm->krho[t] = rho;
                    sm->kf[t] = sm->zD / (sm->zT * rho);
                }
            }
        }
        cbar_sync();
        const float pbar = sm->pbar, p = sm->pw;
        const float gnegT = sm->gnegT, gnegD = sm->gnegD;
        const int xs = sm->xs;

        // ---- pass 2: the residual recursion, one sweep per draw ----
        // R_0 = p P, R_j = max(R_{j-1} - D_{j-1} Q, 0), S_j = sum R_j,
        // D_j = (1 - p) + S_j.  Scalars are kept as complements (pbar =
        // 1 - p, cbar = C - 1, Pbs = 1 - P(x*), Qbs = 1 - Q(x*)) so that
        // nothing cancels when p, P or Q is close to 1; the weight p is
        // kept as well, and the terms proportional to it (p P) take it, so
        // that a small weight keeps its digits down a chain of nodes whose
        // ratios P / Q can raise it again.  The shared
        // dominant token x* (the unique maximum of both rows) is left out
        // of the sweeps and carried in closed form:
        //   R_1(x*) = Qbs - Pbs - pbar + pbar Pbs,
        //   R_j(x*) = R_{j-1}(x*) Qbs - (pbar + T_{j-1}) (1 - Qbs),
        // with T_{j-1} the sweep's sum over the other tokens.
        if constexpr (!KSEQ) {
            for (int di = 0; di < nd; ++di) {
                const int k2 = sm->cur.dk[di];
                const bool first_draw = di == 0;
                if (ct == 0) {
                    const int y = sm->cur.y[di];
                    const float D = sm->D;
                    const float cnew = first_draw ? 0.f : sm->cbar + D;
                    const float Pbs = sm->Pbs, Qbs = sm->Qbs;
                    const float Rj = first_draw ? ((Qbs - Pbs) - pbar) + pbar * Pbs
                                                : sm->Rs * Qbs - (pbar + sm->Ts) * (1.f - Qbs);
                    sm->Rj = Rj;
                    float R, Qy, abar_num;
                    if (y == xs) {
                        Qy = 1.f - Qbs;
                        R = first_draw ? p * (1.f - Pbs) : sm->Rs;
                        abar_num = fmaxf(-Rj, 0.f);
                    } else {
                        const ProbS Py = prob_s(sm, true, y, sm->cur.gT[di], c);
                        const ProbS Qp = prob_s(sm, false, y, sm->cur.gD[di], c);
                        Qy = Qp.P;
                        R = first_draw ? p * Py.P : fmaxf(p * Py.P - (1.f + sm->cbar) * Qp.P, 0.f);
                        abar_num = fmaxf((1.f + cnew) * Qp.P - p * Py.P, 0.f);
                    }
                    // a = min(R / (D Q(y)), 1) and its complement, each in its
                    // own right: a ratio within 6e-8 of 1 rounds to 1 in fp32,
                    // while 1 - a = (D Q(y) - R) / (D Q(y)) keeps its digits
                    float a, abar;
                    const bool dq = D > 0.f && Qy > 0.f;
                    if (!dq) {
                        a = 1.f;
                        abar = 0.f;
                    } else if (!(R > 0.f)) {
                        a = 0.f;
                        abar = 1.f;
                    } else {
                        a = fminf((R / D) / Qy, 1.f);
                        abar = fminf((abar_num / D) / Qy, 1.f);
                    }
                    sm->cbar = cnew;
                    pb.ws.a[sbase + k2] = a;
                    bool first_of_token = true;  // this draw's child is new: it owns it
                    for (int e = 0; e < di; ++e) first_of_token &= sm->cur.y[e] != y;
                    if (pb.mode != SDV_MODE_TOKEN) {
                        const size_t sc = sbase + K + k2;
                        // child first reached by this draw: its weight (never NaN:
                        // the child waits for a value of 0 or more)
                        if (first_of_token) st_weight(&pb.ws.wt[sc], fmaxf(abar, 0.f), a);
                    }
                    sm->aT = p / sm->zT;
                    sm->aD = (1.f + cnew) / sm->zD;
                    sm->rD = sm->aT > 0.f ? sm->aD / sm->aT : 3.402823466e38f;
                    if (di == nd - 1) {
                        bool skip = lazy_last;
                        if (lazy_block) {
                            if (j == 0) {
                                skip = true;  // (the copy warp knows: no word)
                            } else {
                                // the bound on h_v from S_{n-1}, D_{n-1} (held since the
                                // previous sweep; p and 1 before the first)
                                const float hhi = sm->D > 0.f ? sm->S / sm->D : 1.f;
                                const float uv = pb.accept_u[((size_t)b * K + k) * L + (j - 1)];
                                skip = uv > hhi * (1.f + 1e-6f) + 1e-7f;
                                sm->last_go = !skip;
                                mbar_arrive(&sm->lastdec);
                            }
                        }
                        sm->skip_last = skip;
                    }
                }
                cbar_sync();
                if (di == nd - 1 && sm->skip_last) {
                    // no sweep: R_n(x*) is known in closed form, and the
                    // rest of S_n is summed where it is needed
                    if (ct == 0) sm->Rs = xs >= 0 ? fmaxf(sm->Rj, 0.f) : 0.f;
                    break;
                }
                // sweep di is pass di + 1 of the node: backward for even di
                float tot = sweep<DT>(sm, g, timed_out, nc, n_units, V, c, gnegT, gnegD, sm->aT, sm->rD, xs, cw, lane,
                                      (di & 1) == 0, lim);
                tot = warp_sum(tot);
                if (lane == 0) sm->redf[2][cw] = tot;
                cbar_sync();
                if (ct == 0) {
                    float Sj = 0.f;
                    for (int i = 0; i < kSW; ++i) Sj += sm->redf[2][i];
                    if (xs >= 0) {  // the sweeps left x* out: their sum is the mass elsewhere
                        const float Rs = fmaxf(sm->Rj, 0.f);
                        sm->Ts = Sj;
                        sm->Rs = Rs;
                        Sj += Rs;
                    }
                    sm->S = fmaxf(Sj, 0.f);
                    sm->D = pbar + sm->S;
                }
            }
            if (ct == 0) {
                // the node's block acceptance and, for the correction draw
                // should the decision end here, its final residual
                // R_n = aT max(e_T - (aD / aT) e_D, 0) with R_n(x*) apart
                const float S = sm->S, D = sm->D;
                const bool skipped = nd > 0 && sm->skip_last;
                // a skipped node's test fails for sure (h below any uniform);
                // its S_n, below 0, is summed by the decision kernel should the
                // node end the decision (only a root or a token-rule node can)
                pb.ws.h[slot] = skipped ? -1.f : (D > 0.f ? S / D : 1.f);
                pb.ws.S[slot] = skipped ? -1.f : S;
                float* prm = pb.ws.prm + (size_t)slot * 6;
                prm[0] = gnegT;
                prm[1] = gnegD;
                prm[2] = sm->aT;
                prm[3] = sm->rD;
                prm[4] = sm->Rs;
                prm[5] = 0.f;
                pb.ws.xs[slot] = xs;
            }
        } else {
            // ---- K-SEQ: the search for rho, one pass per round ----
            // beta(rho) = sum_x min(Q(x), P(x) / rho); a rho qualifies when
            // gamma(beta(rho)) <= rho.  rho = 1 if it qualifies, else each
            // round keeps the quarter of [lo, hi] ending at the first of its
            // three points that qualifies (the last quarter if none does);
            // rho is the final hi.
            const int rounds = nd > 1 ? kKseqRounds : 1;
            for (int r = 0; r < rounds; ++r) {
                float f[5], acc[5];
#pragma unroll
                for (int k = 0; k < 5; ++k) f[k] = sm->kf[k];
                const int np = sm->knp;
                const bool back = (r & 1) == 0;  // pass r + 1 of the node
                if (np == 5)
                    kseq_sweep<DT, 5>(sm, g, timed_out, nc, n_units, V, c, gnegT, gnegD, f, acc, cw, lane, back, lim);
                else if (np == 3)
                    kseq_sweep<DT, 3>(sm, g, timed_out, nc, n_units, V, c, gnegT, gnegD, f, acc, cw, lane, back, lim);
                else
                    kseq_sweep<DT, 1>(sm, g, timed_out, nc, n_units, V, c, gnegT, gnegD, f, acc, cw, lane, back, lim);
#pragma unroll
                for (int k = 0; k < 5; ++k) {
                    const float v = warp_sum(acc[k]);
                    if (lane == 0) sm->redf[k][cw] = v;
                }
                cbar_sync();
                if (ct == 0) {
                    float beta[5];
                    for (int k = 0; k < np; ++k) {
                        float z = 0.f;
                        for (int i = 0; i < kSW; ++i) z += sm->redf[k][i];
                        beta[k] = z / sm->zD;
                    }
                    // the round's three points are beta[first .. first + 2]
                    int first = 0;
                    if (r == 0) {
                        if (nd == 1 || kseq_gamma(beta[0], nd) <= 1.f) {
                            sm->kdone = 1;
                            sm->khi = 1.f;
                            sm->kbhi = beta[0];
                        } else {
                            sm->kbhi = beta[4];  // beta at hi = n
                        }
                        first = 1;
                    }
                    if (!sm->kdone) {
                        const float lo = sm->klo;
                        int i = 0;
                        while (i < 3 && !(kseq_gamma(beta[first + i], nd) <= sm->krho[first + i])) ++i;
                        if (i < 3) {
                            sm->klo = i == 0 ? lo : sm->krho[first + i - 1];
                            sm->khi = sm->krho[first + i];
                            sm->kbhi = beta[first + i];
                        } else {
                            sm->klo = sm->krho[first + 2];
                        }
                        // the next round's points
                        const float l = sm->klo, h = sm->khi;
                        for (int t = 0; t < 3; ++t) {
                            const float rho = l + (h - l) * (float)(t + 1) / 4.f;
                            sm->krho[t] = rho;
                            sm->kf[t] = sm->zD / (sm->zT * rho);
                        }
                    }
                    sm->knp = 3;
                }
                cbar_sync();
            }
            if (ct == 0) {
                // acceptance of each draw, and the residual for the correction
                // draw should the decision end here:
                // P - gamma min(Q, P / rho) = (1/Z_T) max(e_T - gamma (Z_T/Z_D) e_D, (1 - gamma/rho) e_T)
                const float rho = sm->khi, beta = fminf(fmaxf(sm->kbhi, 0.f), 1.f);
                const float gam = kseq_gamma(beta, nd);
                for (int di = 0; di < nd; ++di) {
                    const int y = sm->cur.y[di];
                    const float Py = prob_s(sm, true, y, sm->cur.gT[di], c).P;
                    const float Qy = prob_s(sm, false, y, sm->cur.gD[di], c).P;
                    const float den = rho * Qy;
                    pb.ws.a[sbase + sm->cur.dk[di]] = den > 0.f ? fminf(Py / den, 1.f) : 1.f;
                }
                pb.ws.h[slot] = 0.f;
                pb.ws.S[slot] = expf((float)nd * log1pf(-beta));  // the residual's mass, (1 - beta)^n
                float* prm = pb.ws.prm + (size_t)slot * 6;
                prm[0] = gnegT;
                prm[1] = gnegD;
                prm[2] = 1.f / sm->zT;
                prm[3] = gam * sm->zT / sm->zD;
                prm[4] = 0.f;
                prm[5] = fmaxf(1.f - gam / rho, 0.f);
                pb.ws.xs[slot] = -1;
            }
        }
        // a timed-out wait anywhere stops every consumer together (the
        // decision is read after the node's last barrier, so it is uniform)
        if (timed_out) atomicExch(&sm->abort, 1);
        cbar_sync();
        if (*static_cast<volatile int*>(&sm->abort)) {
            if (ct == 0) {
                atomicOr(&pb.ws.req[b], SDV_DEV_TIMEOUT);
                if (pb.device_status) atomicOr(pb.device_status, SDV_DEV_TIMEOUT);
            }
            break;
        }
        // the node's records are complete (all written by this thread): a
        // release, then one node fewer for the request's decision to wait on
        if (ct == 0) {
            __threadfence();
            atomicSub(&pb.ws.left[b], 1);
        }
    }
}

}  // namespace

size_t stream_smem_bytes() { return sizeof(StreamSmem); }
int stream_threads() { return kSThreads; }
int stream_ctas_per_sm() { return kCtasPerSm; }

cudaError_t launch_stream(const Problem& pb, cudaStream_t st)
{
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    if (sms <= 0) sms = 1;
    const bool kseq = pb.mode == SDV_MODE_KSEQ;
    const void* fn = pb.dtype == SDV_BF16
                         ? (kseq ? reinterpret_cast<const void*>(stream_kernel<SDV_BF16, true>)
                                 : reinterpret_cast<const void*>(stream_kernel<SDV_BF16, false>))
                         : (kseq ? reinterpret_cast<const void*>(stream_kernel<SDV_F32, true>)
                                 : reinterpret_cast<const void*>(stream_kernel<SDV_F32, false>));
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sizeof(StreamSmem));
    if (e != cudaSuccess) return e;
    // inner nodes: the root and at most one per draft at depths 1..L-1
    if (pb.L == 0) return cudaSuccess;
    const long long upper = (long long)pb.B * (1 + (long long)pb.K * (pb.L - 1));
    const int grid = (int)std::max(1LL, std::min((long long)sms * kCtasPerSm, upper));
    if (pb.dtype == SDV_BF16) {
        if (kseq)
            stream_kernel<SDV_BF16, true><<<grid, kSThreads, sizeof(StreamSmem), st>>>(pb);
        else
            stream_kernel<SDV_BF16, false><<<grid, kSThreads, sizeof(StreamSmem), st>>>(pb);
    } else {
        if (kseq)
            stream_kernel<SDV_F32, true><<<grid, kSThreads, sizeof(StreamSmem), st>>>(pb);
        else
            stream_kernel<SDV_F32, false><<<grid, kSThreads, sizeof(StreamSmem), st>>>(pb);
    }
    return cudaGetLastError();
}

}  // namespace sdv
