// sdv_sample.cu -- draft-token sampling: inverse-CDF draws from the
// distribution softmax(logits / T) of vocabulary rows (the step before
// verification, in which a draft model proposes its tokens: "SpecTr-GBV:
// Multi-Draft Block Verification Accelerating Speculative Decoding",
// section 1).
//
// One CTA per row, one pass over it: the row is cut into segments of 256
// contiguous 16-byte units, one per warp and step.  Each segment's mass
// sum 2^(x c - m c) is taken against the segment's own maximum m, so it
// needs no running reference; the row maximum M rescales the segments
// afterwards.  Each draw then scans the segment masses in index order for
// the first one whose running sum exceeds u * S, re-reads that 4 KB
// segment (from L2) and finds the element the same way.  When rounding
// leaves no crossing, the last element of nonzero mass is taken, as the
// rule states.  T = 0 gives the argmax, lowest index on ties.
//
// The same machinery draws verification's correction (or bonus) token, once
// per request (finish_kernel, after the request's decision), at the end
// node the decision chose: from the node's final
// residual R_n = aT max(e_T - (aD / aT) e_D, 0) with R_n(x*) apart (kept by
// the node kernel), or from P at a leaf or where S_n = 0 ("SpecTr-GBV"
// page, section 2, step 4: the correction comes from the adjusted
// residual at the end of the accepted sub-block).
#include "sdv_device.cuh"
#include "sdv_internal.h"

namespace sdv {
namespace {

constexpr int kRU = 8;                                    // units per lane per step
constexpr int kRSeg = 32 * kRU;                           // units per segment (one warp, one step)
constexpr int kRMaxSeg = (SDV_MAX_V / 4 + kRSeg - 1) / kRSeg;  // segments of the longest row

struct RowSmem {
    float mass[kRMaxSeg];  // per segment: sum of its masses (softmax: against its maximum)
    float ref[kRMaxSeg];   // softmax: the segment's maximum; residual: unused
    int bad;
};

// A draw compares u times the row's total with running sums over the
// segments, of the same size as the total; in fp32 their rounding alone
// (half an ulp: 3e-8 near 0.5) would settle a draw whose u lies that close
// to an interval's end.  The total and the running sums over segments are
// therefore kept in double (a few dozen additions a draw); a segment's own
// mass and the running sum inside one are fp32, at most 1/32 of the total
// for a row of 65536 elements or more.
__device__ __forceinline__ double warp_sum_d(double v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Inclusive prefix sum over the warp's lanes.
__device__ __forceinline__ double warp_scan_d(double v, int lane)
{
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const double n = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += n;
    }
    return v;
}

// The distribution a draw is taken from.
struct Dist {
    const char* rowT;  // softmax: the row; residual: the target row
    const char* rowD;  // residual: the draft row
    float c;           // log2(e) / T (0: argmax)
    int residual;      // 0: softmax(row / T); 1: aT max(e_T - rD e_D, 0), x* apart
    float negT, negD, aT, rD, Rs;  // residual: references -(M c), scale, ratio, mass at x*
    float cT;                      // residual: floor, aT cT e_T (0 for SpecTr-GBV; K-SEQ's 1 - gamma/rho)
    int xs;                        // residual: x*, or -1
    float M, negM;                 // softmax, after the pass: row maximum, -(M c)
};

// Masses of one unit's elements (ug: its index in the row; tu, du: the
// unit of the row and, for a residual, of the draft row).
template <int DT>
__device__ __forceinline__ void masses_of(const Dist& d, const uint4& tu, const uint4& du, int ug, int n_units, int V,
                                          bool greedy, float (&w)[Elem<DT>::kPerUnit])
{
    constexpr int EPU = Elem<DT>::kPerUnit;
    float t[EPU];
    if (ug < n_units) {
        unpack_masked<DT>(tu, ug * EPU, V, t);
    } else {
#pragma unroll
        for (int e = 0; e < EPU; ++e) t[e] = -INFINITY;
    }
    if (!d.residual) {
#pragma unroll
        for (int e = 0; e < EPU; ++e) w[e] = greedy ? (t[e] == d.M ? 1.f : 0.f) : ex2(fmaf(t[e], d.c, d.negM));
        return;
    }
    float q[EPU];
    if (ug < n_units) {
        unpack_masked<DT>(du, ug * EPU, V, q);
    } else {
#pragma unroll
        for (int e = 0; e < EPU; ++e) q[e] = -INFINITY;
    }
    const float2 c2 = make_float2(d.c, d.c), nT = make_float2(d.negT, d.negT), nD = make_float2(d.negD, d.negD);
    const float2 mr = make_float2(-d.rD, -d.rD), ct = make_float2(d.cT, d.cT), at = make_float2(d.aT, d.aT);
#pragma unroll
    for (int e = 0; e < EPU; e += 2) {
        const float2 xt = ffma2(make_float2(t[e], t[e + 1]), c2, nT);
        const float2 xq = ffma2(make_float2(q[e], q[e + 1]), c2, nD);
        const float2 eT = make_float2(ex2(xt.x), ex2(xt.y));
        const float2 v = ffma2(mr, make_float2(ex2(xq.x), ex2(xq.y)), eT);
        const float2 fl = fmul2(ct, eT);
        const float2 r = fmul2(at, make_float2(fmaxf(v.x, fl.x), fmaxf(v.y, fl.y)));
        w[e] = ug * EPU + e == d.xs ? d.Rs : r.x;
        w[e + 1] = ug * EPU + e + 1 == d.xs ? d.Rs : r.y;
    }
}

template <int DT>
__device__ __forceinline__ uint4 unit_at(const char* row, int ug, int n_units)
{
    return ug < n_units && row ? __ldg(reinterpret_cast<const uint4*>(row) + ug) : make_uint4(0u, 0u, 0u, 0u);
}

template <int DT>
__device__ __forceinline__ void unit_masses(const Dist& d, int ug, int n_units, int V, bool greedy,
                                            float (&w)[Elem<DT>::kPerUnit])
{
    const uint4 tu = unit_at<DT>(d.rowT, ug, n_units);
    const uint4 du = d.residual ? unit_at<DT>(d.rowD, ug, n_units) : tu;
    masses_of<DT>(d, tu, du, ug, n_units, V, greedy, w);
}

// Inverse CDF inside segment seg: the first element whose running sum
// exceeds `local` (the last element of nonzero mass if rounding leaves
// none).  Warp-wide; every lane gets the result.
template <int DT>
__device__ int pick_in_segment(const Dist& d, int seg, int n_units, int V, float local, bool greedy, int lane)
{
    constexpr int EPU = Elem<DT>::kPerUnit;
    float run = 0.f;
    int lastx = -1;
#pragma unroll 1
    for (int i = 0; i < kRU; ++i) {
        const int ug = seg * kRSeg + i * 32 + lane;
        float v[EPU];
        unit_masses<DT>(d, ug, n_units, V, greedy, v);
        float lsum = 0.f;
        int lnz = -1;
#pragma unroll
        for (int e = 0; e < EPU; ++e) {
            lsum += v[e];
            if (v[e] > 0.f) lnz = ug * EPU + e;
        }
        float incl = lsum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float n = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += n;
        }
        const unsigned cross = __ballot_sync(0xffffffffu, lsum > 0.f && run + incl > local);
        const unsigned nz = __ballot_sync(0xffffffffu, lnz >= 0);
        if (cross) {
            const int l = __ffs(cross) - 1;
            int pick = -1;
            if (lane == l) {
                float acc = run + incl - lsum;
                for (int e = 0; e < EPU; ++e) {
                    if (v[e] > 0.f) {
                        acc += v[e];
                        if (acc > local) {
                            pick = ug * EPU + e;
                            break;
                        }
                    }
                }
                if (pick < 0) pick = lnz;
            }
            return __shfl_sync(0xffffffffu, pick, l);
        }
        if (nz) lastx = __shfl_sync(0xffffffffu, lnz, 31 - __clz(nz));
        run += __shfl_sync(0xffffffffu, incl, 31);
    }
    return lastx;
}

// Softmax pass over a row (all warps): per segment its maximum and its mass
// against that maximum; NaN or +Inf sets sm.bad.
template <int DT>
__device__ void softmax_pass(const char* row, int V, float c, bool greedy, RowSmem& sm, int lane, int w)
{
    using E = Elem<DT>;
    constexpr int EPU = E::kPerUnit;
    const int n_units = (V + EPU - 1) / EPU;
    const int n_seg = (n_units + kRSeg - 1) / kRSeg;
    const int nw = blockDim.x >> 5;  // warps per CTA (one segment each per step)
    const int n_steps = (n_units + nw * kRSeg - 1) / (nw * kRSeg);
    bool bad = false;
#pragma unroll 1
    for (int st = 0; st < n_steps; ++st) {
        const int seg = st * nw + w;
        const int ug0 = seg * kRSeg + lane;
        uint4 u[kRU];
#pragma unroll
        for (int i = 0; i < kRU; ++i)
            u[i] = ug0 + i * 32 < n_units ? __ldg(reinterpret_cast<const uint4*>(row) + ug0 + i * 32)
                                          : make_uint4(0u, 0u, 0u, 0u);
        float cm = -INFINITY;
#pragma unroll
        for (int i = 0; i < kRU; ++i) {
            const int ug = ug0 + i * 32;
            if (ug < n_units) {
                if ((ug + 1) * EPU <= V) {
                    cm = E::unit_max(u[i], cm);
                } else {
                    float v[EPU];
                    unpack_masked<DT>(u[i], ug * EPU, V, v);
#pragma unroll
                    for (int e = 0; e < EPU; ++e) cm = max_nan(cm, v[e]);
                }
            }
        }
        bad |= (cm != cm) || cm == INFINITY;
        const float m = warp_max_redux(cm);
        float z = 0.f;
        if (!greedy && m > -INFINITY && m < INFINITY) {
            const float negm = -(m * c);
#pragma unroll
            for (int i = 0; i < kRU; ++i) {
                const int ug = ug0 + i * 32;
                if (ug < n_units) {
                    float v[EPU];
                    unpack_masked<DT>(u[i], ug * EPU, V, v);
                    const float2 c2 = make_float2(c, c), n2 = make_float2(negm, negm);
#pragma unroll
                    for (int e = 0; e < EPU; e += 2) {
                        const float2 x = ffma2(make_float2(v[e], v[e + 1]), c2, n2);
                        v[e] = ex2(x.x);
                        v[e + 1] = ex2(x.y);
                    }
#pragma unroll
                    for (int s2 = 1; s2 < EPU; s2 *= 2)
#pragma unroll
                        for (int e = 0; e + s2 < EPU; e += 2 * s2) v[e] += v[e + s2];
                    z += v[0];
                }
            }
        }
        z = warp_sum(z);
        if (lane == 0 && seg < n_seg) {
            sm.mass[seg] = z;
            sm.ref[seg] = m;
        }
    }
    if (bad) atomicOr(&sm.bad, 1);
}

// Residual pass over a node's two rows (all warps): per segment the mass of
// aT max(e_T - rD e_D, 0), x* apart with mass Rs.
template <int DT>
__device__ void residual_pass(const Dist& d, int V, RowSmem& sm, int lane, int w)
{
    constexpr int EPU = Elem<DT>::kPerUnit;
    const int n_units = (V + EPU - 1) / EPU;
    const int n_seg = (n_units + kRSeg - 1) / kRSeg;
    const int nw = blockDim.x >> 5;  // warps per CTA (one segment each per step)
    const int n_steps = (n_units + nw * kRSeg - 1) / (nw * kRSeg);
    constexpr int kHalf = kRU / 2;  // units of both rows loaded before they are used
#pragma unroll 1
    for (int st = 0; st < n_steps; ++st) {
        const int seg = st * nw + w;
        float z = 0.f;
#pragma unroll
        for (int h = 0; h < kRU; h += kHalf) {
            uint4 tu[kHalf], du[kHalf];
#pragma unroll
            for (int i = 0; i < kHalf; ++i) {
                const int ug = seg * kRSeg + (h + i) * 32 + lane;
                tu[i] = unit_at<DT>(d.rowT, ug, n_units);
                du[i] = unit_at<DT>(d.rowD, ug, n_units);
            }
#pragma unroll
            for (int i = 0; i < kHalf; ++i) {
                float v[EPU];
                masses_of<DT>(d, tu[i], du[i], seg * kRSeg + (h + i) * 32 + lane, n_units, V, false, v);
#pragma unroll
                for (int s2 = 1; s2 < EPU; s2 *= 2)
#pragma unroll
                    for (int e = 0; e + s2 < EPU; e += 2 * s2) v[e] += v[e + s2];
                z += v[0];
            }
        }
        z = warp_sum(z);
        if (lane == 0 && seg < n_seg) {
            sm.mass[seg] = z;
            sm.ref[seg] = 0.f;
        }
    }
}

// Segment i's mass against the row's reference.  A softmax pass summed the
// segment's elements as 2^(x c + negm) with its own offset negm = -(m c)
// rounded to float, and a draw's elements are taken as 2^(x c + negM); the
// factor between the two is 2 to the difference of those float offsets.
// The difference of two floats is exact as a float plus a remainder
// (TwoSum); the factor is exp2f of the first times a first-order term for
// the second.  The operations are written with rounding intrinsics so
// that the compiler cannot fuse the product into the first sum (an FMA
// there would add the unrounded product, 2 to whose rounding error, up to
// 5e-6 relative at 1/T = 10, would then scale the segment).
__device__ __forceinline__ float seg_mass(const Dist& d, const RowSmem& sm, int i)
{
    if (d.residual) return sm.mass[i];
    const float ref = sm.ref[i];
    if (!(ref > -INFINITY)) return 0.f;
    const float a = d.negM, b = __fmul_rn(ref, d.c);  // delta = a + b, b = -negm
    const float hi = __fadd_rn(a, b);
    const float bb = __fsub_rn(hi, a);
    const float lo = __fadd_rn(__fsub_rn(a, __fsub_rn(hi, bb)), __fsub_rn(b, bb));
    return sm.mass[i] * (exp2f(hi) * fmaf(lo, 0.693147180559945309f, 1.f));
}

// The row's total mass as every draw sums it (per warp, lanes in order).
__device__ __forceinline__ double row_total(const Dist& d, const RowSmem& sm, int n_seg, int lane)
{
    double tot = 0.0;
    for (int i = lane; i < n_seg; i += 32) tot += (double)seg_mass(d, sm, i);
    return warp_sum_d(tot);
}

// One draw with uniform u (warp-wide).  Softmax distributions rescale each
// segment from its own maximum to the row's.
template <int DT>
__device__ int draw(const Dist& d, const RowSmem& sm, int V, float u, bool greedy, int lane)
{
    constexpr int EPU = Elem<DT>::kPerUnit;
    const int n_units = (V + EPU - 1) / EPU;
    const int n_seg = (n_units + kRSeg - 1) / kRSeg;
    int seg = -1;
    double base = 0.0, thr = 0.5;
    if (greedy) {  // the first segment holding the maximum; its first element equal to it
        for (int i0 = 0; i0 < n_seg && seg < 0; i0 += 32) {
            const int i = i0 + lane;
            const unsigned hit = __ballot_sync(0xffffffffu, i < n_seg && sm.ref[i] == d.M);
            if (hit) seg = i0 + __ffs(hit) - 1;
        }
    } else {
        thr = (double)u * row_total(d, sm, n_seg, lane);
        double run = 0.0, lbase = 0.0;
        int last_nz = -1;
        for (int i0 = 0; i0 < n_seg && seg < 0; i0 += 32) {
            const int i = i0 + lane;
            const double v = i < n_seg ? (double)seg_mass(d, sm, i) : 0.0;
            const double incl = warp_scan_d(v, lane);
            const unsigned cross = __ballot_sync(0xffffffffu, v > 0.0 && run + incl > thr);
            const unsigned nz = __ballot_sync(0xffffffffu, v > 0.0);
            if (cross) {
                const int l = __ffs(cross) - 1;
                seg = i0 + l;
                base = run + __shfl_sync(0xffffffffu, incl - v, l);
            } else if (nz) {
                const int l = 31 - __clz(nz);
                last_nz = i0 + l;
                lbase = run + __shfl_sync(0xffffffffu, incl - v, l);
            }
            run += __shfl_sync(0xffffffffu, incl, 31);
        }
        if (seg < 0) {  // rounding: the last segment of nonzero mass
            seg = last_nz;
            base = lbase;
        }
    }
    return seg >= 0 ? pick_in_segment<DT>(d, seg, n_units, V, (float)(thr - base), greedy, lane) : -1;
}

// The row maximum after a softmax pass (every thread); false if the row
// holds NaN or +Inf or no finite logit.
__device__ __forceinline__ bool row_max(const RowSmem& sm, int n_seg, int lane, float& M)
{
    M = -INFINITY;
    for (int i = lane; i < n_seg; i += 32) M = max_nan(M, sm.ref[i]);
    M = warp_max_redux(M);
    return sm.bad == 0 && M > -INFINITY && M == M;
}

template <int DT, int NT>
__global__ void __launch_bounds__(NT, 1024 / NT) sample_rows_kernel(SampleArgs a)
{
    using E = Elem<DT>;
    constexpr int EPU = E::kPerUnit;
    __shared__ RowSmem sm;
    const int r = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const int V = a.V;
    const int n_seg = ((V + EPU - 1) / EPU + kRSeg - 1) / kRSeg;
    const bool greedy = a.c == 0.f;
    if (tid == 0) sm.bad = 0;
    __syncthreads();
    Dist d;
    d.rowT = static_cast<const char*>(a.logits) + (size_t)r * (size_t)a.stride * E::kBytes;
    d.rowD = nullptr;
    d.c = a.c;
    d.residual = 0;
    d.xs = -1;
    d.cT = 0.f;
    softmax_pass<DT>(d.rowT, V, a.c, greedy, sm, lane, w);
    __syncthreads();
    float M;
    const bool ok = row_max(sm, n_seg, lane, M);
    int* const out = a.tokens + (size_t)r * a.n_samples;
    if (!ok) {
        for (int s = tid; s < a.n_samples; s += NT) out[s] = -1;
        if (tid == 0 && a.device_status) atomicOr(a.device_status, SDV_REQ_NONFINITE);
        return;
    }
    d.M = M;
    d.negM = -(M * a.c);
    // warp w takes draws w, w + NT / 32, ...
#pragma unroll 1
    for (int s = w; s < a.n_samples; s += NT / 32) {
        const float u = greedy ? 0.f : a.u[(size_t)r * a.n_samples + s];
        const int x = draw<DT>(d, sm, V, u, greedy, lane);
        if (lane == 0) out[s] = x;
    }
}

// ------------------------------------------------------------------------
// decision: one warp per request; the request's node records are copied to
// shared memory first, then lane 0 walks them

constexpr int kSlotsMax = (SDV_MAX_L + 1) * SDV_MAX_K;

struct DecideSmem {
    unsigned char own[kSlotsMax];
    float val[kSlotsMax];  // a (token), h (block) or argmax bits (greedy)
    float u[SDV_MAX_K * SDV_MAX_L];
    int tok[SDV_MAX_K * SDV_MAX_L];
    signed char sib[kSlotsMax];  // next sibling's draft, or -1
    int endn;                    // the end node: slot | leaf << 30, or -1 (no draw)
    int token;                   // the correction token once known (greedy, no draw), else -1
};

// Decide request b (one warp): accept_len, accept_draft, accept_prob,
// residual_mass, the status; the greedy token; s.endn for the draw.
__device__ void decide_request(const Problem& pb, int b, bool greedy, DecideSmem& s, int lane)
{
    const int K = pb.K, L = pb.L;
    if (lane == 0) {
        s.endn = -1;
        s.token = -1;
        if (pb.leaf_pending) pb.leaf_pending[b] = -1;
    }
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
    // the token walk: per-position rules (token-level sampling and K-SEQ)
    const bool token = pb.mode == SDV_MODE_TOKEN || pb.mode == SDV_MODE_KSEQ;
    unsigned char* own = s.own;
    float* val = s.val;
    float* uu = s.u;
    int* tk = s.tok;
    for (int i = lane; i < (Lb + 1) * K; i += 32) {
        own[i] = pb.ws.owner[s0 + i];
        float v;
        if (greedy)
            v = __int_as_float(pb.ws.am[s0 + i]);
        else if (token)
            v = pb.ws.a[s0 + i];
        else  // a leaf's block acceptance is its weight p (the node kernel skips leaves)
            v = i >= Lb * K ? (Lb == 0 ? 1.f : pb.ws.wt[s0 + i].y) : pb.ws.h[s0 + i];
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
        if (pb.residual_mass) pb.residual_mass[b] = 1.f;
        const size_t se = s0 + (size_t)ej * K + eo;
        if (ej < Lb) {
            pb.out_token[b] = s.token = __float_as_int(val[ej * K + eo]);
        } else if (pb.leaf_pending) {  // the LM head computes this leaf's row afterwards
            pb.out_token[b] = -1;
            pb.leaf_pending[b] = (int)se;
        } else {  // a leaf: its row is read now, by the CTA (its argmax is the correction)
            s.endn = (int)(se | (1u << 30));
        }
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
        signed char* sib = s.sib;
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
    s.endn = (int)(se | (leaf ? (1u << 30) : 0u));
    if (pb.residual_mass)
        pb.residual_mass[b] = leaf ? (token || Lb == 0 ? 1.f : pb.ws.wt[se].y) : pb.ws.S[se];
}

// A request found invalid after its decision (one warp): the outputs an
// invalid request gets, and its status bit.
__device__ __noinline__ void invalidate_request(const Problem& pb, int b, int lane)
{
    const int n = pb.K * pb.L;
    if (pb.accept_prob)
        for (int i = lane; i < n; i += 32) pb.accept_prob[(size_t)b * n + i] = 0.f;
    if (lane == 0) {
        pb.accept_len[b] = 0;
        pb.accept_draft[b] = 0;
        pb.out_token[b] = -1;
        if (pb.residual_mass) pb.residual_mass[b] = 0.f;
        atomicOr(&pb.ws.req[b], SDV_REQ_NONFINITE);
        if (pb.device_status) atomicOr(pb.device_status, SDV_REQ_NONFINITE);
    }
}

// The debug output residual_out[b][0..V): the normalised distribution the
// correction (or bonus) token was drawn from, written by every thread of
// the CTA after the draw.  tok >= 0 with one_hot: a one-hot row at tok
// (greedy); tok < 0 with one_hot: a zero row (an invalid request);
// otherwise each element's mass under d over the total the draw used.
template <int DT>
__device__ void write_residual_row(const Problem& pb, int b, const Dist& d, const RowSmem& sm, bool one_hot, int tok,
                                   int tid, int lane)
{
    constexpr int EPU = Elem<DT>::kPerUnit;
    const int V = pb.V;
    float* row = pb.residual_out + (size_t)b * V;
    if (one_hot) {
        for (int x = tid; x < V; x += (int)blockDim.x) row[x] = x == tok ? 1.f : 0.f;
        return;
    }
    const int n_units = (V + EPU - 1) / EPU;
    const int n_seg = (n_units + kRSeg - 1) / kRSeg;
    // the total, summed as the draw sums it (every warp for itself)
    const float tot = (float)row_total(d, sm, n_seg, lane);
    for (int ug = tid; ug < n_units; ug += (int)blockDim.x) {
        float v[EPU];
        unit_masses<DT>(d, ug, n_units, V, false, v);
#pragma unroll
        for (int e = 0; e < EPU; ++e)
            if (ug * EPU + e < V) row[ug * EPU + e] = v[e] / tot;
    }
}

// One CTA per request: the decision (warp 0), then the correction (or
// bonus) token at the end node it chose: from the node's final residual R_n
// (kept by the node kernel), or from P at a leaf or where S_n = 0.
template <int DT, int NT>
__global__ void __launch_bounds__(NT, 1024 / NT) finish_kernel(Problem pb, int greedy, int wait_nodes)
{
    using E = Elem<DT>;
    constexpr int EPU = E::kPerUnit;
    __shared__ RowSmem sm;
    __shared__ DecideSmem ds;
    const int b = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    if (wait_nodes) {
        // launched while the node kernel still runs: wait (bounded) until it
        // has finished every node of this request (its release, our acquire)
        if (tid == 0) {
            const int* left = pb.ws.left + b;
            int n;
            asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(n) : "l"(left) : "memory");
            if (n > 0) {
                const uint64_t t0 = globaltimer();
                do {
                    __nanosleep(256);  // leave issue slots to the node kernel's CTAs on this SM
                    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(n) : "l"(left) : "memory");
                } while (n > 0 && globaltimer() - t0 <= pb.wait_ns);
                if (n > 0) {
                    atomicOr(&pb.ws.req[b], SDV_DEV_TIMEOUT);
                    if (pb.device_status) atomicOr(pb.device_status, SDV_DEV_TIMEOUT);
                }
            }
        }
        __syncthreads();
    }
    if (w == 0) decide_request(pb, b, greedy != 0, ds, lane);
    if (tid == 0) sm.bad = 0;
    __syncthreads();
    const int e = ds.endn;
    if (e < 0) {  // greedy, or an invalid request: the decision wrote the outputs
        if (pb.residual_out) {
            Dist none = {};
            write_residual_row<DT>(pb, b, none, sm, true, ds.token, tid, lane);
        }
        return;
    }
    const int K = pb.K, L = pb.L, V = pb.V;
    const size_t slot = (size_t)(e & ((1 << 30) - 1));
    const bool leaf = (e >> 30) != 0;
    const int k = (int)(slot % K), j = (int)((slot / K) % (L + 1));
    const float u = greedy ? 0.f : pb.sample_u[((size_t)b * K + k) * (L + 1) + j];
    const int n_seg = ((V + EPU - 1) / EPU + kRSeg - 1) / kRSeg;
    Dist d;
    // a leaf's row may live elsewhere (e.g. host memory the device can read)
    const void* tsrc = leaf && pb.leaf_target ? pb.leaf_target : pb.target;
    d.rowT = static_cast<const char*>(tsrc) + (((size_t)b * K + k) * (L + 1) + j) * (size_t)pb.stride * E::kBytes;
    d.rowD = leaf ? nullptr
                  : static_cast<const char*>(pb.draft) + (((size_t)b * K + k) * L + j) * (size_t)pb.stride * E::kBytes;
    d.c = pb.c;
    // the end node's residual mass S_n; below 0 when the node kernel left it
    // to this pass (the token rule's last sweep): it is then the residual's
    // total here, and the residual, or P where it has no mass, is drawn from
    const float Sn = leaf ? 0.f : pb.ws.S[slot];
    const bool sum_here = !leaf && Sn < 0.f;
    d.residual = !leaf && (Sn > 0.f || sum_here);
    d.xs = -1;
    d.cT = 0.f;
    if (d.residual) {
        const float* prm = pb.ws.prm + slot * 6;
        d.negT = prm[0];
        d.negD = prm[1];
        d.aT = prm[2];
        d.rD = prm[3];
        d.Rs = prm[4];
        d.cT = prm[5];
        d.xs = pb.ws.xs[slot];
        residual_pass<DT>(d, V, sm, lane, w);
        __syncthreads();
        if (sum_here) {
            const double tot = fmax(row_total(d, sm, n_seg, lane), 0.0);  // as the draw sums it
            if (tid == 0 && pb.residual_mass) pb.residual_mass[b] = (float)tot;
            d.residual = tot > 0.0;
        }
    }
    if (!d.residual) {
        softmax_pass<DT>(d.rowT, V, d.c, greedy != 0, sm, lane, w);
        __syncthreads();
        float M;
        if (!row_max(sm, n_seg, lane, M)) {
            // an unusable row: only a leaf's can be (the node kernel checked
            // every inner node's rows), and a leaf's row is read here alone,
            // so the request is found invalid now: its outputs are replaced
            if (w == 0) invalidate_request(pb, b, lane);
            if (pb.residual_out) write_residual_row<DT>(pb, b, d, sm, true, -1, tid, lane);
            return;
        }
        d.M = M;
        d.negM = -(M * d.c);
    }
    if (w == 0) {
        const int x = draw<DT>(d, sm, V, u, greedy != 0, lane);
        if (lane == 0) pb.out_token[b] = ds.token = x;
    }
    if (pb.residual_out) {
        __syncthreads();
        write_residual_row<DT>(pb, b, d, sm, greedy != 0, ds.token, tid, lane);
    }
}

}  // namespace


namespace {

// The device's SM count, asked once per device.
cudaError_t sm_count_cached(int* n_sm)
{
    constexpr int kDevs = 64;
    static int sms[kDevs];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    int n = dev >= 0 && dev < kDevs ? sms[dev] : 0;
    if (n == 0) {
        e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        if (n <= 0) n = 1;
        if (dev >= 0 && dev < kDevs) sms[dev] = n;
    }
    *n_sm = n;
    return cudaSuccess;
}

}  // namespace

cudaError_t launch_finish(const Problem& pb, bool greedy, cudaStream_t st, bool after_nodes)
{
    if (pb.B == 0) return cudaSuccess;
    // One CTA per request; its passes over the end node's rows are bound by
    // instruction issue within the CTA, so when the requests are no more
    // than the SMs (one CTA per SM) each CTA takes 32 warps, else 16 (two
    // CTAs per SM).
    int n_sm = 0;
    const cudaError_t e = sm_count_cached(&n_sm);
    if (e != cudaSuccess) return e;
    const bool wide = pb.B <= n_sm;
    // after the node kernel: a programmatic dependent launch, so that the
    // decisions of finished requests overlap the node kernel's last nodes
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)pb.B);
    cfg.blockDim = dim3(wide ? 1024 : 512);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = after_nodes ? 1 : 0;
    const int g = greedy ? 1 : 0, wait = after_nodes ? 1 : 0;
    if (pb.dtype == SDV_BF16)
        return wide ? cudaLaunchKernelEx(&cfg, finish_kernel<SDV_BF16, 1024>, pb, g, wait)
                    : cudaLaunchKernelEx(&cfg, finish_kernel<SDV_BF16, 512>, pb, g, wait);
    return wide ? cudaLaunchKernelEx(&cfg, finish_kernel<SDV_F32, 1024>, pb, g, wait)
                : cudaLaunchKernelEx(&cfg, finish_kernel<SDV_F32, 512>, pb, g, wait);
}

cudaError_t launch_sample_rows(const SampleArgs& a, cudaStream_t st)
{
    if (a.n_rows == 0 || a.n_samples == 0) return cudaSuccess;
    // One CTA per row; its warps share the row's pass, then take one draw
    // each at a time.  The CTAs are sized so that the launch holds about
    // 32 warps per SM: with many rows, small CTAs, many per SM, so that
    // while one CTA draws (a serial scan and a 4 KB re-read) the others
    // stream their rows; with few rows, larger CTAs, so that each row's
    // pass has warps enough to keep its loads in flight.  At least one warp
    // per draw, up to 16.  Measured on rows of V = 151936 bf16, one draw
    // each, single calls alternated in one process (against 16 warps):
    // 512 rows 8 warps 4% faster (4 warps 19% slower), 1024 rows 4 warps
    // 10.5% faster, 2048 rows 2 warps 6.5% faster.
    int n_sm = 0;
    const cudaError_t e = sm_count_cached(&n_sm);
    if (e != cudaSuccess) return e;
    int warps = 2;
    while (warps < 16 && (long long)warps * 2 * a.n_rows <= 32LL * n_sm) warps *= 2;
    while (warps < 16 && warps < a.n_samples) warps *= 2;
    const int nt = 32 * warps;
    if (a.dtype == SDV_BF16) {
        if (nt == 64) sample_rows_kernel<SDV_BF16, 64><<<a.n_rows, 64, 0, st>>>(a);
        else if (nt == 128) sample_rows_kernel<SDV_BF16, 128><<<a.n_rows, 128, 0, st>>>(a);
        else if (nt == 256) sample_rows_kernel<SDV_BF16, 256><<<a.n_rows, 256, 0, st>>>(a);
        else sample_rows_kernel<SDV_BF16, 512><<<a.n_rows, 512, 0, st>>>(a);
    } else {
        if (nt == 64) sample_rows_kernel<SDV_F32, 64><<<a.n_rows, 64, 0, st>>>(a);
        else if (nt == 128) sample_rows_kernel<SDV_F32, 128><<<a.n_rows, 128, 0, st>>>(a);
        else if (nt == 256) sample_rows_kernel<SDV_F32, 256><<<a.n_rows, 256, 0, st>>>(a);
        else sample_rows_kernel<SDV_F32, 512><<<a.n_rows, 512, 0, st>>>(a);
    }
    return cudaGetLastError();
}

}  // namespace sdv
