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
#include "sdv_device.cuh"
#include "sdv_internal.h"

namespace sdv {
namespace {

constexpr int kRW = 16;                                   // warps per CTA
constexpr int kRT = 32 * kRW;                             // threads per CTA
constexpr int kRU = 8;                                    // units per lane per step
constexpr int kRSeg = 32 * kRU;                           // units per segment (one warp, one step)
constexpr int kRStep = kRW * kRSeg;                       // units per step
constexpr int kRMaxSeg = (SDV_MAX_V / 4 + kRSeg - 1) / kRSeg;  // segments of the longest row

struct RowSmem {
    float mass[kRMaxSeg];  // per segment: sum of 2^(x c - ref c)
    float ref[kRMaxSeg];   // per segment: its maximum (the reference)
    float redm[kRW];
    int bad;
};

template <int DT>
__device__ __forceinline__ uint4 load_unit(const char* row, int ug, int n_units)
{
    if (ug >= n_units) return make_uint4(0u, 0u, 0u, 0u);  // never summed: the caller masks it
    return __ldg(reinterpret_cast<const uint4*>(row) + ug);
}

// Inverse CDF inside segment seg of a row: the masses of its elements are
// recomputed (2^(x c - M c), or 1 at the maximum for T = 0) and the first
// element whose running sum exceeds `local` is returned (the last element
// of nonzero mass if rounding leaves none).  Warp-wide; every lane gets it.
template <int DT>
__device__ int pick_in_segment(const char* row, int seg, int n_units, int V, float c, float negM, float local,
                               bool greedy, float M, int lane)
{
    constexpr int EPU = Elem<DT>::kPerUnit;
    float run = 0.f;
    int lastx = -1;
#pragma unroll 1
    for (int i = 0; i < kRU; ++i) {
        const int ug = seg * kRSeg + i * 32 + lane;
        float v[EPU];
        if (ug < n_units) {
            unpack_masked<DT>(__ldg(reinterpret_cast<const uint4*>(row) + ug), ug * EPU, V, v);
        } else {
#pragma unroll
            for (int e = 0; e < EPU; ++e) v[e] = -INFINITY;
        }
        float lsum = 0.f;
        int lnz = -1;
#pragma unroll
        for (int e = 0; e < EPU; ++e) {
            const float w = greedy ? (v[e] == M ? 1.f : 0.f) : ex2(fmaf(v[e], c, negM));
            v[e] = w;
            lsum += w;
            if (w > 0.f) lnz = ug * EPU + e;
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

template <int DT>
__global__ void __launch_bounds__(kRT, 2) sample_rows_kernel(SampleArgs a)
{
    using E = Elem<DT>;
    constexpr int EPU = E::kPerUnit;
    __shared__ RowSmem sm;
    const int r = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const int V = a.V;
    const int n_units = (V + EPU - 1) / EPU;
    const int n_seg = (n_units + kRSeg - 1) / kRSeg;
    const int n_steps = (n_units + kRStep - 1) / kRStep;
    const char* row = static_cast<const char*>(a.logits) + (size_t)r * (size_t)a.stride * E::kBytes;
    const bool greedy = a.c == 0.f;
    const float c = a.c;
    if (tid == 0) sm.bad = 0;

    // ---- one pass: per-segment maximum and mass ----
    bool bad = false;
#pragma unroll 1
    for (int st = 0; st < n_steps; ++st) {
        const int seg = st * kRW + w;
        const int ug0 = seg * kRSeg + lane;
        uint4 u[kRU];
#pragma unroll
        for (int i = 0; i < kRU; ++i) u[i] = load_unit<DT>(row, ug0 + i * 32, n_units);
        // the segment's maximum: whole units packed, the row's last unit masked
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
        bad |= (cm != cm) || cm == INFINITY;  // NaN or +Inf makes the row unusable
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
#pragma unroll
                    for (int e = 0; e < EPU; ++e) v[e] = ex2(fmaf(v[e], c, negm));
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
    __syncthreads();

    // ---- the row maximum, and whether the row can be used ----
    float M = -INFINITY;
    for (int i = lane; i < n_seg; i += 32) M = max_nan(M, sm.ref[i]);
    M = warp_max_redux(M);
    const bool unusable = sm.bad != 0 || !(M > -INFINITY) || M != M;
    int* const out = a.tokens + (size_t)r * a.n_samples;
    if (unusable) {
        for (int s = tid; s < a.n_samples; s += kRT) out[s] = -1;
        if (tid == 0 && a.device_status) atomicOr(a.device_status, SDV_REQ_NONFINITE);
        return;
    }
    const float negM = -(M * c);

    // ---- draws: warp w takes draws w, w + 16, ... ----
#pragma unroll 1
    for (int s = w; s < a.n_samples; s += kRW) {
        int seg = -1;
        float base = 0.f, thr = 0.f;
        if (greedy) {
            // the first segment holding the maximum
            for (int i0 = 0; i0 < n_seg && seg < 0; i0 += 32) {
                const int i = i0 + lane;
                const unsigned hit = __ballot_sync(0xffffffffu, i < n_seg && sm.ref[i] == M);
                if (hit) seg = i0 + __ffs(hit) - 1;
            }
            thr = 0.5f;  // the first element equal to M (mass 1) crosses 0.5
        } else {
            // segment masses in the row's reference; their total S
            float tot = 0.f;
            for (int i = lane; i < n_seg; i += 32) {
                const float ref = sm.ref[i];
                tot += ref > -INFINITY ? sm.mass[i] * ex2((ref - M) * c) : 0.f;
            }
            tot = warp_sum(tot);
            thr = a.u[(size_t)r * a.n_samples + s] * tot;
            float run = 0.f, lbase = 0.f;
            int last_nz = -1;
            for (int i0 = 0; i0 < n_seg && seg < 0; i0 += 32) {
                const int i = i0 + lane;
                const float ref = i < n_seg ? sm.ref[i] : -INFINITY;
                const float v = ref > -INFINITY ? sm.mass[i] * ex2((ref - M) * c) : 0.f;
                float incl = v;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const float n = __shfl_up_sync(0xffffffffu, incl, o);
                    if (lane >= o) incl += n;
                }
                const unsigned cross = __ballot_sync(0xffffffffu, v > 0.f && run + incl > thr);
                const unsigned nz = __ballot_sync(0xffffffffu, v > 0.f);
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
        const int x = seg >= 0 ? pick_in_segment<DT>(row, seg, n_units, V, c, negM, thr - base, greedy, M, lane) : -1;
        if (lane == 0) out[s] = x;
    }
}

}  // namespace

int sample_threads() { return kRT; }

cudaError_t launch_sample_rows(const SampleArgs& a, cudaStream_t st)
{
    if (a.n_rows == 0 || a.n_samples == 0) return cudaSuccess;
    if (a.dtype == SDV_BF16)
        sample_rows_kernel<SDV_BF16><<<a.n_rows, kRT, 0, st>>>(a);
    else
        sample_rows_kernel<SDV_F32><<<a.n_rows, kRT, 0, st>>>(a);
    return cudaGetLastError();
}

}  // namespace sdv
