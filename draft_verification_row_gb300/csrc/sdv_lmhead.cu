// sdv_lmhead.cu -- the target model's LM head on the 5th-generation tensor
// cores, with greedy verification folded into its epilogue.
//
// The target model's pass ends in its LM head, logits = hidden . W^T
// ("Speculative Decoding: Performance or Illusion?", section 3.2: the target
// pass is the verification step).  That is a dense contraction of M rows
// (the trie nodes whose target rows verification reads) by V vocabulary
// entries over the hidden size d, so it runs on tcgen05:
//
// lm_head_kernel    persistent, one CTA per SM, 192 threads:
//                     warp 0     TMA producer: 128 x 64 tiles of hidden and
//                                256 x 64 tiles of W (bf16, 128-byte
//                                swizzle) into a 4-stage shared-memory ring;
//                     warp 1     one thread issues tcgen05.mma (kind::f16,
//                                bf16 in, fp32 accumulate) into a 128 x 256
//                                accumulator in tensor memory; two
//                                accumulators (all 512 TMEM columns), so the
//                                epilogue of one tile overlaps the MMAs of
//                                the next;
//                     warps 2-5  epilogue: tcgen05.ld, one row per thread.
//                   Epilogues: ARGMAX folds the tile's maximum and its first
//                   index into one 64-bit atomicMax per row (the logits
//                   never reach memory); LOGITS stores the fp32 logits.
// lm_rows_kernel    one CTA per request: numbers the request's inner trie
//                   nodes (one per distinct draft prefix of length
//                   0..L_b - 1) and copies their hidden rows into one
//                   contiguous block, the GEMM's A operand.
// lm_argmax_kernel  one thread per node: its argmax out of the 64-bit key.
// Leaves (depth L_b) are not listed: greedy matching uses the inner nodes'
// argmaxes only, and a leaf's argmax is the correction only where the
// decision ends there.  After the decision, lm_leaf_rows_kernel lists those
// leaves (one per request at most), the LM head runs again over them, and
// lm_leaf_token_kernel writes their tokens.
//
// Tiles are ordered vocabulary-major (consecutive tiles share a W tile), so
// the CTAs running at one time read the same few MB of W from L2 while all
// hidden rows stay L2-resident.
#include <cuda.h>
#include <cuda_bf16.h>

#include "sdv_internal.h"
#include "sdv_device.cuh"

namespace sdv {
namespace {

constexpr int kBM = 128;  // rows per tile: the 128 TMEM lanes
constexpr int kBN = 256;  // vocabulary entries per tile: TMEM columns of one accumulator
constexpr int kBK = 64;   // hidden elements per stage: one 128-byte swizzle atom of bf16
constexpr int kUK = 16;   // K of one tcgen05.mma kind::f16
constexpr int kStages = 4;
constexpr uint32_t kTileA = kBM * kBK * 2;  // 16 KB
constexpr uint32_t kTileB = kBN * kBK * 2;  // 32 KB
constexpr int kLmThreads = 192;
constexpr uint32_t kTmemCols = 2 * kBN;  // two fp32 accumulators: all 512 columns

// Instruction descriptor of tcgen05.mma kind::f16: fp32 accumulator (bits
// 4-5 = 1), bf16 A and B (bits 7-9 and 10-12 = 1), both K-major (bits 15,
// 16 = 0), N >> 3 in bits 17-22, M >> 4 in bits 24-28.
constexpr uint32_t kIdesc =
    (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(kBN >> 3) << 17) | ((uint32_t)(kBM >> 4) << 24);

struct LmBars {
    uint64_t full[kStages];   // TMA -> MMA: the stage's tiles landed
    uint64_t empty[kStages];  // MMA -> TMA: the stage's MMAs have read it
    uint64_t tfull[2];        // MMA -> epilogue: accumulator complete
    uint64_t tempty[2];       // epilogue -> MMA: accumulator read (4 warps)
    uint64_t drain;           // MMA: nothing of ours in flight
    uint32_t tmem_base;
};

constexpr size_t kBarsBytes = (sizeof(LmBars) + 127) / 128 * 128;
// ROWS_BF16 epilogue: each epilogue warp stages its 32 rows x 64 columns of
// bf16 (rows 128 B apart plus 16 B of padding against bank conflicts), then
// writes whole 128-byte row segments.
constexpr int kStageCols = 64;
constexpr int kStagePitch = kStageCols * 2 + 16;   // 144 B
constexpr int kStageWarpBytes = 32 * kStagePitch;  // 4608 B
constexpr size_t kLmSmem = 1024 + (size_t)kStages * (kTileA + kTileB) + kBarsBytes + 4 * kStageWarpBytes;

// The CTA-pair form (tcgen05 cta_group::2): a cluster of two CTAs on one TPC
// computes 256 x 256 tiles.  Each CTA holds its own 128 rows of hidden and
// half (128 rows) of W's 256-row tile; one MMA of M = 256 reads both CTAs'
// halves, and each CTA's tensor memory receives its own 128 rows by all 256
// columns.  Per SM, a 128 x 256 x 16 step then reads 8 KB of operands from
// shared memory instead of 12 KB, and TMA writes 32 KB per stage instead of
// 48 KB, so deeper pipelining fits in the same space.
constexpr int kPairStages = 6;
constexpr uint32_t kHalfB = (kBN / 2) * kBK * 2;  // 16 KB
constexpr uint32_t kIdescPair =
    (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(kBN >> 3) << 17) | ((uint32_t)((2 * kBM) >> 4) << 24);

struct PairBars {
    uint64_t full[kPairStages];   // TMA (both CTAs) -> MMA: the stage's four tiles landed (leader's)
    uint64_t empty[kPairStages];  // MMA -> TMA: the stage's MMAs have read it (each CTA's)
    uint64_t tfull[2];            // MMA -> epilogue (each CTA's)
    uint64_t tempty[2];           // epilogues of both CTAs -> MMA (leader's, 8 warps)
    uint64_t drain;
    uint32_t tmem_base;
};
constexpr size_t kPairBarsBytes = (sizeof(PairBars) + 127) / 128 * 128;
constexpr size_t kPairSmem = 1024 + (size_t)kPairStages * (kTileA + kHalfB) + kPairBarsBytes + 4 * kStageWarpBytes;

// ------------------------------------------------------------------------
// PTX: TMA, tcgen05

__device__ __forceinline__ void mbar_arrive(uint64_t* bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// A tile into shared memory, with an L2 eviction-priority hint.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar,
                                            uint64_t pol)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, "
        "{%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(pol)
        : "memory");
}

// L2 hints of the operands: the hidden rows are read again for every
// vocabulary tile (evict_last); a tile of W is read by the CTAs working on
// it at about the same time and never again (evict_first).  Measured with
// the CTA-pair form at d = 4096, V = 151936, 6401 rows, single calls of the
// two builds alternated in one process: 0.8-0.9% faster than evict_normal.
__device__ __forceinline__ uint64_t policy_keep()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t policy_stream()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot)),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish()
{
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor of a K-major bf16 tile written by TMA with
// the 128-byte swizzle: rows of 128 B, 8-row groups 1024 B apart (stride
// byte offset), descriptor version 1, layout 2 = 128-byte swizzle.  The
// leading byte offset is unused for this layout.  The tile must start on a
// 1024-byte boundary; a step of 16 elements along K adds 32 B (2 in the
// address field, which counts 16-byte units).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr)
{
    return (uint64_t)((saddr >> 4) & 0x3fffu) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
           ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t da, uint64_t db, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(da), "l"(db), "r"(kIdesc), "r"(accumulate)
        : "memory");
}

// Arrives on the barrier once every tcgen05 operation this thread issued
// before it has completed.
__device__ __forceinline__ void mma_commit(uint64_t* bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

// 32 consecutive fp32 columns of this thread's TMEM lane; the wait is in the
// same statement, so the registers are valid when it returns.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
          "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]),
          "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]),
          "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
        : "r"(taddr)
        : "memory");
}

// ---- the CTA-pair form

__device__ __forceinline__ uint32_t cluster_ctarank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Every thread of both CTAs (release / acquire at cluster scope).
__device__ __forceinline__ void cluster_sync()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// The address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t peer_smem(uint32_t saddr, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
    return r;
}

// A tile into this CTA's shared memory whose completion is counted on a
// barrier of either CTA of the pair (bar: a shared::cluster address), with
// an L2 eviction-priority hint (pol: a createpolicy value).
__device__ __forceinline__ void tma_load_2d_pair(void* dst, const CUtensorMap* map, int x, int y, uint32_t bar,
                                                 uint64_t pol)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
        "[%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar), "l"(pol)
        : "memory");
}

// Allocation and release of tensor memory in both CTAs of the pair (one
// warp of each CTA takes part).
__device__ __forceinline__ void tmem_alloc_pair(uint32_t* slot, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot)),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish_pair()
{
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void mma_bf16_pair(uint32_t d_tmem, uint64_t da, uint64_t db, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(da), "l"(db), "r"(kIdescPair), "r"(accumulate)
        : "memory");
}

// Arrives on the barrier at this offset in both CTAs once every MMA this
// thread issued before it has completed.
__device__ __forceinline__ void mma_commit_pair_both(uint64_t* bar)
{
    const unsigned short both = 3;
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
            smem_u32(bar)),
        "h"(both)
        : "memory");
}

// The same, on this CTA's barrier only.
__device__ __forceinline__ void mma_commit_pair_local(uint64_t* bar)
{
    asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

// Arrival on a barrier of the other CTA (bar: a shared::cluster address).
__device__ __forceinline__ void mbar_arrive_remote(uint32_t bar)
{
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar) : "memory");
}

// A bounded wait that also acquires at cluster scope (arrivals made by the
// other CTA's threads).
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t* bar, uint32_t phase)
{
    auto try_once = [&]() {
        uint32_t ok;
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(ok)
            : "r"(smem_u32(bar)), "r"(phase)
            : "memory");
        return ok != 0;
    };
    if (try_once()) return true;
    const uint64_t t0 = globaltimer();
    while (!try_once()) {
        if (globaltimer() - t0 > kWaitNs) return false;
    }
    return true;
}

// A row's (maximum, first index) as one integer whose unsigned order is the
// order of the pair: larger value first, then lower index.  -0 is taken as
// +0 (they compare equal).  An unusable row (NaN or +Inf) gets the largest
// key, which decodes to NaN.
__device__ __forceinline__ unsigned long long argmax_key(float best, int idx, bool bad)
{
    if (bad) return ~0ull;
    if (best == 0.f) best = 0.f;
    const uint32_t u = __float_as_uint(best);
    const uint32_t ord = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    return ((unsigned long long)ord << 32) | (unsigned long long)(0xffffffffu - (uint32_t)idx);
}

__device__ __forceinline__ float key_value(unsigned long long key)
{
    const uint32_t ord = (uint32_t)(key >> 32);
    return __uint_as_float((ord & 0x80000000u) ? (ord & 0x7fffffffu) : ~ord);
}

// ------------------------------------------------------------------------
// the LM head

// One tile's epilogue for one warp: its 32 TMEM lanes (rows row0 + lane)
// by kBN columns from n0 (vocabulary indices).  ARGMAX returns the lane's
// (maximum, first index) key; the other forms write their rows.
template <int EPI>
__device__ __forceinline__ unsigned long long epilogue_tile(const LmArgs& a, uint32_t taddr, int row0, int n0, int M,
                                                            unsigned char* stage, int lane)
{
    const int row = row0 + lane;
    const int dest = EPI == LM_EPI_ROWS_BF16 && row < M ? a.dest_row[row] : 0;
    float best = -INFINITY;
    int bidx = n0;
    bool bad = false;
#pragma unroll 1
    for (int c = 0; c < kBN / 32; ++c) {
        uint32_t v[32];
        tmem_ld32(taddr + (uint32_t)(c * 32), v);
        const int x0 = n0 + c * 32;
        if (EPI == LM_EPI_ARGMAX) {
#pragma unroll
            for (int e = 0; e < 32; ++e) {
                const float f = __uint_as_float(v[e]);
                if (x0 + e < a.V) {
                    bad |= (f != f) || (f == INFINITY);
                    if (f > best) {
                        best = f;
                        bidx = x0 + e;
                    }
                }
            }
        } else if (EPI == LM_EPI_ROWS_BF16) {
            // this lane's 32 columns, rounded to bf16 (nearest even),
            // into its staging row
            const int half = c & 1;
#pragma unroll
            for (int e = 0; e < 32; e += 8) {
                uint32_t p[4];
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    const __nv_bfloat162 b2 = __floats2bfloat162_rn(__uint_as_float(v[e + 2 * h]),
                                                                    __uint_as_float(v[e + 2 * h + 1]));
                    p[h] = *reinterpret_cast<const uint32_t*>(&b2);
                }
                *reinterpret_cast<uint4*>(stage + lane * kStagePitch + half * 64 + e * 2) =
                    make_uint4(p[0], p[1], p[2], p[3]);
            }
            if (half == 1) {
                // 32 rows x 64 columns staged: 8 lanes per row, four
                // rows per store, each row's 128 bytes in one piece
                __syncwarp();
                const int xs = n0 + (c - 1) * 32;
                const int seg = lane & 7;
#pragma unroll 1
                for (int it = 0; it < 8; ++it) {
                    const int rl = it * 4 + (lane >> 3);
                    const int drow = __shfl_sync(0xffffffffu, dest, rl);
                    const int col = xs + seg * 8;
                    if (row0 + rl < M && col < a.V) {
                        const unsigned char* src = stage + rl * kStagePitch + seg * 16;
                        __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out_bf16) +
                                             (size_t)drow * (size_t)a.out_stride + col;
                        if (col + 8 <= a.V) {  // streaming: the logits should not evict W from L2
                            __stcs(reinterpret_cast<uint4*>(out), *reinterpret_cast<const uint4*>(src));
                        } else {
                            for (int e = 0; e < 8 && col + e < a.V; ++e)
                                out[e] = reinterpret_cast<const __nv_bfloat16*>(src)[e];
                        }
                    }
                }
                __syncwarp();
            }
        } else if (row < M) {
            float* out = a.logits + (size_t)row * (size_t)a.out_stride + x0;
            if (x0 + 32 <= a.V) {
#pragma unroll
                for (int e = 0; e < 32; e += 4)
                    *reinterpret_cast<float4*>(out + e) =
                        make_float4(__uint_as_float(v[e]), __uint_as_float(v[e + 1]),
                                    __uint_as_float(v[e + 2]), __uint_as_float(v[e + 3]));
            } else {
#pragma unroll
                for (int e = 0; e < 32; ++e)
                    if (x0 + e < a.V) out[e] = __uint_as_float(v[e]);
            }
        }
    }
    return EPI == LM_EPI_ARGMAX ? argmax_key(best, bidx, bad) : 0ull;
}


template <int EPI>
__global__ void __launch_bounds__(kLmThreads, 1)
    lm_head_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, LmArgs a)
{
    extern __shared__ unsigned char lm_raw[];
    // the swizzled tiles start on a 1024-byte boundary
    unsigned char* tiles = lm_raw + ((1024u - (smem_u32(lm_raw) & 1023u)) & 1023u);
    LmBars& s = *reinterpret_cast<LmBars*>(tiles + (size_t)kStages * (kTileA + kTileB));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int M = a.rows_dev ? *a.rows_dev : a.rows;
    const int mt = (M + kBM - 1) / kBM, nt = (a.V + kBN - 1) / kBN;
    const long long n_tiles = (long long)mt * nt;
    const int nkb = (a.d + kBK - 1) / kBK;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&s.full[i], 1);
            mbar_init(&s.empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&s.tfull[i], 1);
            mbar_init(&s.tempty[i], 4);
        }
        mbar_init(&s.drain, 1);
        mbar_fence_init();
    }
    if (warp == 1) {
        tmem_alloc(&s.tmem_base, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s.tmem_base;
    bool ok = true;

    if (warp == 0) {
        if (lane == 0) {  // TMA producer
            const uint64_t pol_a = policy_keep(), pol_b = policy_stream();
            uint32_t st = 0, ph = 0;
            long long issued = 0;
            for (long long t = blockIdx.x; t < n_tiles && ok; t += gridDim.x) {
                const int m0 = (int)(t % mt) * kBM, n0 = (int)(t / mt) * kBN;
                for (int kb = 0; kb < nkb; ++kb) {
                    if (!mbar_wait_bounded(&s.empty[st], ph ^ 1)) {
                        ok = false;
                        break;
                    }
                    mbar_expect_tx(&s.full[st], kTileA + kTileB);
                    tma_load_2d(tiles + st * kTileA, &tmA, kb * kBK, m0, &s.full[st], pol_a);
                    tma_load_2d(tiles + kStages * kTileA + st * kTileB, &tmB, kb * kBK, n0, &s.full[st], pol_b);
                    ++issued;
                    if (++st == kStages) {
                        st = 0;
                        ph ^= 1;
                    }
                }
            }
            if (ok) {
                // every stage's last release has arrived before the CTA exits
                for (int i = 0; i < kStages && ok; ++i) {
                    ok = mbar_wait_bounded(&s.empty[st], ph ^ 1);
                    if (++st == kStages) {
                        st = 0;
                        ph ^= 1;
                    }
                }
            } else {
                // gave up: wait (bounded) for the copies already issued
                for (int i = 0; i < kStages; ++i) {
                    const long long fills = issued > i ? (issued - 1 - i) / kStages + 1 : 0;
                    if (fills) mbar_wait_bounded(&s.full[i], (uint32_t)((fills - 1) & 1));
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {  // MMA issuer
            uint32_t st = 0, ph = 0;
            int i = 0;
            bool issued = false;
            for (long long t = blockIdx.x; t < n_tiles && ok; t += gridDim.x, ++i) {
                const int acc = i & 1;
                if (!mbar_wait_bounded(&s.tempty[acc], (((uint32_t)i >> 1) & 1) ^ 1)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem + (uint32_t)(acc * kBN);
                for (int kb = 0; kb < nkb; ++kb) {
                    if (!mbar_wait_bounded(&s.full[st], ph)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    issued = true;
                    const uint64_t da = sw128_desc(smem_u32(tiles + st * kTileA));
                    const uint64_t db = sw128_desc(smem_u32(tiles + kStages * kTileA + st * kTileB));
#pragma unroll
                    for (int k = 0; k < kBK / kUK; ++k)
                        mma_bf16(d_tmem, da + 2 * k, db + 2 * k, (kb | k) != 0 ? 1u : 0u);
                    mma_commit(&s.empty[st]);  // the stage is free once these MMAs have read it
                    if (++st == kStages) {
                        st = 0;
                        ph ^= 1;
                    }
                }
                if (!ok) break;
                mma_commit(&s.tfull[acc]);
            }
            if (issued) {  // nothing of ours in flight when TMEM is released
                mma_commit(&s.drain);
                if (!mbar_wait_bounded(&s.drain, 0)) ok = false;
            }
        }
    } else {  // epilogue: warp w may read TMEM lanes 32 (w % 4) .. + 31
        const int q = warp & 3;
        unsigned char* const stage =
            tiles + (size_t)kStages * (kTileA + kTileB) + kBarsBytes + (size_t)(warp - 2) * kStageWarpBytes;
        int i = 0;
        for (long long t = blockIdx.x; t < n_tiles; t += gridDim.x, ++i) {
            const int acc = i & 1;
            const int m0 = (int)(t % mt) * kBM, n0 = (int)(t / mt) * kBN;
            ok = __all_sync(0xffffffffu, mbar_wait_bounded(&s.tfull[acc], ((uint32_t)i >> 1) & 1));
            if (!ok) break;
            tc_fence_after();
            const uint32_t taddr = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * kBN);
            const int row = m0 + q * 32 + lane;
            const unsigned long long key = epilogue_tile<EPI>(a, taddr, m0 + q * 32, n0, M, stage, lane);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&s.tempty[acc]);
            if (EPI == LM_EPI_ARGMAX && row < M) atomicMax(a.keys + row, key);
        }
    }

    if (!ok && a.device_status) atomicOr(a.device_status, SDV_DEV_TIMEOUT);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

// The CTA-pair form of the same GEMM.  Clusters of two CTAs; rank 0 (the
// leader) issues the MMAs of M = 256 for both.  A pair tile is two 128-row
// tiles of hidden (row tiles 2p and 2p + 1) by 256 vocabulary entries.
// Both CTAs' TMA loads count on the leader's full barrier; the leader's
// commits arrive on both CTAs' empty and tfull barriers; both CTAs'
// epilogue warps arrive on the leader's tempty barrier.
template <int EPI>
__global__ void __launch_bounds__(kLmThreads, 1)
    lm_head_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, LmArgs a)
{
    extern __shared__ unsigned char lm_raw[];
    unsigned char* tiles = lm_raw + ((1024u - (smem_u32(lm_raw) & 1023u)) & 1023u);
    PairBars& s = *reinterpret_cast<PairBars*>(tiles + (size_t)kPairStages * (kTileA + kHalfB));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const long long cluster = blockIdx.x >> 1, n_clusters = gridDim.x >> 1;
    const int M = a.rows_dev ? *a.rows_dev : a.rows;
    const int mt = (M + kBM - 1) / kBM, mp = (mt + 1) / 2, nt = (a.V + kBN - 1) / kBN;
    const long long n_tiles = (long long)mp * nt;
    const int nkb = (a.d + kBK - 1) / kBK;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kPairStages; ++i) {
            mbar_init(&s.full[i], 1);
            mbar_init(&s.empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&s.tfull[i], 1);
            mbar_init(&s.tempty[i], 8);
        }
        mbar_init(&s.drain, 1);
        mbar_fence_init();
    }
    if (warp == 1) {
        tmem_alloc_pair(&s.tmem_base, kTmemCols);
        tmem_relinquish_pair();
    }
    // the barriers of both CTAs are initialised before either uses the other's
    tc_fence_before();
    cluster_sync();
    tc_fence_after();
    const uint32_t tmem = s.tmem_base;
    bool ok = true;

    if (warp == 0) {
        if (lane == 0) {  // TMA producer (both CTAs): this CTA's row tile and half of W's
            const uint64_t pol_a = policy_keep(), pol_b = policy_stream();
            uint32_t st = 0, ph = 0;
            long long issued = 0;
            for (long long t = cluster; t < n_tiles && ok; t += n_clusters) {
                const int m0 = (int)(2 * (t % mp) + rank) * kBM;
                const int n0 = (int)(t / mp) * kBN + (int)rank * (kBN / 2);
                for (int kb = 0; kb < nkb; ++kb) {
                    if (!mbar_wait_bounded(&s.empty[st], ph ^ 1)) {
                        ok = false;
                        break;
                    }
                    if (rank == 0) mbar_expect_tx(&s.full[st], 2 * (kTileA + kHalfB));
                    const uint32_t fb = peer_smem(smem_u32(&s.full[st]), 0);
                    tma_load_2d_pair(tiles + st * kTileA, &tmA, kb * kBK, m0, fb, pol_a);
                    tma_load_2d_pair(tiles + kPairStages * kTileA + st * kHalfB, &tmB, kb * kBK, n0, fb, pol_b);
                    ++issued;
                    if (++st == kPairStages) {
                        st = 0;
                        ph ^= 1;
                    }
                }
            }
            if (ok) {
                // every stage's last release has arrived before the CTA exits
                for (int i = 0; i < kPairStages && ok; ++i) {
                    ok = mbar_wait_bounded(&s.empty[st], ph ^ 1);
                    if (++st == kPairStages) {
                        st = 0;
                        ph ^= 1;
                    }
                }
            } else if (rank == 0) {
                // gave up: wait (bounded) for the copies already issued
                for (int i = 0; i < kPairStages; ++i) {
                    const long long fills = issued > i ? (issued - 1 - i) / kPairStages + 1 : 0;
                    if (fills) mbar_wait_bounded(&s.full[i], (uint32_t)((fills - 1) & 1));
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && rank == 0) {  // MMA issuer: the leader only
            uint32_t st = 0, ph = 0;
            int i = 0;
            bool issued = false;
            for (long long t = cluster; t < n_tiles && ok; t += n_clusters, ++i) {
                const int acc = i & 1;
                if (!mbar_wait_cluster(&s.tempty[acc], (((uint32_t)i >> 1) & 1) ^ 1)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem + (uint32_t)(acc * kBN);
                for (int kb = 0; kb < nkb; ++kb) {
                    if (!mbar_wait_bounded(&s.full[st], ph)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    issued = true;
                    const uint64_t da = sw128_desc(smem_u32(tiles + st * kTileA));
                    const uint64_t db = sw128_desc(smem_u32(tiles + kPairStages * kTileA + st * kHalfB));
#pragma unroll
                    for (int k = 0; k < kBK / kUK; ++k)
                        mma_bf16_pair(d_tmem, da + 2 * k, db + 2 * k, (kb | k) != 0 ? 1u : 0u);
                    mma_commit_pair_both(&s.empty[st]);  // both CTAs' stage is free once read
                    if (++st == kPairStages) {
                        st = 0;
                        ph ^= 1;
                    }
                }
                if (!ok) break;
                mma_commit_pair_both(&s.tfull[acc]);
            }
            if (issued) {  // nothing of ours in flight when tensor memory is released
                mma_commit_pair_local(&s.drain);
                if (!mbar_wait_bounded(&s.drain, 0)) ok = false;
            }
        }
    } else {  // epilogue (both CTAs): warp w reads TMEM lanes 32 (w % 4) .. + 31
        const int q = warp & 3;
        unsigned char* const stage = tiles + (size_t)kPairStages * (kTileA + kHalfB) + kPairBarsBytes +
                                     (size_t)(warp - 2) * kStageWarpBytes;
        const uint32_t tempty0 = peer_smem(smem_u32(&s.tempty[0]), 0);
        const uint32_t tempty1 = peer_smem(smem_u32(&s.tempty[1]), 0);
        int i = 0;
        for (long long t = cluster; t < n_tiles; t += n_clusters, ++i) {
            const int acc = i & 1;
            const int m0 = (int)(2 * (t % mp) + rank) * kBM, n0 = (int)(t / mp) * kBN;
            ok = __all_sync(0xffffffffu, mbar_wait_bounded(&s.tfull[acc], ((uint32_t)i >> 1) & 1));
            if (!ok) break;
            tc_fence_after();
            const uint32_t taddr = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * kBN);
            const int row = m0 + q * 32 + lane;
            const unsigned long long key = epilogue_tile<EPI>(a, taddr, m0 + q * 32, n0, M, stage, lane);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_remote(acc ? tempty1 : tempty0);
            if (EPI == LM_EPI_ARGMAX && row < M) atomicMax(a.keys + row, key);
        }
    }

    if (!ok && a.device_status) atomicOr(a.device_status, SDV_DEV_TIMEOUT);
    // neither CTA leaves (or releases tensor memory) while the other may
    // still signal its barriers or the MMAs may write its tensor memory
    tc_fence_before();
    cluster_sync();
    tc_fence_after();
    if (warp == 1) tmem_dealloc_pair(tmem, kTmemCols);
}

// ------------------------------------------------------------------------
// trie nodes of the fused greedy call

__global__ void __launch_bounds__(512) lm_rows_kernel(Problem pb, LmRows r)
{
    const int b = blockIdx.x;
    if (pb.ws.req[b] & (SDV_REQ_BAD_LENGTH | SDV_REQ_BAD_TOKEN)) return;
    const int K = pb.K, L = pb.L;
    const int Lb = pb.lengths ? pb.lengths[b] : L;
    const int n = K * (r.leaves ? Lb + 1 : Lb);  // slots of depths 0..L_b - 1 (and L_b), depth-major
    const size_t s0 = (size_t)b * (L + 1) * K;
    __shared__ short local[SDV_MAX_K * (SDV_MAX_L + 1)];
    __shared__ int cnt, base;
    if (threadIdx.x == 0) cnt = 0;
    __syncthreads();
    for (int i = threadIdx.x; i < n; i += blockDim.x)
        local[i] = pb.ws.owner[s0 + i] == i % K ? (short)atomicAdd(&cnt, 1) : (short)-1;
    __syncthreads();
    if (threadIdx.x == 0) base = atomicAdd(r.count, cnt);
    __syncthreads();
    const int c0 = base;
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
        if (local[i] < 0) continue;
        r.compact[s0 + i] = c0 + local[i];
        r.keys[c0 + local[i]] = 0ull;
        if (r.row_of) r.row_of[c0 + local[i]] = (b * K + i % K) * (L + 1) + i / K;
    }
    // copy the nodes' hidden rows: 16 bytes per thread and load, four loads
    // in flight per thread
    constexpr int U = 4;
    const int units = r.d / 8;
    const int total = n * units;
    const uint4* hid = reinterpret_cast<const uint4*>(r.hidden);
    uint4* rows = reinterpret_cast<uint4*>(r.rows);
    for (int u0 = threadIdx.x; u0 < total; u0 += U * blockDim.x) {
        uint4 v[U];
#pragma unroll
        for (int q = 0; q < U; ++q) {
            const int u = u0 + q * blockDim.x;
            if (u < total && local[u / units] >= 0) {
                const int i = u / units, j = i / K, k = i % K;
                v[q] = hid[(((size_t)b * K + k) * (L + 1) + j) * units + u % units];
            }
        }
#pragma unroll
        for (int q = 0; q < U; ++q) {
            const int u = u0 + q * blockDim.x;
            if (u < total && local[u / units] >= 0)
                rows[(size_t)(c0 + local[u / units]) * units + u % units] = v[q];
        }
    }
}

__global__ void lm_argmax_kernel(Problem pb, LmRows r)
{
    const size_t slot = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int K = pb.K, L = pb.L;
    if (slot >= slot_count(pb.B, K, L)) return;
    const int k = (int)(slot % K);
    const int j = (int)((slot / K) % (L + 1));
    const int b = (int)(slot / ((size_t)K * (L + 1)));
    if (pb.ws.req[b] & (SDV_REQ_BAD_LENGTH | SDV_REQ_BAD_TOKEN)) return;
    const int Lb = pb.lengths ? pb.lengths[b] : L;
    if (j >= Lb || pb.ws.owner[slot] != k) return;
    const unsigned long long key = r.keys[r.compact[slot]];
    const float v = key_value(key);
    int am = (int)(0xffffffffu - (uint32_t)key);
    if (!(v > -INFINITY && v < INFINITY)) {  // NaN, +Inf, or no finite value
        atomicOr(&pb.ws.req[b], SDV_REQ_NONFINITE);
        if (pb.device_status) atomicOr(pb.device_status, SDV_REQ_NONFINITE);
        am = -1;
    }
    pb.ws.am[slot] = am;
}

// The end leaves the decision reached: one CTA per request copies its
// leaf's hidden row, if it has one, into the leaf block.
__global__ void __launch_bounds__(128) lm_leaf_rows_kernel(Problem pb, LmRows r)
{
    const int b = blockIdx.x;
    const int slot = pb.leaf_pending[b];
    if (slot < 0) return;
    const int K = pb.K, L = pb.L;
    const int k = slot % K, j = (slot / K) % (L + 1);
    __shared__ int c;
    if (threadIdx.x == 0) {
        c = atomicAdd(r.leaf_count, 1);
        r.leaf_req[c] = b;
        r.leaf_keys[c] = 0ull;
    }
    __syncthreads();
    const int units = r.d / 8;
    const uint4* src = reinterpret_cast<const uint4*>(r.hidden) + (((size_t)b * K + k) * (L + 1) + j) * units;
    uint4* dst = reinterpret_cast<uint4*>(r.leaf_rows) + (size_t)c * units;
    for (int e = threadIdx.x; e < units; e += blockDim.x) dst[e] = src[e];
}

// The reached leaves' tokens: the argmax, or the request made invalid when
// the leaf's logits hold NaN or +Inf (or nothing finite).
__global__ void lm_leaf_token_kernel(Problem pb, LmRows r)
{
    const int c = blockIdx.x * blockDim.x + threadIdx.x;
    if (c >= *r.leaf_count) return;
    const int b = r.leaf_req[c];
    const unsigned long long key = r.leaf_keys[c];
    const float v = key_value(key);
    if (v > -INFINITY && v < INFINITY) {
        pb.out_token[b] = (int)(0xffffffffu - (uint32_t)key);
        return;
    }
    const int n = pb.K * pb.L;
    if (pb.accept_prob)
        for (int i = 0; i < n; ++i) pb.accept_prob[(size_t)b * n + i] = 0.f;
    pb.accept_len[b] = 0;
    pb.accept_draft[b] = 0;
    pb.out_token[b] = -1;
    atomicOr(&pb.ws.req[b], SDV_REQ_NONFINITE);
    if (pb.device_status) atomicOr(pb.device_status, SDV_REQ_NONFINITE);
}

// ------------------------------------------------------------------------
// host: tensor maps

typedef CUresult (*EncodeTiled)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiled encoder()
{
    static EncodeTiled fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        fn = reinterpret_cast<EncodeTiled>(p);
    }
    return fn;
}

// [rows][d] bf16, row pitch d * 2 bytes, boxes of box_rows x 64 elements
// with the 128-byte swizzle; reads past the tensor return zeros.
bool make_map(CUtensorMap* m, const void* base, long long rows, int d, int box_rows)
{
    EncodeTiled enc = encoder();
    if (!enc) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)d, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)d * 2};
    const cuuint32_t box[2] = {(cuuint32_t)kBK, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int sm_count()
{
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) !=
                                                  cudaSuccess)
        return 0;
    return n;
}

}  // namespace

size_t lm_head_smem_bytes() { return kLmSmem > kPairSmem ? kLmSmem : kPairSmem; }

int g_lm_single_cta = 0;

namespace {

template <int EPI>
cudaError_t launch_single(const CUtensorMap& ma, const CUtensorMap& mb, const LmArgs& a, long long grid,
                          cudaStream_t st)
{
    const cudaError_t e =
        cudaFuncSetAttribute(lm_head_kernel<EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kLmSmem);
    if (e != cudaSuccess) return e;
    lm_head_kernel<EPI><<<(unsigned)grid, kLmThreads, kLmSmem, st>>>(ma, mb, a);
    return cudaGetLastError();
}

// The pair form, with as many clusters as fit on the device at once (at
// most `max_clusters`).  cudaErrorNotSupported: no cluster of two fits.
// The number that fits is asked once per device and form.
template <int EPI>
cudaError_t launch_pair(const CUtensorMap& ma, const CUtensorMap& mb, const LmArgs& a, long long max_clusters,
                        cudaStream_t st)
{
    constexpr int kDevs = 64;
    static int fits[kDevs];  // 0: not asked yet; -1: none fits
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(lm_head_pair_kernel<EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kPairSmem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cfg.blockDim = dim3(kLmThreads);
    cfg.dynamicSmemBytes = kPairSmem;
    cfg.stream = st;
    int fit = dev >= 0 && dev < kDevs ? fits[dev] : 0;
    if (fit == 0) {
        cfg.gridDim = dim3(2);
        e = cudaOccupancyMaxActiveClusters(&fit, lm_head_pair_kernel<EPI>, &cfg);
        if (e != cudaSuccess) return e;
        if (fit <= 0) fit = -1;
        if (dev >= 0 && dev < kDevs) fits[dev] = fit;
    }
    if (fit < 0) return cudaErrorNotSupported;
    const long long clusters = max_clusters < fit ? max_clusters : fit;
    cfg.gridDim = dim3(2 * (unsigned)clusters);
    return cudaLaunchKernelEx(&cfg, lm_head_pair_kernel<EPI>, ma, mb, a);
}

template <int EPI>
cudaError_t launch_epi(const void* hidden, long long hidden_rows, const void* lm_head, const LmArgs& a,
                       cudaStream_t st)
{
    const int n_sm = sm_count();
    if (n_sm <= 0) return cudaErrorInvalidDevice;
    long long row_tiles = -1;  // unknown when the row count is on the device
    if (!a.rows_dev) {
        row_tiles = (a.rows + kBM - 1) / kBM;
        if (row_tiles == 0 || a.V <= 0) return cudaSuccess;
    }
    const long long col_tiles = (a.V + kBN - 1) / kBN;
    if (!g_lm_single_cta) {
        CUtensorMap ma, mb;
        if (!make_map(&ma, hidden, hidden_rows, a.d, kBM) || !make_map(&mb, lm_head, a.V, a.d, kBN / 2))
            return cudaErrorInvalidValue;
        long long clusters = n_sm / 2;
        if (row_tiles >= 0) {
            const long long pair_tiles = (row_tiles + 1) / 2 * col_tiles;
            clusters = clusters < pair_tiles ? clusters : pair_tiles;
        }
        const cudaError_t e = launch_pair<EPI>(ma, mb, a, clusters, st);
        if (e != cudaErrorNotSupported) return e;
        cudaGetLastError();
    }
    CUtensorMap ma, mb;
    if (!make_map(&ma, hidden, hidden_rows, a.d, kBM) || !make_map(&mb, lm_head, a.V, a.d, kBN))
        return cudaErrorInvalidValue;
    long long grid = n_sm;
    if (row_tiles >= 0) grid = grid < row_tiles * col_tiles ? grid : row_tiles * col_tiles;
    return launch_single<EPI>(ma, mb, a, grid, st);
}

}  // namespace

cudaError_t launch_lm_head(const void* hidden, long long hidden_rows, const void* lm_head, const LmArgs& a,
                           int epi, cudaStream_t st)
{
    if (epi == LM_EPI_ROWS_BF16) return launch_epi<LM_EPI_ROWS_BF16>(hidden, hidden_rows, lm_head, a, st);
    if (epi == LM_EPI_ARGMAX) return launch_epi<LM_EPI_ARGMAX>(hidden, hidden_rows, lm_head, a, st);
    return launch_epi<LM_EPI_LOGITS>(hidden, hidden_rows, lm_head, a, st);
}

cudaError_t launch_lm_rows(const Problem& pb, const LmRows& r, cudaStream_t st)
{
    lm_rows_kernel<<<pb.B, 512, 0, st>>>(pb, r);
    return cudaGetLastError();
}

cudaError_t launch_lm_leaf_rows(const Problem& pb, const LmRows& r, cudaStream_t st)
{
    lm_leaf_rows_kernel<<<pb.B, 128, 0, st>>>(pb, r);
    return cudaGetLastError();
}

cudaError_t launch_lm_leaf_token(const Problem& pb, const LmRows& r, cudaStream_t st)
{
    lm_leaf_token_kernel<<<(pb.B + 127) / 128, 128, 0, st>>>(pb, r);
    return cudaGetLastError();
}

cudaError_t launch_lm_argmax(const Problem& pb, const LmRows& r, cudaStream_t st)
{
    const size_t n = slot_count(pb.B, pb.K, pb.L);
    if (n == 0) return cudaSuccess;
    lm_argmax_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(pb, r);
    return cudaGetLastError();
}

}  // namespace sdv
