// sdv_device.cuh -- device helpers shared by the verification kernels:
// inline PTX (ex2, NaN-propagating max, mbarrier waits), element unpacking
// of 16-byte units, warp reductions.
#pragma once

#include <cstdint>

#include "sdv_internal.h"

namespace sdv {
namespace {

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

// Packed pairs of fp32 (f32x2): one instruction for two independent FMAs,
// adds or multiplies, each lane rounded as its scalar form.
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c)
{
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
        "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}

__device__ __forceinline__ float2 fadd2(float2 a, float2 b)
{
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}

__device__ __forceinline__ float2 fmul2(float2 a, float2 b)
{
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "mul.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
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

// Waits for phase `phase` of the barrier for at most limit_ns; once a wait
// of the caller has run out (gave_up), only one try is made.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t phase, uint64_t limit_ns = kWaitNs,
                                                  bool gave_up = false)
{
    if (mbar_try_wait(bar, phase)) return true;  // the common case reads no clock
    if (gave_up) return false;
    const uint64_t t0 = globaltimer();
    while (!mbar_try_wait(bar, phase)) {
        if (globaltimer() - t0 > limit_ns) return false;
    }
    return true;
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
    // maximum over two whole units (a balanced tree)
    __device__ static __forceinline__ float pair_max(const uint4& a, const uint4& b)
    {
        const float p = max_nan(max_nan(__uint_as_float(a.x), __uint_as_float(a.y)),
                                max_nan(__uint_as_float(a.z), __uint_as_float(a.w)));
        const float q = max_nan(max_nan(__uint_as_float(b.x), __uint_as_float(b.y)),
                                max_nan(__uint_as_float(b.z), __uint_as_float(b.w)));
        return max_nan(p, q);
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
    // maximum over two whole units: packed pairs first, one unpack at the end
    __device__ static __forceinline__ float pair_max(const uint4& a, const uint4& b)
    {
        const uint32_t p = max_nan_bf16x2(max_nan_bf16x2(a.x, a.y), max_nan_bf16x2(a.z, a.w));
        const uint32_t q = max_nan_bf16x2(max_nan_bf16x2(b.x, b.y), max_nan_bf16x2(b.z, b.w));
        const uint32_t r = max_nan_bf16x2(p, q);
        return max_nan(bf_lo(r), bf_hi(r));
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

// Warp-wide maximum in one instruction; NaN in any lane gives NaN.
__device__ __forceinline__ float warp_max_redux(float v)
{
    float r;
    asm volatile("redux.sync.max.NaN.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
    return r;
}

}  // namespace
}  // namespace sdv
