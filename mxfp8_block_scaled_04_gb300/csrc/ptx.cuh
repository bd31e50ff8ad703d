// Inline-PTX building blocks for sm_103a: mbarriers, 2-D TMA tile loads,
// programmatic dependent launch, packed 16-bit max, packed f32x2 arithmetic,
// FP8x2 conversion.  Every wait here is bounded.
#pragma once

#include <cstdint>
#include <cuda.h>

namespace mxfp8 {

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Make mbarrier initialisation visible to the async (TMA) proxy.
__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Order this thread's generic-proxy shared-memory accesses before later
// async-proxy (TMA) accesses of the same shared memory.
__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait_parity(uint32_t bar, uint32_t parity)
{
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.b32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0;
}

__device__ __forceinline__ uint64_t globaltimer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Wait for the mbarrier phase with the given parity to complete; gives up
// after limit_ns nanoseconds of wall time and returns false.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, uint64_t limit_ns)
{
    if (mbar_try_wait_parity(bar, parity))
        return true;
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait_parity(bar, parity)) {
        if (globaltimer_ns() - t0 > limit_ns)
            return false;
    }
    return true;
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap *map)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Programmatic dependent launch.  The library's kernels are launched so that the
// next kernel on the stream may start while this one drains: each lets its
// successor launch at once, and waits, before its first global memory access,
// until the kernel before it has finished and its writes are visible.  Without
// the launch attribute both are no-ops.
__device__ __forceinline__ void pdl_wait_and_release()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// 2-D tiled TMA load of one box into shared memory; completion is signalled
// as transaction bytes on `bar`.  x is the innermost (column) coordinate.  The
// input is read exactly once, so its lines are marked evict-first in L2, which
// leaves L2 to the outputs being written (measured 1.2% faster on GB300).
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, uint32_t bar,
                                            int32_t x, int32_t y)
{
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar), "l"(pol)
        : "memory");
}

// Lane-wise unsigned max of two packed 16-bit halves.
__device__ __forceinline__ uint32_t max_u16x2(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("max.u16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// Two fp32 -> two FP8 codes, round to nearest even, finite values saturate.
// Returns lo's code in bits 0..7 and hi's in bits 8..15.
template <int FMT>
__device__ __forceinline__ uint32_t cvt_fp8x2(float lo, float hi)
{
    uint16_t r;
    if constexpr (FMT == 0)
        asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    else
        asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// Shared-memory vector loads (plain C++ loads: the compiler sees the shared
// address space and is free to schedule them).
__device__ __forceinline__ uint4 lds128(const void *p) { return *reinterpret_cast<const uint4 *>(p); }
__device__ __forceinline__ uint2 lds64(const void *p) { return *reinterpret_cast<const uint2 *>(p); }
__device__ __forceinline__ float4 lds128f(const void *p) { return *reinterpret_cast<const float4 *>(p); }
__device__ __forceinline__ void sts64(void *p, uint32_t a, uint32_t b) { *reinterpret_cast<uint2 *>(p) = make_uint2(a, b); }

// 16-byte global store that does not allocate in L1.
__device__ __forceinline__ void stg128(void *p, uint32_t a, uint32_t b, uint32_t c, uint32_t d)
{
    asm volatile("st.global.L1::no_allocate.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(a), "r"(b), "r"(c),
                 "r"(d)
                 : "memory");
}

// 8-byte global store that does not allocate in L1.
__device__ __forceinline__ void stg64(void *p, uint32_t a, uint32_t b)
{
    asm volatile("st.global.L1::no_allocate.v2.u32 [%0], {%1, %2};" ::"l"(p), "r"(a), "r"(b) : "memory");
}

// The 16 FP8 codes of one row segment, stored at p.  Rows are 16-byte aligned when
// N % 16 == 0 (one 16-byte store); when N % 16 == 8 they are only 8-byte aligned
// (two 8-byte stores), and the row's last segment holds 8 columns (first half only).
__device__ __forceinline__ void store_codes(uint8_t *p, uint32_t o0, uint32_t o1, uint32_t o2, uint32_t o3,
                                            bool rows16, bool half)
{
    if (rows16) {
        stg128(p, o0, o1, o2, o3);
    } else {
        stg64(p, o0, o1);
        if (!half)
            stg64(p + 8, o2, o3);
    }
}

// BF16 halves of a packed word, widened exactly to fp32.
// Two fp32 values in one 64-bit register pair, for Blackwell's packed
// add / mul / fma.rn.f32x2 (each lane rounds exactly as the scalar operation).
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi)
{
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float &lo, float &hi)
{
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_splat(float a) { return f2_pack(a, a); }
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b)
{
    uint64_t r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b)
{
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c)
{
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}

// cvt_fp8x2 of (v0 * m.lo, v1 * m.hi), the two products as one f32x2 multiply.
template <int FMT>
__device__ __forceinline__ uint32_t cvt_fp8x2_scaled(float v0, float v1, uint64_t m)
{
    float a, b;
    f2_unpack(f2_mul(f2_pack(v0, v1), m), a, b);
    return cvt_fp8x2<FMT>(a, b);
}

// Lane-wise signed maximum of two BF16 pairs (the larger BF16 value, exactly).
__device__ __forceinline__ uint32_t max_bf16x2(uint32_t a, uint32_t b)
{
    uint32_t r;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// Lane-wise BF16 pair whose magnitude is max(|a|, |b|) (its sign is the xor of
// the two signs: callers keep only the magnitude bits, & 0x7FFF per lane).
__device__ __forceinline__ uint32_t absmax_bf16x2(uint32_t a, uint32_t b)
{
    uint32_t r;
    asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// acc + (the low / high BF16 of w), one mixed-precision add (the BF16 operand
// widens exactly, the sum rounds to nearest as an fp32 add).
__device__ __forceinline__ float add_bf16_lo(float acc, uint32_t w)
{
    float r;
    asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\tadd.rn.f32.bf16 %0, lo, %1;\n\t}"
        : "=f"(r) : "f"(acc), "r"(w));
    return r;
}
__device__ __forceinline__ float add_bf16_hi(float acc, uint32_t w)
{
    float r;
    asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\tadd.rn.f32.bf16 %0, hi, %1;\n\t}"
        : "=f"(r) : "f"(acc), "r"(w));
    return r;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

}  // namespace mxfp8
