// Inline-PTX helpers for sm_103a: shared-memory mbarriers, bulk async copies
// (TMA engine, non-tensor form), legacy warp MMA, programmatic dependent launch
// and bounded waits.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace tfq {

__device__ __forceinline__ uint32_t smem_u32(const void* p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- mbarrier

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Non-blocking test of the phase with parity `parity`.
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Device-scope fetch-and-add with acquire-release semantics: the caller's earlier
// writes (and those ordered before them by a warp or CTA barrier) are visible to
// whoever reads the counter after it, and the caller sees the writes released by
// the earlier adders.
__device__ __forceinline__ unsigned atom_add_acq_rel_gpu(unsigned* ptr, unsigned v)
{
    unsigned old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(ptr), "r"(v) : "memory");
    return old;
}

__device__ __forceinline__ uint64_t globaltimer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Wait for the phase of `bar` with parity `parity`, giving up after about
// `limit_ns` nanoseconds (counted in SM cycles at 2 per ns). Returns false on time-out.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, uint64_t limit_ns)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const long long start = clock64();
    const long long limit = (long long)(limit_ns * 2);  // 2 cycles per ns
    while (true) {
        if (mbar_try_wait(bar, parity))
            return true;
        if (clock64() - start > limit)
            return false;
    }
}

// ---------------------------------------------------------------- bulk copy

// Global -> shared bulk copy through the TMA engine; completion is signalled as
// transaction bytes on `bar`. dst, src 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                         uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// Same, without a cache-policy hint.
__device__ __forceinline__ void bulk_g2s_plain(void* dst, const void* src, uint32_t bytes, uint64_t* bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_u32(dst)),
                 "l"(src), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// 16 bytes of read-only global memory through the non-coherent path, issued where it
// stands: the asm is volatile, so the load keeps its place among the other volatile asm
// (a grid-dependency wait, a barrier) instead of sinking to its first use.
__device__ __forceinline__ uint4 ld_nc_v4_here(const void* ptr)
{
    uint4 r;
    asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(ptr));
    return r;
}

// ---------------------------------------------------------------- PDL

__device__ __forceinline__ void pdl_wait()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void pdl_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------- named barriers

__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t nthreads)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ---------------------------------------------------------------- warp MMA

// D[16x8] (+)= A[16x16] * B[16x8], bf16 inputs, fp32 accumulation.
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1)
{
    // not volatile: the compiler may interleave independent MMAs of different tiles
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// The same with fp16 inputs.
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                              uint32_t b0, uint32_t b1)
{
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// (a & b) | c in one LOP3.
__device__ __forceinline__ uint32_t lop3_and_or(uint32_t a, uint32_t b, uint32_t c)
{
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// Two 4-bit codes (bits 0-3 and 16-19 of w) as the bf16 pair (128 + lo, 128 + hi):
// 0x43 is the bf16 exponent of 128, whose unit in the last place is 1, so a
// code in the low mantissa bits adds exactly its value.
__device__ __forceinline__ uint32_t nib2_bf16(uint32_t w)
{
    return lop3_and_or(w, 0x000F000Fu, 0x43004300u);
}

// fp16 has 10 mantissa bits and 0x64 is the exponent of 1024 (unit in the last place
// 1): the codes in bits 0-3 / 16-19 become the pair (1024 + lo, 1024 + hi) and those in
// bits 4-7 / 20-23 the pair (1024 + 16 lo, 1024 + 16 hi), one LOP3 each, no shift.
__device__ __forceinline__ uint32_t nib2_f16(uint32_t w) { return lop3_and_or(w, 0x000F000Fu, 0x64006400u); }
__device__ __forceinline__ uint32_t nib2_f16_x16(uint32_t w) { return lop3_and_or(w, 0x00F000F0u, 0x64006400u); }

__device__ __forceinline__ float bf16lo_f32(uint32_t pair) { return __uint_as_float(pair << 16); }
__device__ __forceinline__ float bf16hi_f32(uint32_t pair) { return __uint_as_float(pair & 0xFFFF0000u); }

__device__ __forceinline__ uint32_t f32x2_to_bf16x2(float lo, float hi)
{
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

// A bf16 pair as an fp16 pair (exact for |v| < 65536, apart from fp16 subnormals).
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t pair)
{
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(bf16hi_f32(pair)), "f"(bf16lo_f32(pair)));
    return r;
}

// ---------------------------------------------------------------- NVFP4 conversions

// The four bytes of w, each two E2M1 codes (low nibble first), as four fp16 pairs:
// r0 from byte 0 ... r3 from byte 3, the low nibble in the low half. Exact: every
// E2M1 value (0, +-0.5 ... +-6) is an fp16 value.
__device__ __forceinline__ void e2m1x8_to_f16x2(uint32_t w, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3)
{
    asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %4;\n"
        " cvt.rn.f16x2.e2m1x2 %0, b0;\n cvt.rn.f16x2.e2m1x2 %1, b1;\n"
        " cvt.rn.f16x2.e2m1x2 %2, b2;\n cvt.rn.f16x2.e2m1x2 %3, b3;\n}"
        : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
        : "r"(w));
}

// Bits 0-15 of v, two E4M3 bytes, as an fp16 pair (low byte in the low half). Exact:
// every finite E4M3 value is an fp16 value.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t v)
{
    uint32_t d;
    const unsigned short h = (unsigned short)(v & 0xFFFFu);
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(d) : "h"(h));
    return d;
}

// a * (low half of s, twice) and a * (high half of s, twice), fp16 pairs.
__device__ __forceinline__ uint32_t hmul2_lo(uint32_t a, uint32_t s)
{
    const __half2 r = __hmul2(*reinterpret_cast<const __half2*>(&a), __low2half2(*reinterpret_cast<const __half2*>(&s)));
    return *reinterpret_cast<const uint32_t*>(&r);
}
__device__ __forceinline__ uint32_t hmul2_hi(uint32_t a, uint32_t s)
{
    const __half2 r = __hmul2(*reinterpret_cast<const __half2*>(&a), __high2half2(*reinterpret_cast<const __half2*>(&s)));
    return *reinterpret_cast<const uint32_t*>(&r);
}

// An fp16 pair as a bf16 pair, rounded to nearest even (exact when the values have
// at most 8 significant bits and lie in bf16's normal range).
__device__ __forceinline__ uint32_t f16x2_to_bf16x2(uint32_t a)
{
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&a));
    return f32x2_to_bf16x2(f.x, f.y);
}

}  // namespace tfq
