// pmqa_mla_ptx.cuh -- inline-PTX wrappers used by the sparse MLA decode on top
// of pmqa_ptx.cuh: TMEM stores, non-blocking mbarrier tests, descriptors with
// other strides and swizzles (MN-major, 64-byte), cp.async with mbarrier
// arrival, ex2 and fp8 packing.
#pragma once

#include <cuda_fp16.h>

#include <cstdint>

#include "pmqa_ptx.cuh"

namespace pmqa {

// 32 consecutive TMEM columns of this thread's lane from registers (32x32b
// shape, x32); tmem_st_wait orders them before later tcgen05 work.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t *r)
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
        "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
        "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

__device__ __forceinline__ void tmem_st_wait()
{
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Non-blocking test of an mbarrier phase (never suspends the thread).
__device__ __forceinline__ bool mbar_test(uint64_t *bar, uint32_t parity)
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

// Shared-memory matrix descriptor, 128-byte swizzle, K-major, with groups of
// 8 rows `sbo` bytes apart (a multiple of 1024; the group base 1024-aligned).
__device__ __forceinline__ uint64_t sw128_kmajor_desc_sbo(uint32_t smem_addr, uint32_t sbo)
{
    uint64_t d = 0;
    d |= (uint64_t)((smem_addr & 0x3FFFFu) >> 4);
    d |= (uint64_t)1u << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1u << 46;
    d |= (uint64_t)2u << 61;
    return d;
}

// Shared-memory matrix descriptor, 64-byte swizzle, K-major: rows of 64
// bytes, 16-byte chunk c of row r at chunk c ^ ((r >> 1) & 3), groups of 8 rows
// (512-byte atoms, 512-byte aligned) `sbo` bytes apart; swizzle mode 4 = 64B.
__device__ __forceinline__ uint64_t sw64_kmajor_desc(uint32_t smem_addr, uint32_t sbo)
{
    uint64_t d = 0;
    d |= (uint64_t)((smem_addr & 0x3FFFFu) >> 4);
    d |= (uint64_t)1u << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1u << 46;
    d |= (uint64_t)4u << 61;
    return d;
}

// Shared-memory matrix descriptor for an MN-major operand in the 128-byte
// swizzle: rows of 128 bytes run along M (or N), one row per K index, 16-byte
// chunk c of row k at chunk c ^ (k & 7); groups of 8 K rows are `sbo` bytes
// apart and 128-element blocks along M are `lbo` bytes apart. The same bytes
// are the K-major operand whose rows are the K indices, so a tile stored for
// one product serves as the transposed operand of another.
__device__ __forceinline__ uint64_t sw128_mnmajor_desc(uint32_t smem_addr, uint32_t lbo,
                                                       uint32_t sbo)
{
    uint64_t d = 0;
    d |= (uint64_t)((smem_addr & 0x3FFFFu) >> 4);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1u << 46;
    d |= (uint64_t)2u << 61;
    return d;
}

// Bit 15 of the kind::f8f6f4 instruction descriptor: A is MN-major.
constexpr uint32_t kIdescAMnMajor = 1u << 15;

// 16-byte asynchronous copy that reads src_bytes (0 or 16) bytes of src and
// zero-fills the rest.
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void *src, uint32_t src_bytes)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
                 "r"(src_bytes)
                 : "memory");
}

// Arrive on the mbarrier once every cp.async this thread issued so far has
// landed (the arrival counts toward the barrier's expected count).
__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t *bar)
{
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

// 2^x, the hardware approximation (relative error about 2^-22; 2^-inf = 0).
__device__ __forceinline__ float ex2_approx(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// (lo, hi) -> two e4m3 bytes, round to nearest even, saturating: lo in bits
// 0-7, hi in bits 8-15.
__device__ __forceinline__ uint32_t f32x2_to_e4m3x2(float lo, float hi)
{
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// Two e4m3 bytes (bits 0-7, 8-15) -> their exact values.
__device__ __forceinline__ void e4m3x2_to_f32x2(uint32_t b, float &lo, float &hi)
{
    uint32_t h2;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"((uint16_t)b));
    lo = __half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFFu)));
    hi = __half2float(__ushort_as_half((unsigned short)(h2 >> 16)));
}

// Named barrier that also returns whether `pred` held in any participating
// thread.
__device__ __forceinline__ bool named_bar_or(uint32_t id, uint32_t count, bool pred)
{
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %3, 0;\n\t"
        "bar.red.or.pred q, %1, %2, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(id), "r"(count), "r"(pred ? 1u : 0u)
        : "memory");
    return r != 0;
}

}  // namespace pmqa
