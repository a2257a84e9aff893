// pmqa_ptx.cuh -- thin inline-PTX wrappers for sm_103a: mbarrier, cp.async,
// tcgen05 (TMEM allocation, MMA, commit, loads) and a few cache/proxy fences.
// Every spin on an mbarrier is bounded in time; on expiry the caller records a
// status bit and unwinds instead of hanging the GPU.
#pragma once

#include <cstdint>

namespace pmqa {

// Limit for any single wait on an mbarrier. The longest legitimate wait is a
// few tens of microseconds (a top-k merge running on the consumer side).
constexpr uint64_t kWaitLimitNs = 200ull * 1000 * 1000;

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---------------------------------------------------------------- mbarrier

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void mbar_init_fence()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity)
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

// try_wait with a suspend-time hint: the thread sleeps until the phase
// completes or about `hint_ns` pass, instead of returning at once to spin.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t *bar, uint32_t parity, uint32_t hint_ns)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
}

// Wait for the phase with the given parity to complete. Returns false if the
// CTA-wide abort flag (when given) was raised or the time limit passed. A
// waiting warp sleeps in the barrier unit rather than spinning, so it takes
// no issue slots from the warps that do the work.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity,
                                          const volatile int *abort_flag)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const uint64_t t0 = global_timer_ns();
    for (;;) {
        // a few sleeps between the checks of the abort flag and the clock
#pragma unroll 1
        for (int k = 0; k < 8; ++k)
            if (mbar_try_wait_sleep(bar, parity, 100000u))
                return true;
        if (abort_flag != nullptr && *abort_flag)
            return false;
        if (global_timer_ns() - t0 > kWaitLimitNs)
            return false;
    }
}

// ---------------------------------------------------------------- shared memory

// Explicit shared-memory accesses by 32-bit shared address. Volatile: they keep
// their order against the barrier, copy-wait and tcgen05 statements around
// them.
__device__ __forceinline__ uint4 lds128(uint32_t addr)
{
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr));
    return v;
}

__device__ __forceinline__ uint32_t lds32(uint32_t addr)
{
    uint32_t v;
    asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}

// Non-volatile: for data that stays fixed while it is read (the weights of a
// request). The compiler may schedule these loads freely between the
// statements that order them: derive the address from launder_u32 after the
// wait that makes the data valid.
__device__ __forceinline__ float4 lds128f_nv(uint32_t addr)
{
    float4 v;
    asm("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr));
    return v;
}

// An opaque copy of x, produced in program order among the volatile statements.
__device__ __forceinline__ uint32_t launder_u32(uint32_t x)
{
    uint32_t y;
    asm volatile("mov.b32 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

__device__ __forceinline__ void sts128(uint32_t addr, uint32_t x, uint32_t y, uint32_t z, uint32_t w)
{
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(x), "r"(y), "r"(z), "r"(w)
                 : "memory");
}

// ---------------------------------------------------------------- cp.async

__device__ __forceinline__ uint64_t l2_evict_first_policy()
{
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

__device__ __forceinline__ uint64_t l2_evict_normal_policy()
{
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

__device__ __forceinline__ uint64_t l2_evict_last_policy()
{
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// 16-byte asynchronous copy that reads only the first src_bytes (1..16) bytes of
// src and zero-fills the rest of the 16-byte destination.
__device__ __forceinline__ void cp_async_16_zfill(uint32_t dst, const void *src, uint32_t src_bytes,
                                                  uint64_t policy)
{
    asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2, %3;" ::"r"(dst),
                 "l"(src), "r"(src_bytes), "l"(policy)
                 : "memory");
}

// (a0, a1) += (w0, w1) * (x0, x1): one packed fp32x2 fused multiply-add.
__device__ __forceinline__ void ffma2(float &a0, float &a1, float w0, float w1, float x0, float x1)
{
    asm("{\n\t.reg .b64 ra, rw, rx;\n\t"
        "mov.b64 ra, {%0, %1};\n\t"
        "mov.b64 rw, {%2, %3};\n\t"
        "mov.b64 rx, {%4, %5};\n\t"
        "fma.rn.f32x2 ra, rw, rx, ra;\n\t"
        "mov.b64 {%0, %1}, ra;\n\t}"
        : "+f"(a0), "+f"(a1)
        : "f"(w0), "f"(w1), "f"(x0), "f"(x1));
}

// (a0, a1) = (w0, w1) * (x0, x1): one packed fp32x2 multiply.
__device__ __forceinline__ void fmul2(float &a0, float &a1, float w0, float w1, float x0, float x1)
{
    asm("{\n\t.reg .b64 ra, rw, rx;\n\t"
        "mov.b64 rw, {%2, %3};\n\t"
        "mov.b64 rx, {%4, %5};\n\t"
        "mul.rn.f32x2 ra, rw, rx;\n\t"
        "mov.b64 {%0, %1}, ra;\n\t}"
        : "=f"(a0), "=f"(a1)
        : "f"(w0), "f"(w1), "f"(x0), "f"(x1));
}

// (a0, a1) += (b0, b1): one packed fp32x2 add.
__device__ __forceinline__ void fadd2(float &a0, float &a1, float b0, float b1)
{
    asm("{\n\t.reg .b64 ra, rb;\n\t"
        "mov.b64 ra, {%0, %1};\n\t"
        "mov.b64 rb, {%2, %3};\n\t"
        "add.rn.f32x2 ra, ra, rb;\n\t"
        "mov.b64 {%0, %1}, ra;\n\t}"
        : "+f"(a0), "+f"(a1)
        : "f"(b0), "f"(b1));
}

// Programmatic dependent launch: let the next kernel of the stream start
// launching (its CTAs still wait in griddep_wait until this grid is done).
__device__ __forceinline__ void griddep_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Wait until every grid this one depends on has completed and its memory
// operations are visible; returns at once when launched without a dependency.
__device__ __forceinline__ void griddep_wait()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// ---------------------------------------------------------------- TMA

// Expect `bytes` more transaction bytes on the barrier and arrive once.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

// 2-D tiled tensor load (box given by the tensor map) into shared memory,
// completion signalled as transaction bytes on `bar`. x is the innermost
// coordinate (bytes for a uint8 map) and must keep the 16-byte rule.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void *tmap, int x, int y,
                                            uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, "
        "{%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

// 1-D bulk copy global -> shared; addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes,
                                          uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            dst),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// Global store with an L2 eviction-priority hint.
__device__ __forceinline__ void st_global_hint(float *p, float v, uint64_t policy)
{
    asm volatile("st.global.L2::cache_hint.f32 [%0], %1, %2;" ::"l"(p), "f"(v), "l"(policy)
                 : "memory");
}

__device__ __forceinline__ void cp_async_commit()
{
    asm volatile("cp.async.commit_group;" ::: "memory");
}

template <int N>
__device__ __forceinline__ void cp_async_wait_group()
{
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void cp_async_wait_all()
{
    asm volatile("cp.async.wait_all;" ::: "memory");
}

// Make this thread's completed generic-proxy writes to shared memory visible
// to later async-proxy reads (the tensor core reading MMA operands).
__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------- tcgen05

// Shared-memory matrix descriptor for a K-major operand stored as 128-byte rows
// with the 128-byte swizzle: 16-byte chunk c of row r sits at chunk c ^ (r & 7),
// groups of 8 rows are 1024 bytes apart. Fields: start address >> 4 (bits 0-13),
// leading-dimension offset (unused for this layout, 16 B), stride-dimension
// offset 1024 B >> 4 (bits 32-45), descriptor version 1 (bits 46-47), swizzle
// mode 2 = 128B (bits 61-63). The tile base must be 1024-byte aligned.
__device__ __forceinline__ uint64_t sw128_kmajor_desc(uint32_t smem_addr)
{
    uint64_t d = 0;
    d |= (uint64_t)((smem_addr & 0x3FFFFu) >> 4);
    d |= (uint64_t)1u << 16;
    d |= (uint64_t)(1024u >> 4) << 32;
    d |= (uint64_t)1u << 46;
    d |= (uint64_t)2u << 61;
    return d;
}

// Instruction descriptor, kind::f8f6f4: D fp32 (bits 4-5 = 1), A and B e4m3
// (bits 7-9, 10-12 = 0), both K-major (bits 15, 16 = 0), N >> 3 in bits 17-22,
// M >> 4 in bits 24-28.
__host__ __device__ constexpr uint32_t idesc_e4m3_f32(int m, int n)
{
    return (1u << 4) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

__device__ __forceinline__ void tmem_alloc(uint32_t *dst_smem, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, one CTA, fp8 e4m3 inputs, fp32 accumulate.
__device__ __forceinline__ void umma_e4m3(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                          uint32_t idesc, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive once on the mbarrier when all tcgen05 operations issued so far by this
// thread have completed.
__device__ __forceinline__ void umma_commit(uint64_t *bar)
{
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void tc_fence_before_sync()
{
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after_sync()
{
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Each thread of the warp reads 16 consecutive 32-bit columns of its own TMEM
// lane (lane = 32 * (warp % 4) + lane id, folded into taddr by the caller).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t *r)
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}

// No memory clobber: the wait orders TMEM loads only (their destination
// registers are tied to it through reg_fence16), and shared/global loads that
// do not depend on it may still be scheduled across it.
__device__ __forceinline__ void tmem_ld_wait()
{
    asm volatile("tcgen05.wait::ld.sync.aligned;");
}

// Register a dependency of r on the preceding tcgen05.wait::ld.
__device__ __forceinline__ void reg_fence16(uint32_t *r)
{
    asm volatile(""
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                   "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                   "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]));
}

// 32 consecutive TMEM columns of this thread's lane (32x32b shape, x32).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t *r)
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr));
}

// NC (16 or 32) consecutive TMEM columns of this thread's lane, and the
// matching register fence after tmem_ld_wait.
template <int NC>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, uint32_t (&r)[NC])
{
    static_assert(NC == 16 || NC == 32, "16 or 32 columns");
    if constexpr (NC == 16)
        tmem_ld16(taddr, r);
    else
        tmem_ld32(taddr, r);
}

template <int NC>
__device__ __forceinline__ void reg_fence_cols(uint32_t (&r)[NC])
{
    reg_fence16(r);
    if constexpr (NC == 32)
        reg_fence16(r + 16);
}

// Named barrier over `count` threads (a multiple of 32).
__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t count)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Named barrier that also returns whether `pred` held in every participating
// thread.
__device__ __forceinline__ bool named_bar_and(uint32_t id, uint32_t count, bool pred)
{
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %3, 0;\n\t"
        "bar.red.and.pred q, %1, %2, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(id), "r"(count), "r"(pred ? 1u : 0u)
        : "memory");
    return r != 0;
}

}  // namespace pmqa
