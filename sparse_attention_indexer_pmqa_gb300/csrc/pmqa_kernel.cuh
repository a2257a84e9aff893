// pmqa_kernel.cuh -- the persistent FP8 paged MQA-logits kernel (the KV pass
// of pmqa_main.cuh): prologue, schedule, -inf tail of the full logits rows,
// the warpgroups' tile loop, TMEM release.
#pragma once

#include "pmqa_main.cuh"

namespace pmqa {

// ---------------------------------------------------------------- kernel

static_assert(kMaxThreads <= 32 * 32, "CtaCtl holds per-warp sums for at most 32 warps");

// NN = next_n; POOL32: every byte offset of the pool fits in 31 bits (window
// mode only).
template <int H, int NN, bool SLICED, bool PAGE, bool POOL32>
__global__ void __launch_bounds__(kMaxThreads, 1)
    pmqa_main_kernel(const __grid_constant__ MainArgs a)
{
    extern __shared__ uint8_t smem_raw[];
    __shared__ CtaCtl ctl;
    // 1024-byte aligned (128B-swizzled operands); pointer arithmetic on the
    // shared array keeps the pointer in the shared address space
    uint8_t *const smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // the selection launched after this kernel may start launching now; it
    // waits for this grid's completion before it reads anything
    griddep_launch_dependents();
    if (threadIdx.x == 0) {
        ctl.abort = 0;
        const Bars B(a, smem);
        for (int q = 0; q < a.QS; ++q)
            mbar_init(&B.qfull[q], 1);
        for (int g = 0; g < kGroups; ++g)
            mbar_init(&B.mma[g], 1);
        for (int w = 0; w < kNumWarps; ++w)
            mbar_init(&B.run[w], 1);
        for (int h = 0; h < 2; ++h)
            mbar_init(&B.tfree[h], 4);  // one arrival per warp of the user
        mbar_init_fence();
    }
    __syncwarp();
    if (warp == 0)
        tmem_alloc(&ctl.tmem_base, (uint32_t)a.tmem_cols);

    balance_schedule(a.bs, [&](int i) { return (long long)tiles_of<SLICED>(a, i); }, ctl);
    for (int n = threadIdx.x; n < kCtxCache; n += blockDim.x)
        ctl.ctx[n] = ctl.i0 + n < a.bs ? ctx_of(a, ctl.i0 + n) : 0;
    if (blockIdx.x == 0) {
        const long long lim = min((long long)a.mml, (long long)a.W * a.P);
        for (int i = threadIdx.x; i < a.bs; i += blockDim.x) {
            const int cx = __ldg(a.ctx_lens + i);
            if (cx < 0 || cx > lim)
                atomicOr(a.status, 0x2u);
        }
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();

    // -inf beyond the last tile of each row: this CTA's share of every row.
    // Each warp takes 32 rows at a time (one coalesced load of their context
    // lengths), then writes the rows' shares one after another.
    if (a.logits) {
        const int rows = a.bs * a.nn;
        const long long mml = a.mml;
        const float NEG_INF = -__int_as_float(0x7f800000);
        for (int base = warp * 32; base < rows; base += kMaxThreads) {
            const int my_row = base + lane;
            const int my_cx = my_row < rows ? ctx_of(a, my_row / a.nn) : 0;
            const int nr = min(32, rows - base);
            for (int u = 0; u < nr; ++u) {
                const int cx = __shfl_sync(kFullMask, my_cx, u);
                const long long lo =
                    min((long long)(cx + kTileTokens - 1) / kTileTokens * kTileTokens, mml);
                const long long L = mml - lo;
                const long long s0 = lo + L * blockIdx.x / gridDim.x;
                const long long s1 = lo + L * (blockIdx.x + 1) / gridDim.x;
                float *row = a.logits + (long long)(base + u) * mml;
                for (long long t = s0 + lane; t < s1; t += 32)
                    row[t] = NEG_INF;
            }
        }
    }

    group_role<H, NN, SLICED, PAGE, POOL32>(a, smem, ctl, warp >> 2, warp & 3);

    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    __syncwarp();
    if (warp == 0)
        tmem_dealloc(ctl.tmem_base, (uint32_t)a.tmem_cols);
}

}  // namespace pmqa
