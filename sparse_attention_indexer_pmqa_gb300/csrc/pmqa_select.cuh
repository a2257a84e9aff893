// pmqa_select.cuh -- exact per-row top-k from a key histogram.
//
// Row top-k as in the `test` driver on the page "[Bug] aiter ops triton
// attention pa" (section "Minimal reproduction"): the positions of the
// min(k, valid_len) largest logits among t < valid_len, k = min(2048, ctx)
// there; here the remaining slots hold -1 and ties may go either way.
//
// Radix select, first digit done ahead: every row carries a histogram of the
// top 11 bits of its order keys (built in the logits epilogue of the fused
// kernel, or by pmqa_hist_kernel). The select kernel reads the histogram,
// finds the bin b* holding the k-th largest key and makes one pass over the
// row: entries in bins above b* are written straight to the output, entries
// in b* go to a per-row tie list. The last CTA of the row (an arrival counter,
// no waiting) resolves the tie list exactly with two more digits (11 and 10
// bits), pads the output and returns the row's workspace state to zero.
#pragma once

#include <cstdint>

#include "pmqa_main.cuh"

namespace pmqa {

struct SelectArgs {
    const float *logits;  // [rows, mml]; positions t < valid_len are read
    const int32_t *ctx_lens;
    int bs, nn, mml, k;
    int32_t *idx;       // [rows, k]
    float *vals;        // [rows, k] or null
    uint32_t *hist;     // [rows, 2048]
    uint32_t *sel_cnt;  // [rows]
    uint32_t *tie_cnt;  // [rows]
    uint32_t *arrive;   // [rows]
    int32_t *ties;      // [rows, mml]
    uint32_t *status;
    int splits;  // CTAs per row (gridDim.x)
    int chunk;   // positions per CTA
};

constexpr int kSelThreads = 256;

__device__ __forceinline__ int sel_valid_len(const SelectArgs &a, int row)
{
    const int c = clamp_ctx(__ldg(a.ctx_lens + row / a.nn), (long long)a.mml);
    return valid_len(c, a.nn, row % a.nn);
}

// Per-row histogram of the top 11 bits of the order keys (stand-alone top-k).
__global__ void __launch_bounds__(kSelThreads) pmqa_hist_kernel(const __grid_constant__ SelectArgs a)
{
    __shared__ uint32_t h[kHistBins];
    const int row = blockIdx.y, lane = threadIdx.x & 31;
    const int n = sel_valid_len(a, row);
    const long long t0 = (long long)blockIdx.x * a.chunk;
    const long long t1 = min(t0 + a.chunk, (long long)n);
    if (t0 >= t1)
        return;
    for (int e = threadIdx.x; e < kHistBins; e += kSelThreads)
        h[e] = 0;
    __syncthreads();
    const float *src = a.logits + (long long)row * a.mml;
    for (long long base = t0; base < t1; base += kSelThreads) {
        const long long t = base + threadIdx.x;
        const bool in = t < t1;
        const uint32_t bin = in ? f32_order_key(__ldcs(src + t)) >> kHistShift : 0u;
        const uint32_t grp = __match_any_sync(kFullMask, in ? bin : 0x10000u + (uint32_t)lane);
        if (in && (__ffs(grp) - 1) == lane)
            atomicAdd(&h[bin], (uint32_t)__popc(grp));
    }
    __syncthreads();
    for (int e = threadIdx.x; e < kHistBins; e += kSelThreads)
        if (h[e])
            atomicAdd(a.hist + (long long)row * kHistBins + e, h[e]);
}

struct SelShared {
    uint32_t h[kHistBins];
    uint32_t wsum[kSelThreads / 32];
    uint32_t bstar, above, digit, above2, eq_taken, last;
};

// Find the bin b of h[0..nbins) (scanning from the top) where the running
// count first reaches `need`; *above = count strictly above b. need >= 1 and
// the total >= need. Every thread calls; results in s.digit / s.above2.
__device__ void find_bin(SelShared &s, const uint32_t *h, int nbins, uint32_t need)
{
    const int per = nbins / kSelThreads;  // 8 or 4 bins per thread, highest first
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int hi = nbins - 1 - tid * per;
    if (tid == 0) {
        // defaults if the counts cannot reach `need` (inconsistent input):
        // nothing above, lowest digit
        s.digit = 0;
        s.above2 = 0;
    }
    uint32_t loc = 0;
    for (int q = 0; q < per; ++q)
        loc += h[hi - q];
    uint32_t incl = loc;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t v = __shfl_up_sync(kFullMask, incl, o);
        if (lane >= o)
            incl += v;
    }
    if (lane == 31)
        s.wsum[wid] = incl;
    __syncthreads();
    uint32_t woff = 0;
    for (int w = 0; w < wid; ++w)
        woff += s.wsum[w];
    incl += woff;
    const uint32_t excl = incl - loc;
    if (excl < need && need <= incl) {
        uint32_t acc = excl;
        for (int q = 0; q < per; ++q) {
            const uint32_t v = h[hi - q];
            if (acc + v >= need) {
                s.digit = (uint32_t)(hi - q);
                s.above2 = acc;
                break;
            }
            acc += v;
        }
    }
    __syncthreads();
}

__global__ void __launch_bounds__(kSelThreads) pmqa_select_kernel(const __grid_constant__ SelectArgs a)
{
    __shared__ SelShared s;
    const int row = blockIdx.y, tid = threadIdx.x, lane = tid & 31;
    const int n = sel_valid_len(a, row);
    const uint32_t keff = (uint32_t)min(a.k, n);
    const float NEG_INF = -__int_as_float(0x7f800000);
    const long long rbase = (long long)row * a.mml;
    int32_t *orow = a.idx + (long long)row * a.k;
    float *vrow = a.vals ? a.vals + (long long)row * a.k : nullptr;

    // threshold bin of the k-th largest key
    for (int e = tid; e < kHistBins; e += kSelThreads)
        s.h[e] = __ldcg(a.hist + (long long)row * kHistBins + e);
    if (tid == 0) {
        s.bstar = kHistBins;  // nothing selected when keff == 0
        s.above = 0;
    }
    __syncthreads();
    if (keff > 0) {
        find_bin(s, s.h, kHistBins, keff);
        if (tid == 0) {
            s.bstar = s.digit;
            s.above = s.above2;
        }
        __syncthreads();
    }
    const uint32_t bstar = s.bstar;

    // one pass over this CTA's positions
    const long long t0 = (long long)blockIdx.x * a.chunk;
    const long long t1 = min(t0 + a.chunk, (long long)n);
    if (keff > 0) {
        for (long long base = t0; base < t1; base += kSelThreads) {
            const long long t = base + tid;
            float v = 0.f;
            uint32_t bin = kHistBins + 1;
            if (t < t1) {
                v = __ldcg(a.logits + rbase + t);
                bin = f32_order_key(v) >> kHistShift;
            }
            const bool sel = bin != kHistBins + 1 && bin > bstar && bin < kHistBins;
            const bool tie = bin == bstar;
            const uint32_t ms = __ballot_sync(kFullMask, sel);
            if (ms) {
                uint32_t b0 = 0;
                if (lane == 0)
                    b0 = atomicAdd(a.sel_cnt + row, (uint32_t)__popc(ms));
                b0 = __shfl_sync(kFullMask, b0, 0);
                if (sel) {
                    const uint32_t o = b0 + __popc(ms & ((1u << lane) - 1u));
                    if (o < keff) {
                        orow[o] = (int32_t)t;
                        if (vrow)
                            vrow[o] = v;
                    } else {
                        atomicOr(a.status, 0x8u);
                    }
                }
            }
            const uint32_t mt = __ballot_sync(kFullMask, tie);
            if (mt) {
                uint32_t b0 = 0;
                if (lane == 0)
                    b0 = atomicAdd(a.tie_cnt + row, (uint32_t)__popc(mt));
                b0 = __shfl_sync(kFullMask, b0, 0);
                if (tie) {
                    const uint32_t o = b0 + __popc(mt & ((1u << lane) - 1u));
                    if (o < (uint32_t)a.mml)
                        a.ties[rbase + o] = (int32_t)t;
                    else
                        atomicOr(a.status, 0x8u);
                }
            }
        }
    }

    // the last CTA of the row finishes it
    __threadfence();
    __syncthreads();
    if (tid == 0)
        s.last = atomicAdd(a.arrive + row, 1u) == (uint32_t)(a.splits - 1) ? 1u : 0u;
    __syncthreads();
    if (!s.last)
        return;
    __threadfence();
    const uint32_t above = s.above;
    const uint32_t need = keff > above ? keff - above : 0u;
    const uint32_t ntie = keff > 0 ? min(__ldcg(a.tie_cnt + row), (uint32_t)a.mml) : 0u;
    const int32_t *tl = a.ties + rbase;
    if (keff > 0 && __ldcg(a.sel_cnt + row) != above)
        atomicOr(a.status, 0x8u);
    if (need >= ntie) {
        // every tie is selected
        for (uint32_t e = tid; e < ntie && above + e < keff; e += kSelThreads) {
            const int32_t t = __ldcg(tl + e);
            orow[above + e] = t;
            if (vrow)
                vrow[above + e] = __ldcg(a.logits + rbase + t);
        }
        if (need > ntie)
            atomicOr(a.status, 0x8u);
    } else if (need > 0) {
        // second digit: key bits 20..10 of the tie entries
        for (int e = tid; e < kHistBins; e += kSelThreads)
            s.h[e] = 0;
        __syncthreads();
        for (uint32_t e = tid; e < ntie; e += kSelThreads) {
            const uint32_t key = f32_order_key(__ldcg(a.logits + rbase + __ldcg(tl + e)));
            atomicAdd(&s.h[(key >> 10) & 2047u], 1u);
        }
        __syncthreads();
        find_bin(s, s.h, kHistBins, need);
        const uint32_t d2 = s.digit, above2 = s.above2;
        const uint32_t need2 = need - above2;
        __syncthreads();
        // third digit: key bits 9..0 of the entries in sub-bin d2
        for (int e = tid; e < 1024; e += kSelThreads)
            s.h[e] = 0;
        __syncthreads();
        for (uint32_t e = tid; e < ntie; e += kSelThreads) {
            const uint32_t key = f32_order_key(__ldcg(a.logits + rbase + __ldcg(tl + e)));
            if (((key >> 10) & 2047u) == d2)
                atomicAdd(&s.h[key & 1023u], 1u);
        }
        __syncthreads();
        find_bin(s, s.h, 1024, need2);
        const uint32_t d3 = s.digit, above3 = s.above2;
        const uint32_t T = (bstar << kHistShift) | (d2 << 10) | d3;  // the k-th largest key
        const uint32_t eq_need = need2 - above3;
        if (tid == 0) {
            s.eq_taken = 0;
            s.above = 0;  // reused as the output cursor within the tie range
        }
        __syncthreads();
        for (uint32_t e = tid; e < ntie; e += kSelThreads) {
            const int32_t t = __ldcg(tl + e);
            const float v = __ldcg(a.logits + rbase + t);
            const uint32_t key = f32_order_key(v);
            bool take = key > T;
            if (key == T)
                take = atomicAdd(&s.eq_taken, 1u) < eq_need;
            if (take) {
                const uint32_t o = above + atomicAdd(&s.above, 1u);
                if (o < keff) {
                    orow[o] = t;
                    if (vrow)
                        vrow[o] = v;
                } else {
                    atomicOr(a.status, 0x8u);
                }
            }
        }
    }
    for (int e = (int)keff + tid; e < a.k; e += kSelThreads) {
        orow[e] = -1;
        if (vrow)
            vrow[e] = NEG_INF;
    }
    // leave the row's workspace state at zero for the next call, once every
    // thread of this CTA is past its last read of it
    __syncthreads();
    for (int e = tid; e < kHistBins; e += kSelThreads)
        a.hist[(long long)row * kHistBins + e] = 0;
    if (tid == 0) {
        a.sel_cnt[row] = 0;
        a.tie_cnt[row] = 0;
        a.arrive[row] = 0;
    }
}

}  // namespace pmqa
