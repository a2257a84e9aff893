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
// in b* go to a per-row candidate list; each CTA takes its output ranges with
// one atomic per list. The last CTA of the row (an arrival counter, no
// waiting) resolves the candidates exactly with two more digits (11 and 10
// bits), from shared memory when they fit, pads the output and returns the
// row's workspace state to zero.
#pragma once

#include <cstdint>

#include "pmqa_main.cuh"

namespace pmqa {

struct SelectArgs {
    const float *logits;  // [rows, mml]; positions t < valid_len are read
    const int32_t *ctx_lens;
    int bs, nn, mml, k;
    int ctx_lim;        // contexts are clamped to [0, ctx_lim]: the KV pass's limit
                        // min(mml, P * max_blocks_per_seq) on the fused path, mml alone
    const int32_t *tok_begin, *tok_end;  // a slice of each request's tokens, or null
    int32_t *idx;       // [rows, k]
    float *vals;        // [rows, k] or null
    uint32_t *hist;     // [rows, 2048]
    uint32_t *sel_cnt;  // [rows]
    uint32_t *tie_cnt;  // [rows]
    uint32_t *arrive;   // [rows]
    uint2 *ties;        // [rows, mml] candidates: (position, order key)
    uint32_t *status;
    int splits;  // CTAs per row in the grid (gridDim.x); a row uses ceil(valid_len / chunk)
    int chunk;   // positions per CTA
};

constexpr int kSelThreads = 512;
constexpr int kSelPer = 16;  // positions per thread: one CTA covers 512 * 16 = 8192

// Positions [lo, hi) that row `row` selects from: the admitted positions
// t < valid_len, inside its request's slice [tok_begin, tok_end) when one is
// given (the clamps of the KV pass).
__device__ __forceinline__ void sel_window(const SelectArgs &a, int row, int &lo, int &hi)
{
    const int i = row / a.nn;
    const int c = clamp_ctx(__ldg(a.ctx_lens + i), (long long)a.ctx_lim);
    hi = valid_len(c, a.nn, row % a.nn);
    lo = 0;
    if (a.tok_begin) {
        const int tb = clamp_ctx(__ldg(a.tok_begin + i), (long long)c);
        const int te = max(tb, clamp_ctx(__ldg(a.tok_end + i), (long long)c));
        lo = tb;
        hi = max(tb, min(hi, te));
    }
}

// Per-row histogram of the top 11 bits of the order keys (stand-alone top-k).
__global__ void __launch_bounds__(kSelThreads) pmqa_hist_kernel(const __grid_constant__ SelectArgs a)
{
    __shared__ uint32_t h[kHistBins];
    const int row = blockIdx.y;
    int lo, hi;
    sel_window(a, row, lo, hi);
    const int n = hi - lo;
    const long long t0 = (long long)blockIdx.x * a.chunk;
    const long long t1 = min(t0 + a.chunk, (long long)n);
    if (t0 >= t1)
        return;
    for (int e = threadIdx.x; e < kHistBins; e += kSelThreads)
        h[e] = 0;
    __syncthreads();
    const float *src = a.logits + (long long)row * a.mml + lo;
    // all of this CTA's loads in flight first, then plain shared atomics
    float v[kSelPer];
#pragma unroll
    for (int u = 0; u < kSelPer; ++u) {
        const long long t = t0 + u * kSelThreads + threadIdx.x;
        v[u] = t < t1 ? __ldcg(src + t) : 0.0f;
    }
#pragma unroll
    for (int u = 0; u < kSelPer; ++u) {
        const long long t = t0 + u * kSelThreads + threadIdx.x;
        if (t < t1)
            atomicAdd(&h[f32_order_key(v[u]) >> kHistShift], 1u);
    }
    __syncthreads();
    for (int e = threadIdx.x; e < kHistBins; e += kSelThreads)
        if (h[e])
            atomicAdd(a.hist + (long long)row * kHistBins + e, h[e]);
}

constexpr int kTieCap = 4096;    // tie entries resolved from shared memory

struct SelShared {
    uint32_t h[kHistBins];
    uint32_t wsum[kSelThreads / 32];
    uint32_t wsel[kSelThreads / 32], wtie[kSelThreads / 32];  // per-warp counts, then offsets
    uint32_t bstar, above, digit, above2, eq_taken, last, base_sel, base_tie;
    int32_t tpos[kTieCap];   // tie positions of the row (last CTA)
    uint32_t tkey[kTieCap];  // their order keys
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
    // the sums of the warps before this one: lane l holds warp l's, then a
    // warp reduction (exact: integer adds)
    uint32_t woff = lane < wid ? s.wsum[lane] : 0u;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        woff += __shfl_xor_sync(kFullMask, woff, o);
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

// Exclusive prefix over the CTA of a per-thread count; returns this thread's
// offset, the CTA total in *total. Every thread calls.
__device__ uint32_t cta_exclusive_scan(SelShared &s, uint32_t x, uint32_t *total)
{
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    uint32_t incl = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t v = __shfl_up_sync(kFullMask, incl, o);
        if (lane >= o)
            incl += v;
    }
    __syncthreads();
    if (lane == 31)
        s.wsum[wid] = incl;
    __syncthreads();
    uint32_t woff = 0, all = 0;
    for (int w = 0; w < kSelThreads / 32; ++w) {
        woff += w < wid ? s.wsum[w] : 0;
        all += s.wsum[w];
    }
    *total = all;
    return woff + incl - x;
}

__device__ __forceinline__ float f32_from_order_key(uint32_t key)
{
    return __uint_as_float((key & 0x80000000u) ? (key & 0x7FFFFFFFu) : ~key);
}

// One CTA = up to 8192 positions of one row. The CTA holds its positions'
// logits in registers (all loads in flight at once), counts the sure winners
// (key bin above b*) and the candidates (bin b*), takes its output ranges
// with one atomic each and writes them. The last CTA of the row resolves the
// candidates from shared memory.
__global__ void __launch_bounds__(kSelThreads) pmqa_select_kernel(const __grid_constant__ SelectArgs a)
{
    __shared__ SelShared s;
    const int row = blockIdx.y, tid = threadIdx.x;
    // launched as a dependent of the KV pass: its logits and histograms are
    // complete and visible after this
    griddep_wait();
    int lo, hi;
    sel_window(a, row, lo, hi);
    const int n = hi - lo;  // positions lo + t, 0 <= t < n
    const uint32_t keff = (uint32_t)min(a.k, n);
    const float NEG_INF = -__int_as_float(0x7f800000);
    const long long rbase = (long long)row * a.mml + lo;
    int32_t *orow = a.idx + (long long)row * a.k;
    float *vrow = a.vals ? a.vals + (long long)row * a.k : nullptr;
    uint32_t *const status = a.status;
    // the row's CTAs: enough to cover its valid positions (one when it has none)
    const int row_ctas = n > 0 ? (n + a.chunk - 1) / a.chunk : 1;
    if ((int)blockIdx.x >= row_ctas)
        return;

    // this CTA's positions: all loads in flight first
    const long long t0 = (long long)blockIdx.x * a.chunk;
    const long long t1 = min(t0 + a.chunk, (long long)n);
    float v[kSelPer];
#pragma unroll
    for (int u = 0; u < kSelPer; ++u) {
        const long long t = t0 + u * kSelThreads + tid;
        v[u] = (keff > 0 && t < t1) ? __ldcg(a.logits + rbase + t) : NEG_INF;
    }

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

    // bit u of msel / mtie: position u of this thread is a winner / candidate
    uint32_t msel = 0, mtie = 0;
    if (keff > 0) {
#pragma unroll
        for (int u = 0; u < kSelPer; ++u) {
            const long long t = t0 + u * kSelThreads + tid;
            const uint32_t bin = f32_order_key(v[u]) >> kHistShift;
            msel |= (t < t1 && bin > bstar) ? 1u << u : 0u;
            mtie |= (t < t1 && bin == bstar) ? 1u << u : 0u;
        }
    }
    // output ranges: the CTA's from one atomic per list, each warp's after the
    // warps before it
    const int lane = tid & 31, wid = tid >> 5;
    const uint32_t wsel = __reduce_add_sync(kFullMask, (uint32_t)__popc(msel));
    const uint32_t wtie = __reduce_add_sync(kFullMask, (uint32_t)__popc(mtie));
    if (lane == 0) {
        s.wsel[wid] = wsel;
        s.wtie[wid] = wtie;
    }
    __syncthreads();
    if (tid == 0) {
        uint32_t as = 0, at = 0;
        for (int w = 0; w < kSelThreads / 32; ++w) {
            const uint32_t xs = s.wsel[w], xt = s.wtie[w];
            s.wsel[w] = as;
            s.wtie[w] = at;
            as += xs;
            at += xt;
        }
        s.base_sel = as ? atomicAdd(a.sel_cnt + row, as) : 0u;
        s.base_tie = at ? atomicAdd(a.tie_cnt + row, at) : 0u;
    }
    __syncthreads();
    if (wsel | wtie) {
        // position u of the warp's 32 lanes is 32 consecutive t: a warp writes
        // its winners (and candidates) of each u as one contiguous run
        uint32_t o_sel = s.base_sel + s.wsel[wid], o_tie = s.base_tie + s.wtie[wid];
        const uint32_t lt = (1u << lane) - 1u;
        uint2 *const trow = a.ties + (long long)row * a.mml;
#pragma unroll
        for (int u = 0; u < kSelPer; ++u) {
            const bool is_sel = (msel >> u) & 1u, is_tie = (mtie >> u) & 1u;
            const uint32_t bs = __ballot_sync(kFullMask, is_sel), bt = __ballot_sync(kFullMask, is_tie);
            const int32_t t = (int32_t)(lo + t0 + u * kSelThreads + tid);
            if (is_sel) {
                const uint32_t o = o_sel + __popc(bs & lt);
                if (o < keff) {
                    orow[o] = t;
                    if (vrow)
                        vrow[o] = v[u];
                } else {
                    atomicOr(status, 0x8u);
                }
            } else if (is_tie) {
                const uint32_t o = o_tie + __popc(bt & lt);
                if (o < (uint32_t)a.mml)
                    trow[o] = make_uint2((uint32_t)t, f32_order_key(v[u]));
                else
                    atomicOr(status, 0x8u);
            }
            o_sel += __popc(bs);
            o_tie += __popc(bt);
        }
    }

    // the last CTA of the row finishes it
    __threadfence();
    __syncthreads();
    if (tid == 0)
        s.last = atomicAdd(a.arrive + row, 1u) == (uint32_t)(row_ctas - 1) ? 1u : 0u;
    __syncthreads();
    if (!s.last)
        return;
    __threadfence();
    const uint32_t above = s.above;
    const uint32_t need = keff > above ? keff - above : 0u;
    const uint32_t ntie_row = keff > 0 ? min(__ldcg(a.tie_cnt + row), (uint32_t)a.mml) : 0u;
    const uint2 *tl = a.ties + (long long)row * a.mml;
    if (keff > 0 && __ldcg(a.sel_cnt + row) != above)
        atomicOr(status, 0x8u);
    if (need >= ntie_row) {
        // every candidate is selected
        for (uint32_t e = tid; e < ntie_row && above + e < keff; e += kSelThreads) {
            const uint2 c = __ldcg(tl + e);
            orow[above + e] = (int32_t)c.x;
            if (vrow)
                vrow[above + e] = f32_from_order_key(c.y);
        }
        if (need > ntie_row)
            atomicOr(status, 0x8u);
    } else if (need > 0) {
        // Candidates (position, key): from shared memory when they fit, else
        // re-read from the list on every pass.
        const bool cached = ntie_row <= (uint32_t)kTieCap;
        if (cached) {
            for (uint32_t e = tid; e < ntie_row; e += kSelThreads) {
                const uint2 c = __ldcg(tl + e);
                s.tpos[e] = (int32_t)c.x;
                s.tkey[e] = c.y;
            }
        }
        auto key_of = [&](uint32_t e) -> uint32_t { return cached ? s.tkey[e] : __ldcg(tl + e).y; };
        auto pos_of = [&](uint32_t e) -> int32_t { return cached ? s.tpos[e] : (int32_t)__ldcg(tl + e).x; };
        // second digit: key bits 20..10 of the candidates
        for (int e = tid; e < kHistBins; e += kSelThreads)
            s.h[e] = 0;
        __syncthreads();
        for (uint32_t e = tid; e < ntie_row; e += kSelThreads)
            atomicAdd(&s.h[(key_of(e) >> 10) & 2047u], 1u);
        __syncthreads();
        find_bin(s, s.h, kHistBins, need);
        const uint32_t d2 = s.digit, above2 = s.above2;
        const uint32_t need2 = need - above2;
        __syncthreads();
        // third digit: key bits 9..0 of the candidates in sub-bin d2
        for (int e = tid; e < 1024; e += kSelThreads)
            s.h[e] = 0;
        __syncthreads();
        for (uint32_t e = tid; e < ntie_row; e += kSelThreads) {
            const uint32_t key = key_of(e);
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
            s.above = 0;  // reused as the output cursor within the candidate range
        }
        __syncthreads();
        for (uint32_t e = tid; e < ntie_row; e += kSelThreads) {
            const uint32_t key = key_of(e);
            bool take = key > T;
            if (key == T)
                take = atomicAdd(&s.eq_taken, 1u) < eq_need;
            if (take) {
                const uint32_t o = above + atomicAdd(&s.above, 1u);
                if (o < keff) {
                    orow[o] = pos_of(e);
                    if (vrow)
                        vrow[o] = f32_from_order_key(key);
                } else {
                    atomicOr(status, 0x8u);
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

// ---------------------------------------------------------------- one CTA per row

// Rows of at most kRowMaxLen positions are selected by one CTA of kRowThreads
// threads that holds the row's logits in shared memory: the same radix select
// (first digit from the row's histogram, one classifying pass, the boundary
// bin resolved with two more digits), with every count, offset and candidate
// list in shared memory, so no global atomics, arrival counters or second
// CTA are involved.
constexpr int kRowThreads = 1024;
constexpr int kRowMaxLen = 32768;        // 128 KB of logits in dynamic shared memory
constexpr int kRowMaxLenStream = 65536;  // rows read from L2 in place
static_assert(kRowMaxLenStream <= 64 * kRowThreads, "one 64-bit mask per thread covers its positions");

struct RowShared {
    uint32_t h[kHistBins];
    uint32_t wsum[kRowThreads / 32];
    uint32_t digit, above2, bstar, above, eq_taken, cursor;
    uint64_t loaded;  // mbarrier of the row's bulk copy
    int32_t tpos[kTieCap];
    uint32_t tkey[kTieCap];
};

// find_bin for kRowThreads threads (1 or 2 bins each).
__device__ void row_find_bin(RowShared &s, const uint32_t *h, int nbins, uint32_t need)
{
    const int per = nbins / kRowThreads;
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int hi = nbins - 1 - tid * per;
    if (tid == 0) {
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
    // the sums of the warps before this one: lane l holds warp l's, then a
    // warp reduction (exact: integer adds)
    uint32_t woff = lane < wid ? s.wsum[lane] : 0u;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        woff += __shfl_xor_sync(kFullMask, woff, o);
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

// Exclusive prefix of a per-thread count over the CTA; the total in *total.
__device__ uint32_t row_exclusive_scan(RowShared &s, uint32_t x, uint32_t *total)
{
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    uint32_t incl = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t v = __shfl_up_sync(kFullMask, incl, o);
        if (lane >= o)
            incl += v;
    }
    __syncthreads();
    if (lane == 31)
        s.wsum[wid] = incl;
    __syncthreads();
    // warp 0 turns the 32 warp sums into exclusive offsets (and the total)
    if (wid == 0) {
        const uint32_t w = s.wsum[lane];
        uint32_t wi = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t v = __shfl_up_sync(kFullMask, wi, o);
            if (lane >= o)
                wi += v;
        }
        s.wsum[lane] = wi - w;
        if (lane == 31)
            s.cursor = wi;
    }
    __syncthreads();
    *total = s.cursor;
    return s.wsum[wid] + incl - x;
}

// IN_SMEM: the row (at most kRowMaxLen positions) is copied into shared
// memory first; else (at most kRowMaxLenStream) it passes through shared
// memory in halves of kRowMaxLen positions for the counting pass (or is read
// in place when it cannot be bulk-copied), and the writing pass re-reads the
// winners and candidates in place.
template <bool IN_SMEM>
__global__ void __launch_bounds__(kRowThreads, 1) pmqa_select_row_kernel(const __grid_constant__ SelectArgs a)
{
    extern __shared__ __align__(16) float sv[];  // the row's logits, positions 0 .. n - 1
    __shared__ RowShared s;
    constexpr int PER = (IN_SMEM ? kRowMaxLen : kRowMaxLenStream) / kRowThreads;  // positions per thread
    const int row = blockIdx.x, tid = threadIdx.x;
    // launched as a dependent of the KV pass: its logits and histograms are
    // complete and visible after this
    griddep_wait();
    int lo, hi;
    sel_window(a, row, lo, hi);
    const int n = min(hi - lo, PER * kRowThreads);  // positions lo + t, 0 <= t < n
    const uint32_t keff = (uint32_t)min(a.k, n);
    const float NEG_INF = -__int_as_float(0x7f800000);
    const long long rbase = (long long)row * a.mml + lo;
    int32_t *orow = a.idx + (long long)row * a.k;
    float *vrow = a.vals ? a.vals + (long long)row * a.k : nullptr;
    uint32_t *const status = a.status;

    // the row by bulk copy when it is 16-byte aligned (every row is when the
    // logits are, max_model_len is a multiple of 4 and so is lo), else by
    // plain loads; a copy rounded up to 16 bytes stays inside the row
    const float *src = a.logits + rbase;
    const bool bulk = keff > 0 && ((reinterpret_cast<uintptr_t>(src) & 15u) == 0) && (a.mml % 4 == 0);
    // copy positions [c * kRowMaxLen, ...) of the row into sv (thread 0)
    auto copy_chunk = [&](int c) {
        const int p0 = c * kRowMaxLen, len = min(n - p0, kRowMaxLen);
        const uint32_t bytes = (uint32_t)((len + 3) & ~3) * 4u;  // inside the row: mml % 4 == 0
        mbar_arrive_expect_tx(&s.loaded, bytes);
        for (uint32_t off = 0; off < bytes; off += 32768u)
            bulk_load(smem_u32(sv) + off, reinterpret_cast<const uint8_t *>(src + p0) + off,
                      min(32768u, bytes - off), &s.loaded);
    };
    if (bulk && tid == 0) {
        mbar_init(&s.loaded, 1);
        mbar_init_fence();
        copy_chunk(0);
    }
    if (keff > 0) {
        for (int e = tid; e < kHistBins; e += kRowThreads)
            s.h[e] = __ldcg(a.hist + (long long)row * kHistBins + e);
        __syncthreads();  // the mbarrier is initialised
        // the row into shared memory, 16 independent loads in flight per thread
        constexpr int kBatch = 16;
        for (int base = 0; IN_SMEM && !bulk && base < n; base += kRowThreads * kBatch) {
            float v[kBatch];
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                const int t = base + u * kRowThreads + tid;
                v[u] = t < n ? __ldcg(a.logits + rbase + t) : 0.0f;
            }
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                const int t = base + u * kRowThreads + tid;
                if (t < n)
                    sv[t] = v[u];
            }
        }
        __syncthreads();
        row_find_bin(s, s.h, kHistBins, keff);
        const uint32_t bstar = s.digit, above = s.above2;
        // the bulk copy of the row ran during the bin search
        if (IN_SMEM && bulk && !mbar_wait(&s.loaded, 0, nullptr))
            atomicOr(status, 0x4u);
        auto val = [&](int t) -> float { return IN_SMEM ? sv[t] : __ldcg(src + t); };
        // winners (key bin above b*) and candidates (bin b*) of this thread:
        // bit u stands for position tid + u * kRowThreads. The order key is
        // monotone in the value (-0 folded onto +0, which v >= +0 also does),
        // so the bin tests are two float compares against the values whose
        // keys bound bin b*; for finite logits those are finite or +inf, and
        // the key compare stays for the case where one is NaN.
        const bool top = bstar + 1 >= (uint32_t)kHistBins;  // nothing lies above b*
        const float f0 = f32_from_order_key(bstar << kHistShift);
        const float f1 = top ? 0.0f : f32_from_order_key((bstar + 1) << kHistShift);
        const bool by_value = !isnan(f0) && !isnan(f1);
        uint64_t msel = 0, mtie = 0;
        if (!IN_SMEM && bulk && by_value) {
            // half by half through shared memory: half c is bits 32 c .. 32 c + 31
            for (int c = 0; c * kRowMaxLen < n; ++c) {
                if (c > 0 && tid == 0)
                    copy_chunk(c);
                if (!mbar_wait(&s.loaded, (uint32_t)c & 1u, nullptr))
                    atomicOr(status, 0x4u);
                uint32_t ms = 0, mt = 0;
#pragma unroll
                for (int u = 0; u < kRowMaxLen / kRowThreads; ++u) {
                    const int tl0 = tid + u * kRowThreads;  // position within the half
                    if (c * kRowMaxLen + tl0 < n) {
                        const float v = sv[tl0];
                        const bool sel = !top && v >= f1;
                        if (sel)
                            ms |= 1u << u;
                        else if (v >= f0)
                            mt |= 1u << u;
                    }
                }
                msel |= (uint64_t)ms << (32 * c);
                mtie |= (uint64_t)mt << (32 * c);
                __syncthreads();  // every thread is done with the half before the next copy
            }
        } else if (by_value) {
            // (read in place; a first half already on its way lands first)
            if (!IN_SMEM && bulk && !mbar_wait(&s.loaded, 0, nullptr))
                atomicOr(status, 0x4u);
#pragma unroll
            for (int u = 0; u < PER; ++u) {
                const int t = tid + u * kRowThreads;
                if (t < n) {
                    const float v = val(t);
                    const bool sel = !top && v >= f1;
                    if (sel)
                        msel |= 1ull << u;
                    else if (v >= f0)
                        mtie |= 1ull << u;
                }
            }
        } else {
            if (!IN_SMEM && bulk && !mbar_wait(&s.loaded, 0, nullptr))
                atomicOr(status, 0x4u);
#pragma unroll 16
            for (int u = 0; u < PER; ++u) {
                const int t = tid + u * kRowThreads;
                if (t < n) {
                    const uint32_t bin = f32_order_key(val(t)) >> kHistShift;
                    msel |= (uint64_t)(bin > bstar ? 1u : 0u) << u;
                    mtie |= (uint64_t)(bin == bstar ? 1u : 0u) << u;
                }
            }
        }
        const uint32_t cs = (uint32_t)__popcll(msel), ct = (uint32_t)__popcll(mtie);
        uint32_t tot_s, tot_t;
        uint32_t o_s = row_exclusive_scan(s, cs, &tot_s);
        uint32_t o_t = row_exclusive_scan(s, ct, &tot_t);
        if (tid == 0 && tot_s != above)
            atomicOr(status, 0x8u);
        // candidates stay in shared memory when they fit, else go to the
        // row's list in the workspace
        const bool cached = tot_t <= (uint32_t)kTieCap;
        uint2 *const tl = a.ties + (long long)row * a.mml;
        for (uint64_t m = msel; m; m &= m - 1) {
            const int t = tid + (__ffsll((long long)m) - 1) * kRowThreads;
            if (o_s < keff) {
                orow[o_s] = lo + t;
                if (vrow)
                    vrow[o_s] = val(t);
            } else {
                atomicOr(status, 0x8u);
            }
            ++o_s;
        }
        for (uint64_t m = mtie; m; m &= m - 1) {
            const int t = tid + (__ffsll((long long)m) - 1) * kRowThreads;
            const uint32_t key = f32_order_key(val(t));
            if (cached) {
                s.tpos[o_t] = lo + t;
                s.tkey[o_t] = key;
            } else {
                tl[o_t] = make_uint2((uint32_t)(lo + t), key);
            }
            ++o_t;
        }
        if (!cached)
            __threadfence_block();
        __syncthreads();
        const uint32_t need = keff > above ? keff - above : 0u;
        const uint32_t ntie = tot_t;
        auto key_of = [&](uint32_t e) -> uint32_t { return cached ? s.tkey[e] : __ldcg(tl + e).y; };
        auto pos_of = [&](uint32_t e) -> int32_t { return cached ? s.tpos[e] : (int32_t)__ldcg(tl + e).x; };
        if (need >= ntie) {
            // every candidate is selected
            for (uint32_t e = tid; e < ntie && above + e < keff; e += kRowThreads) {
                orow[above + e] = pos_of(e);
                if (vrow)
                    vrow[above + e] = f32_from_order_key(key_of(e));
            }
            if (need > ntie && tid == 0)
                atomicOr(status, 0x8u);
        } else if (need > 0) {
            // second digit: key bits 20..10 of the candidates
            for (int e = tid; e < kHistBins; e += kRowThreads)
                s.h[e] = 0;
            __syncthreads();
            for (uint32_t e = tid; e < ntie; e += kRowThreads)
                atomicAdd(&s.h[(key_of(e) >> 10) & 2047u], 1u);
            __syncthreads();
            row_find_bin(s, s.h, kHistBins, need);
            const uint32_t d2 = s.digit, above2 = s.above2;
            const uint32_t need2 = need - above2;
            __syncthreads();
            // third digit: key bits 9..0 of the candidates in sub-bin d2
            for (int e = tid; e < 1024; e += kRowThreads)
                s.h[e] = 0;
            __syncthreads();
            for (uint32_t e = tid; e < ntie; e += kRowThreads) {
                const uint32_t key = key_of(e);
                if (((key >> 10) & 2047u) == d2)
                    atomicAdd(&s.h[key & 1023u], 1u);
            }
            __syncthreads();
            row_find_bin(s, s.h, 1024, need2);
            const uint32_t d3 = s.digit, above3 = s.above2;
            const uint32_t T = (bstar << kHistShift) | (d2 << 10) | d3;  // the k-th largest key
            const uint32_t eq_need = need2 - above3;
            if (tid == 0) {
                s.eq_taken = 0;
                s.cursor = 0;
            }
            __syncthreads();
            for (uint32_t e = tid; e < ntie; e += kRowThreads) {
                const uint32_t key = key_of(e);
                bool take = key > T;
                if (key == T)
                    take = atomicAdd(&s.eq_taken, 1u) < eq_need;
                if (take) {
                    const uint32_t o = above + atomicAdd(&s.cursor, 1u);
                    if (o < keff) {
                        orow[o] = pos_of(e);
                        if (vrow)
                            vrow[o] = f32_from_order_key(key);
                    } else {
                        atomicOr(status, 0x8u);
                    }
                }
            }
        }
    }
    for (int e = (int)keff + tid; e < a.k; e += kRowThreads) {
        orow[e] = -1;
        if (vrow)
            vrow[e] = NEG_INF;
    }
    // the row's histogram returns to zero for the next call (every read of it
    // happened before the first row_find_bin's barriers)
    for (int e = tid; e < kHistBins; e += kRowThreads)
        a.hist[(long long)row * kHistBins + e] = 0;
}

}  // namespace pmqa

namespace pmqa {

// ---------------------------------------------------------------- merge of shard lists

// Candidate lists of a context-parallel split (section 8 of the scope: each
// GPU holds a slice of every request's tokens, keeps its slice's top-k as
// (position, logit) pairs, and the lists are gathered and merged): the top-k
// of the union of `lists` lists per row. Each global top-k position is in its
// slice's top-k, so the union's top-k is the row's top-k.
struct MergeArgs {
    const int32_t *idx;  // [lists, rows, k_in], -1 for an empty slot
    const float *vals;   // [lists, rows, k_in]
    int lists, rows, k_in, k;
    int32_t *out_idx;    // [rows, k]
    float *out_vals;     // [rows, k] or null
};

// One CTA per row: a histogram of the valid candidates' top 11 key bits, the
// boundary bin, one pass that writes the winners and sets the boundary bin's
// candidates aside, and those resolved with two more digits.
__global__ void __launch_bounds__(kSelThreads, 1) pmqa_merge_kernel(const __grid_constant__ MergeArgs a)
{
    __shared__ SelShared s;
    const int row = blockIdx.x, tid = threadIdx.x;
    const long long n = (long long)a.lists * a.k_in;
    int32_t *orow = a.out_idx + (long long)row * a.k;
    float *vrow = a.out_vals ? a.out_vals + (long long)row * a.k : nullptr;
    // candidate e of the row: slot e % k_in of list e / k_in
    auto load = [&](long long e, int32_t &pos, uint32_t &key) -> bool {
        const long long l = e / a.k_in, c = e - l * a.k_in;
        const long long o = (l * a.rows + row) * a.k_in + c;
        pos = __ldg(a.idx + o);
        key = pos >= 0 ? f32_order_key(__ldg(a.vals + o)) : 0u;
        return pos >= 0;
    };
    for (int e = tid; e < kHistBins; e += kSelThreads)
        s.h[e] = 0;
    __syncthreads();
    uint32_t cnt = 0;
    for (long long e = tid; e < n; e += kSelThreads) {
        int32_t pos;
        uint32_t key;
        if (load(e, pos, key)) {
            atomicAdd(&s.h[key >> kHistShift], 1u);
            ++cnt;
        }
    }
    uint32_t total;
    cta_exclusive_scan(s, cnt, &total);
    __syncthreads();
    const uint32_t keff = min((uint32_t)a.k, total);
    if (keff > 0) {
        find_bin(s, s.h, kHistBins, keff);
        const uint32_t bstar = s.digit, above = s.above2;
        if (tid == 0) {
            s.base_sel = 0;  // output cursor
            s.base_tie = 0;  // candidates of the boundary bin
        }
        __syncthreads();
        for (long long e = tid; e < n; e += kSelThreads) {
            int32_t pos;
            uint32_t key;
            if (!load(e, pos, key))
                continue;
            const uint32_t bin = key >> kHistShift;
            if (bin > bstar) {
                const uint32_t o = atomicAdd(&s.base_sel, 1u);
                if (o < keff) {
                    orow[o] = pos;
                    if (vrow)
                        vrow[o] = f32_from_order_key(key);
                }
            } else if (bin == bstar) {
                const uint32_t q = atomicAdd(&s.base_tie, 1u);
                if (q < (uint32_t)kTieCap) {
                    s.tpos[q] = pos;
                    s.tkey[q] = key;
                }
            }
        }
        __syncthreads();
        const uint32_t need = keff > above ? keff - above : 0u;
        const uint32_t ntie = s.base_tie;
        const bool cached = ntie <= (uint32_t)kTieCap;
        // the boundary bin's candidates: from shared memory, or the lists again
        auto each_tie = [&](auto &&fn) {
            if (cached) {
                for (uint32_t e = tid; e < ntie; e += kSelThreads)
                    fn(s.tpos[e], s.tkey[e]);
            } else {
                for (long long e = tid; e < n; e += kSelThreads) {
                    int32_t pos;
                    uint32_t key;
                    if (load(e, pos, key) && (key >> kHistShift) == bstar)
                        fn(pos, key);
                }
            }
        };
        auto emit = [&](int32_t pos, uint32_t key) {
            const uint32_t o = atomicAdd(&s.base_sel, 1u);
            if (o < keff) {
                orow[o] = pos;
                if (vrow)
                    vrow[o] = f32_from_order_key(key);
            }
        };
        if (need >= ntie) {
            each_tie(emit);
        } else if (need > 0) {
            for (int e = tid; e < kHistBins; e += kSelThreads)
                s.h[e] = 0;
            __syncthreads();
            each_tie([&](int32_t, uint32_t key) { atomicAdd(&s.h[(key >> 10) & 2047u], 1u); });
            __syncthreads();
            find_bin(s, s.h, kHistBins, need);
            const uint32_t d2 = s.digit, need2 = need - s.above2;
            __syncthreads();
            for (int e = tid; e < 1024; e += kSelThreads)
                s.h[e] = 0;
            __syncthreads();
            each_tie([&](int32_t, uint32_t key) {
                if (((key >> 10) & 2047u) == d2)
                    atomicAdd(&s.h[key & 1023u], 1u);
            });
            __syncthreads();
            find_bin(s, s.h, 1024, need2);
            const uint32_t T = (bstar << kHistShift) | (d2 << 10) | s.digit;  // the k-th largest key
            const uint32_t eq_need = need2 - s.above2;
            if (tid == 0)
                s.eq_taken = 0;
            __syncthreads();
            each_tie([&](int32_t pos, uint32_t key) {
                bool take = key > T;
                if (key == T)
                    take = atomicAdd(&s.eq_taken, 1u) < eq_need;
                if (take)
                    emit(pos, key);
            });
        }
    }
    const float NEG_INF = -__int_as_float(0x7f800000);
    for (int e = (int)keff + tid; e < a.k; e += kSelThreads) {
        orow[e] = -1;
        if (vrow)
            vrow[e] = NEG_INF;
    }
}

}  // namespace pmqa
