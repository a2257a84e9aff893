// pmqa_topk_wg.cuh -- exact per-row top-k built from 128-thread work groups.
//
// Row top-k as on the page "[Bug] aiter ops triton attention pa", section
// "Minimal reproduction": the positions of the k largest logits of a row, k =
// min(2048, ctx) there; here k_eff = min(k, valid_len) with -1 in the unused
// slots. Any choice among equal values is accepted.
//
// Scheme. A row's tokens are split into contiguous segments, one per CTA range
// that touches the row. Each segment streams its logits through a shared-memory
// candidate buffer: a value enters only if its order key is >= the buffer's
// threshold; when the buffer is nearly full a radix select finds the k-th
// largest key T, the buffer is compacted to exactly k entries and the threshold
// becomes T + 1 (an entry equal to T can no longer change the answer). At the
// end of the segment the surviving candidates are appended to the row's list in
// the workspace and the segment adds its tile count to the row's arrival
// counter. The work group that completes the count merges the row's list with
// the same buffer machinery and writes the final k positions. No work group
// ever waits for another.
#pragma once

#include <cstdint>

#include "pmqa_ptx.cuh"

namespace pmqa {

constexpr uint32_t kFullMask = 0xFFFFFFFFu;

// fp32 -> uint32 with a > b  <=>  key(a) > key(b); -0 is folded onto +0.
__device__ __forceinline__ uint32_t f32_order_key(float f)
{
    uint32_t u = __float_as_uint(f == 0.0f ? 0.0f : f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float order_key_f32(uint32_t k)
{
    uint32_t u = (k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k;
    return __uint_as_float(u);
}

// Shared-memory scratch of one work group.
struct WgScratch {
    uint32_t hist[256];
    uint32_t wcount[2][4];
    uint32_t digit;
    uint32_t above;
    uint32_t ties;
    uint32_t bcast;
    uint32_t flag;
    uint32_t pad[3];
};

// A candidate buffer: capacity entries of (key, position) plus count/threshold.
struct CandBuf {
    uint32_t *key;
    int32_t *pos;
    uint32_t *count;   // shared scalar
    uint32_t *thresh;  // shared scalar: a value enters iff key >= *thresh
    uint32_t cap;
};

// Work-group context: 128 threads, named barrier `bar`.
struct Wg {
    uint32_t tid;   // 0..127
    uint32_t lane;  // 0..31
    uint32_t warp;  // 0..3
    uint32_t bar;   // named barrier id
    WgScratch *scr;
    __device__ __forceinline__ void sync() const { named_bar_sync(bar, 128); }
};

// Append (key, pos) for the lanes where `pass` holds. All 32 lanes of the
// calling warp must take part. The caller guarantees room for 128 more entries.
__device__ __forceinline__ void cand_append(const CandBuf &b, const Wg &g, uint32_t key,
                                            int32_t pos, bool pass)
{
    const uint32_t m = __ballot_sync(kFullMask, pass);
    if (m == 0)
        return;
    uint32_t base = 0;
    if (g.lane == 0)
        base = atomicAdd(b.count, (uint32_t)__popc(m));
    base = __shfl_sync(kFullMask, base, 0);
    if (pass) {
        const uint32_t o = base + __popc(m & ((1u << g.lane) - 1u));
        b.key[o] = key;
        b.pos[o] = pos;
    }
}

// k-th largest key among key[0..n) (1 <= k <= n), MSB-first radix select over
// four 8-bit digits. Returns T; *n_above receives the number of keys > T.
// Must be called by all 128 threads.
static __device__ uint32_t wg_select(const uint32_t *key, uint32_t n, uint32_t k, const Wg &g,
                              uint32_t *n_above)
{
    uint32_t prefix = 0, pmask = 0, krem = k, above_total = 0;
    WgScratch *s = g.scr;
    for (int shift = 24; shift >= 0; shift -= 8) {
        s->hist[g.tid] = 0;
        s->hist[g.tid + 128] = 0;
        g.sync();
        for (uint32_t base = g.warp * 32; base < n; base += 128) {
            const uint32_t e = base + g.lane;
            const uint32_t kk = e < n ? key[e] : 0u;
            const bool in = e < n && (kk & pmask) == prefix;
            const uint32_t d = in ? ((kk >> shift) & 255u) : (256u + g.lane);
            const uint32_t grp = __match_any_sync(kFullMask, d);
            if (in && (__ffs(grp) - 1) == (int)g.lane)
                atomicAdd(&s->hist[d], (uint32_t)__popc(grp));
        }
        g.sync();
        if (g.warp == 0) {
            // lane l owns digits 255-8l down to 248-8l (largest first)
            const uint32_t hi = 255u - 8u * g.lane;
            uint32_t c = 0;
#pragma unroll
            for (int q = 0; q < 8; ++q)
                c += s->hist[hi - q];
            uint32_t incl = c;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t v = __shfl_up_sync(kFullMask, incl, o);
                if (g.lane >= (uint32_t)o)
                    incl += v;
            }
            const uint32_t excl = incl - c;
            if (excl < krem && krem <= incl) {
                uint32_t acc = excl;
                for (int q = 0; q < 8; ++q) {
                    const uint32_t h = s->hist[hi - q];
                    if (acc + h >= krem) {
                        s->digit = hi - q;
                        s->above = acc;
                        break;
                    }
                    acc += h;
                }
            }
        }
        g.sync();
        const uint32_t dgt = s->digit, abv = s->above;
        above_total += abv;
        krem -= abv;
        prefix |= dgt << shift;
        pmask |= 0xFFu << shift;
    }
    *n_above = above_total;
    return prefix;
}

// Keep every entry with key > T and the first `ties` entries with key == T
// (first in an arbitrary order), packed to the front. Returns the new count.
static __device__ uint32_t wg_compact(const CandBuf &b, uint32_t n, uint32_t T, uint32_t ties,
                               const Wg &g)
{
    WgScratch *s = g.scr;
    if (g.tid == 0)
        s->ties = 0;
    g.sync();
    uint32_t out = 0;
    uint32_t par = 0;
    for (uint32_t c0 = 0; c0 < n; c0 += 128, par ^= 1u) {
        const uint32_t e = c0 + g.tid;
        uint32_t kk = 0;
        int32_t pp = 0;
        bool keep = false;
        if (e < n) {
            kk = b.key[e];
            pp = b.pos[e];
            if (kk > T)
                keep = true;
            else if (kk == T)
                keep = atomicAdd(&s->ties, 1u) < ties;
        }
        const uint32_t m = __ballot_sync(kFullMask, keep);
        if (g.lane == 0)
            s->wcount[par][g.warp] = __popc(m);
        g.sync();
        uint32_t before = 0, total = 0;
#pragma unroll
        for (uint32_t w = 0; w < 4; ++w) {
            const uint32_t v = s->wcount[par][w];
            before += w < g.warp ? v : 0u;
            total += v;
        }
        if (keep) {
            const uint32_t o = out + before + __popc(m & ((1u << g.lane) - 1u));
            b.key[o] = kk;
            b.pos[o] = pp;
        }
        out += total;
    }
    g.sync();
    return out;
}

// Reduce the buffer to its k largest entries (k >= 1) and raise the threshold
// past the k-th key. Called by all 128 threads when *b.count > k.
static __device__ void cand_shrink(const CandBuf &b, uint32_t k, const Wg &g)
{
    const uint32_t n = *b.count;
    uint32_t n_above;
    const uint32_t T = wg_select(b.key, n, k, g, &n_above);
    const uint32_t kept = wg_compact(b, n, T, k - n_above, g);
    if (g.tid == 0) {
        *b.count = kept;
        *b.thresh = T == 0xFFFFFFFFu ? T : T + 1u;
    }
    g.sync();
}

// After a round of appends: make room for the next 128 if needed. All threads.
__device__ __forceinline__ void cand_make_room(const CandBuf &b, uint32_t k, const Wg &g)
{
    g.sync();
    const uint32_t n = *b.count;
    g.sync();
    if (n > b.cap - 128u)
        cand_shrink(b, k, g);
}

__device__ __forceinline__ void cand_reset(const CandBuf &b, const Wg &g)
{
    if (g.tid == 0) {
        *b.count = 0;
        *b.thresh = 0;
    }
    g.sync();
}

// Workspace view shared by the fused kernel and the stand-alone top-k.
struct TopkWs {
    uint32_t *status;
    uint32_t *arrive;     // [rows]
    uint32_t *cand_cnt;   // [rows]
    uint2 *cand;          // [rows][row_cap] (key, position)
    long long row_cap;    // entries per row (= max_model_len)
};

// Merge row `row`: all its segments have appended their candidates. Writes
// idx[row][0..k) (and vals) and returns the row's workspace state to zero.
static __device__ void row_merge(const CandBuf &b, const TopkWs &ws, long long row, uint32_t k,
                          uint32_t k_eff, int32_t *idx, float *vals, const Wg &g)
{
    __threadfence();
    cand_reset(b, g);
    const uint32_t n = __ldcg(ws.cand_cnt + row);
    const uint2 *src = ws.cand + row * ws.row_cap;
    constexpr uint32_t U = 4;
    for (uint32_t c0 = 0; c0 < n; c0 += 128 * U) {
        uint2 v[U];
#pragma unroll
        for (uint32_t u = 0; u < U; ++u) {
            const uint32_t e = c0 + u * 128 + g.tid;
            v[u] = e < n ? __ldcg(src + e) : make_uint2(0u, 0u);
        }
#pragma unroll
        for (uint32_t u = 0; u < U; ++u) {
            const uint32_t e = c0 + u * 128 + g.tid;
            if (c0 + u * 128 >= n)
                break;
            const uint32_t th = *b.thresh;
            cand_append(b, g, v[u].x, (int32_t)v[u].y, e < n && v[u].x >= th);
            if (k_eff > 0)
                cand_make_room(b, k_eff, g);
        }
    }
    g.sync();
    if (k_eff > 0 && *b.count > k_eff)
        cand_shrink(b, k_eff, g);
    g.sync();
    const uint32_t cnt = *b.count;
    int32_t *orow = idx + row * (long long)k;
    float *vrow = vals ? vals + row * (long long)k : nullptr;
    for (uint32_t e = g.tid; e < k; e += 128) {
        const bool have = e < cnt;
        orow[e] = have ? b.pos[e] : -1;
        if (vrow)
            vrow[e] = have ? order_key_f32(b.key[e]) : -__int_as_float(0x7f800000);
    }
    if (g.tid == 0) {
        ws.cand_cnt[row] = 0;
        ws.arrive[row] = 0;
    }
    g.sync();
}

// End of a segment of row `row` that covered seg_tiles of the row's
// total_tiles. Appends the buffer to the row's list; the work group that
// completes the row merges it. Leaves the buffer empty.
static __device__ void segment_finish(const CandBuf &b, const TopkWs &ws, long long row,
                               uint32_t seg_tiles, uint32_t total_tiles, uint32_t k,
                               uint32_t k_eff, int32_t *idx, float *vals, const Wg &g)
{
    g.sync();
    const uint32_t n = *b.count;
    if (g.tid == 0) {
        uint32_t base = atomicAdd(ws.cand_cnt + row, n);
        if ((long long)base + n > ws.row_cap) {
            atomicOr(ws.status, 0x8u);
            base = 0xFFFFFFFFu;
        }
        g.scr->bcast = base;
    }
    g.sync();
    const uint32_t base = g.scr->bcast;
    if (base != 0xFFFFFFFFu) {
        uint2 *dst = ws.cand + row * ws.row_cap + base;
        for (uint32_t e = g.tid; e < n; e += 128)
            __stcg(dst + e, make_uint2(b.key[e], (uint32_t)b.pos[e]));
    }
    __threadfence();
    g.sync();
    if (g.tid == 0) {
        const uint32_t old = atomicAdd(ws.arrive + row, seg_tiles);
        g.scr->bcast = (old + seg_tiles == total_tiles) ? 1u : 0u;
    }
    g.sync();
    const bool last = g.scr->bcast != 0;
    g.sync();
    if (last)
        row_merge(b, ws, row, k, k_eff, idx, vals, g);
    cand_reset(b, g);
}

}  // namespace pmqa
