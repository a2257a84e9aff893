// pmqa_topk_kernel.cuh -- stand-alone per-row top-k over logits rows in HBM.
//
// Row (i, j) keeps the min(k, valid_len) largest entries among t < valid_len =
// clamp(ctx_i - next_n + j + 1, 0, ctx_i), as in the `test` driver on the page
// "[Bug] aiter ops triton attention pa" (section "Minimal reproduction"), which
// takes torch.topk with k = min(2048, ctx) after the causal mask. Entries past
// valid_len are never read.
//
// Each 128-thread CTA takes a contiguous, tile-balanced range of (row,
// 128-position tile) items, streams them through the candidate buffer of
// pmqa_topk_wg.cuh and finishes each row segment; the CTA completing a row
// merges it. Loads run eight tiles ahead of the selection.
#pragma once

#include <cstdint>

#include "pmqa_main.cuh"
#include "pmqa_topk_wg.cuh"

namespace pmqa {

struct TopkArgs {
    const float *logits;
    const int32_t *ctx_lens;
    int bs, nn, mml, k;
    int32_t *idx;
    float *vals;
    TopkWs ws;
    int cap;
};

__device__ __forceinline__ int topk_row_len(const TopkArgs &a, int r)
{
    const int c = clamp_ctx(__ldg(a.ctx_lens + r / a.nn), (long long)a.mml);
    return valid_len(c, a.nn, r % a.nn);
}

struct RowIter {
    int r, m, nt, len;
    __device__ void init(const TopkArgs &a, int r0, int m0)
    {
        r = r0;
        m = m0;
        len = r < a.bs * a.nn ? topk_row_len(a, r) : 0;
        nt = (len + kTileTokens - 1) / kTileTokens;
    }
    __device__ void next(const TopkArgs &a)
    {
        if (++m < nt)
            return;
        m = 0;
        do {
            if (++r >= a.bs * a.nn) {
                nt = 0;
                len = 0;
                return;
            }
            len = topk_row_len(a, r);
            nt = (len + kTileTokens - 1) / kTileTokens;
        } while (nt == 0);
    }
};

__global__ void __launch_bounds__(128) pmqa_topk_kernel(const __grid_constant__ TopkArgs a)
{
    extern __shared__ __align__(16) uint8_t tsm[];
    __shared__ CtaCtl ctl;
    const int rows = a.bs * a.nn;
    const float NEG_INF = -__int_as_float(0x7f800000);

    Wg wg;
    wg.tid = threadIdx.x;
    wg.lane = threadIdx.x & 31;
    wg.warp = threadIdx.x >> 5;
    wg.bar = 1;
    wg.scr = reinterpret_cast<WgScratch *>(tsm);
    CandBuf cb;
    cb.count = reinterpret_cast<uint32_t *>(tsm + sizeof(WgScratch));
    cb.thresh = cb.count + 1;
    cb.key = reinterpret_cast<uint32_t *>(tsm + sizeof(WgScratch) + 16);
    cb.pos = reinterpret_cast<int32_t *>(cb.key + a.cap);
    cb.cap = (uint32_t)a.cap;

    balance_schedule(
        rows, [&](int r) { return (long long)((topk_row_len(a, r) + kTileTokens - 1) / kTileTokens); },
        ctl);
    if (blockIdx.x == 0) {
        for (int i = threadIdx.x; i < a.bs; i += blockDim.x) {
            const int c = __ldg(a.ctx_lens + i);
            if (c < 0 || c > a.mml)
                atomicOr(a.ws.status, 0x2u);
        }
        // rows with nothing to select: no segment will merge them
        for (int r = 0; r < rows; ++r) {
            if (topk_row_len(a, r) > 0)
                continue;
            for (int e = threadIdx.x; e < a.k; e += blockDim.x) {
                a.idx[(long long)r * a.k + e] = -1;
                if (a.vals)
                    a.vals[(long long)r * a.k + e] = NEG_INF;
            }
        }
    }
    cand_reset(cb, wg);

    const int count = (int)ctl.count;
    RowIter it;
    it.init(a, ctl.i0, ctl.m0);
    uint32_t seg_tiles = 0;
    constexpr int U = 8;
    for (int k0 = 0; k0 < count; k0 += U) {
        float v[U];
        int vr[U], vm[U], vlen[U], vnt[U];
        RowIter pre = it;
#pragma unroll
        for (int u = 0; u < U; ++u) {
            vr[u] = pre.r;
            vm[u] = pre.m;
            vlen[u] = pre.len;
            vnt[u] = pre.nt;
            const int t = pre.m * kTileTokens + (int)threadIdx.x;
            v[u] = (k0 + u < count && t < pre.len)
                       ? __ldcs(a.logits + (long long)pre.r * a.mml + t)
                       : 0.f;
            if (k0 + u < count)
                pre.next(a);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (k0 + u >= count)
                break;
            const int t = vm[u] * kTileTokens + (int)threadIdx.x;
            const uint32_t key = f32_order_key(v[u]);
            const uint32_t vl = (uint32_t)vlen[u];
            const uint32_t k_eff = vl < (uint32_t)a.k ? vl : (uint32_t)a.k;
            cand_append(cb, wg, key, t, t < vlen[u] && key >= *cb.thresh);
            cand_make_room(cb, (uint32_t)a.k, wg);
            ++seg_tiles;
            if (k0 + u == count - 1 || vm[u] == vnt[u] - 1) {
                segment_finish(cb, a.ws, vr[u], seg_tiles, (uint32_t)vnt[u], (uint32_t)a.k, k_eff,
                               a.idx, a.vals, wg);
                seg_tiles = 0;
            }
        }
        it = pre;
    }
}

}  // namespace pmqa
