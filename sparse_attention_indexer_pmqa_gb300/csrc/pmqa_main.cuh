// pmqa_main.cuh -- the persistent FP8 paged MQA-logits kernel for sm_103a.
//
// Definition (page "[Bug] aiter ops triton attention pa", section "Minimal
// reproduction", reference function `torch_ref`): for query row r = (i, j) and
// token t, logit = sum_h w[r][h] * relu(s_t * q[i][j][h] . k_t), -inf outside
// t < ctx_i, t <= ctx_i - next_n + j.
//
// One CTA per SM walks a contiguous range of (request, 128-token tile) work
// items, balanced by tile count over all requests. Warp roles:
//   warp 0      allocates TMEM; lane 0 issues tcgen05.mma
//   warp 1      lane 0 loads each request's q (TMA, 128B swizzle) and weights
//               (bulk copy) into a query slot
//   warps 2..5  gather + repack, 32 tokens of every tile each: the block table
//               is read three tiles ahead; every 132-byte row is fetched as its
//               16-byte aligned 144-byte window with 16-byte cp.async into a
//               per-warp staging ring (several tiles in flight); once a tile
//               has landed the warp moves each row's 32 fp8 words (shifted by
//               the row's 0/4/8/12-byte misalignment) into the 128B-swizzled
//               K-major operand tile and its fp32 scale into a scale ring
//   warps 6..   epilogue work groups (1 or 2 x 4 warps): tcgen05.ld of the
//               fp32 scores (one token per thread, all heads of a row in
//               registers), relu * weight head sum, scale, mask; full logits
//               rows and/or the compact logits + an 11-bit key histogram per
//               row for the selection kernel.
// The MMA computes D[token][(j,h)] = K_tile[128 x 128] * Q[(j,h) x 128]^T with
// tokens as M = 128 and N = next_n * heads, fp8 e4m3 in, fp32 accumulate in
// TMEM (NBUF accumulators). All hand-offs are mbarriers; waits are bounded.
#pragma once

#include <cuda.h>

#include <cstdint>

#include "pmqa_ptx.cuh"

namespace pmqa {

constexpr uint32_t kFullMask = 0xFFFFFFFFu;
constexpr int kTileTokens = 128;
constexpr int kHeadDim = 128;
constexpr int kKvRowBytes = kHeadDim + 4;
constexpr int kPRWarps = 4;
constexpr int kFirstPRWarp = 2;
constexpr int kFirstEpiWarp = kFirstPRWarp + kPRWarps;
constexpr uint32_t kStageBytes = kTileTokens * kHeadDim;  // 16 KB operand tile
constexpr uint32_t kWinBytes = 144;                        // aligned window of one row
constexpr uint32_t kWarpSlotBytes = 32 * kWinBytes;        // one warp's rows of a tile
constexpr int kHistBins = 2048;                            // top 11 bits of the order key
constexpr int kHistShift = 21;

struct MainArgs {
    CUtensorMap tmap_q;  // q as [bs * N rows, 128 bytes], 128B swizzle, box [128, q_box]
    const uint8_t *q;
    const uint8_t *kv;
    const float *w;
    const int32_t *ctx_lens;
    const int32_t *bt;
    long long num_blocks;
    long long pool_bytes;  // num_blocks * block_size * 132
    int bs, nn, P, W, mml;
    float *logits;     // full rows [rows, mml], or null
    float *clogits;    // compact logits (valid positions only) for the selection, or null
    uint32_t *hist;    // per-row key histograms [rows, 2048], or null
    uint32_t *status;
    int l2_policy;     // KV stream: 0 evict_first, 1 evict_normal, 2 evict_last
    // shared-memory / pipeline layout, computed on the host
    int N, S, SG, NBUF, QS, RS, cols, tmem_cols, E, rpw;
    int q_box;  // rows per q TMA box: N / ceil(N / 256)
    uint32_t off_op, off_q, off_w, off_scale, off_meta, off_bar, off_hist, smem_bytes;
};

struct CtaCtl {
    long long red[16];
    int wsum[16];
    long long start, count;
    int i0, m0;
    int abort;
    uint32_t tmem_base;
};

// f32 -> u32 with a > b  <=>  key(a) > key(b); -0 is folded onto +0.
__device__ __forceinline__ uint32_t f32_order_key(float f)
{
    uint32_t u = __float_as_uint(f == 0.0f ? 0.0f : f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ int clamp_ctx(int c, long long lim)
{
    return c < 0 ? 0 : (c > lim ? (int)lim : c);
}

__device__ __forceinline__ int ctx_of(const MainArgs &a, int i)
{
    const long long lim = min((long long)a.mml, (long long)a.W * a.P);
    return clamp_ctx(__ldg(a.ctx_lens + i), lim);
}

// Number of positions of draft row j that the causal window admits.
__device__ __forceinline__ int valid_len(int ctx, int nn, int j)
{
    const int v = ctx - nn + j + 1;
    return v < 0 ? 0 : (v > ctx ? ctx : v);
}

// Split the items' total length evenly over the grid (every thread calls).
template <class LenFn>
__device__ void balance_schedule(int n_items, LenFn len_of, CtaCtl &c)
{
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5, nw = blockDim.x >> 5;
    long long loc = 0;
    for (int i = tid; i < n_items; i += blockDim.x)
        loc += len_of(i);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        loc += __shfl_xor_sync(kFullMask, loc, o);
    if (lane == 0)
        c.red[wid] = loc;
    __syncthreads();
    if (tid == 0) {
        long long t = 0;
        for (int w = 0; w < nw; ++w)
            t += c.red[w];
        c.start = (long long)blockIdx.x * t / gridDim.x;
        c.count = (long long)(blockIdx.x + 1) * t / gridDim.x - c.start;
        c.i0 = n_items;
        c.m0 = 0;
    }
    __syncthreads();
    const long long start = c.start;
    long long running = 0;
    for (int base = 0; base < n_items; base += blockDim.x) {
        const int i = base + tid;
        const int nt = i < n_items ? (int)len_of(i) : 0;
        int x = nt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(kFullMask, x, o);
            if (lane >= o)
                x += y;
        }
        if (lane == 31)
            c.wsum[wid] = x;
        __syncthreads();
        long long woff = 0, chunk = 0;
        for (int w = 0; w < nw; ++w) {
            woff += w < wid ? c.wsum[w] : 0;
            chunk += c.wsum[w];
        }
        const long long incl = running + woff + x, excl = incl - nt;
        if (nt > 0 && excl <= start && start < incl) {
            c.i0 = i;
            c.m0 = (int)(start - excl);
        }
        running += chunk;
        __syncthreads();
    }
}

// Walks (request, tile) pairs in order, skipping empty requests.
struct TileIter {
    int i, m, nt, ctx;
    __device__ void init(const MainArgs &a, int i0, int m0)
    {
        i = i0;
        m = m0;
        ctx = i < a.bs ? ctx_of(a, i) : 0;
        nt = (ctx + kTileTokens - 1) / kTileTokens;
    }
    __device__ void next(const MainArgs &a)
    {
        if (++m < nt)
            return;
        m = 0;
        do {
            if (++i >= a.bs) {
                nt = 0;
                ctx = 0;
                return;
            }
            ctx = ctx_of(a, i);
            nt = (ctx + kTileTokens - 1) / kTileTokens;
        } while (nt == 0);
    }
};

struct Bars {
    uint64_t *op_full, *op_empty, *tfull, *tempty, *qfull, *qempty, *sfull, *done;
    __device__ Bars(const MainArgs &a, uint8_t *smem)
    {
        op_full = reinterpret_cast<uint64_t *>(smem + a.off_bar);
        op_empty = op_full + a.S;
        tfull = op_empty + a.S;
        tempty = tfull + a.NBUF;
        qfull = tempty + a.NBUF;
        qempty = qfull + a.QS;
        sfull = qempty + a.QS;
        done = sfull + a.RS;
    }
};

__device__ __forceinline__ void cp_async_wait_upto(int n)
{
    switch (n) {
    case 0: cp_async_wait_group<0>(); break;
    case 1: cp_async_wait_group<1>(); break;
    case 2: cp_async_wait_group<2>(); break;
    case 3: cp_async_wait_group<3>(); break;
    case 4: cp_async_wait_group<4>(); break;
    case 5: cp_async_wait_group<5>(); break;
    case 6: cp_async_wait_group<6>(); break;
    case 7: cp_async_wait_group<7>(); break;
    case 8: cp_async_wait_group<8>(); break;
    case 9: cp_async_wait_group<9>(); break;
    default: cp_async_wait_group<10>(); break;
    }
}

__device__ __forceinline__ void raise_abort(const MainArgs &a, CtaCtl &c)
{
    c.abort = 1;
    atomicOr(a.status, 0x4u);
}

// ---------------------------------------------------------------- query loader

static __device__ void qload_role(const MainArgs &a, uint8_t *smem, CtaCtl &c)
{
    const Bars B(a, smem);
    const int N = a.N, count = (int)c.count;
    TileIter it;
    it.init(a, c.i0, c.m0);
    uint32_t req = 0;
    for (int kk = 0; kk < count; ++kk) {
        if (kk == 0 || it.m == 0) {
            const uint32_t qs = req % a.QS;
            if (!mbar_wait(&B.qempty[qs], ((req / a.QS) & 1) ^ 1, &c.abort)) {
                raise_abort(a, c);
                return;
            }
            mbar_arrive_expect_tx(&B.qfull[qs], (uint32_t)N * (kHeadDim + 4));
            const uint32_t qdst = smem_u32(smem + a.off_q + qs * (uint32_t)N * kHeadDim);
            // boxes of q_box rows tile the request's N rows exactly (N = nbox * q_box)
            for (int nc = 0; nc * a.q_box < N; ++nc)
                tma_load_2d(qdst + nc * a.q_box * kHeadDim, &a.tmap_q, 0, it.i * N + nc * a.q_box,
                            &B.qfull[qs]);
            bulk_load(smem_u32(smem + a.off_w + qs * (uint32_t)N * 4), a.w + (long long)it.i * N,
                      (uint32_t)N * 4, &B.qfull[qs]);
            ++req;
        }
        it.next(a);
    }
}

// ---------------------------------------------------------------- gather + repack

// Block-table entry of this lane's token in tile `t` (-1: no token).
__device__ __forceinline__ int32_t table_entry(const MainArgs &a, const TileIter &t, int lane_tok)
{
    const int tok = t.m * kTileTokens + lane_tok;
    if (t.nt == 0 || tok >= t.ctx)
        return -1;
    return __ldg(a.bt + (long long)t.i * a.W + tok / a.P);
}

static __device__ void gather_role(const MainArgs &a, uint8_t *smem, CtaCtl &c, int pw)
{
    const Bars B(a, smem);
    const int lane = threadIdx.x & 31;
    const int lane_tok = pw * 32 + lane;  // this lane's token row within a tile
    const uint64_t pol = a.l2_policy == 0   ? l2_evict_first_policy()
                         : a.l2_policy == 2 ? l2_evict_last_policy()
                                            : l2_evict_normal_policy();
    const int count = (int)c.count, SG = a.SG;
    uint8_t *stg = smem + (uint32_t)pw * (uint32_t)SG * kWarpSlotBytes;
    // per-lane metadata of the tiles in the staging ring: bit 2 = row present,
    // bits 0-1 = misalignment of the row in 4-byte words
    uint8_t *meta = smem + a.off_meta + (uint32_t)pw * (uint32_t)SG * 32u;
    float *sring = reinterpret_cast<float *>(smem + a.off_scale);

    TileIter iss, tab;
    iss.init(a, c.i0, c.m0);
    tab = iss;
    // block-table entries of the next three tiles to issue
    int32_t e0 = -1, e1 = -1, e2 = -1;
    if (count > 0)
        e0 = table_entry(a, tab, lane_tok);
    if (count > 1) {
        tab.next(a);
        e1 = table_entry(a, tab, lane_tok);
    }
    if (count > 2) {
        tab.next(a);
        e2 = table_entry(a, tab, lane_tok);
    }

    auto issue = [&](int ki) {
        const int32_t b = e0;
        e0 = e1;
        e1 = e2;
        if (ki + 3 < count) {
            tab.next(a);
            e2 = table_entry(a, tab, lane_tok);
        }
        const int t = iss.m * kTileTokens + lane_tok;
        long long w0 = 0;
        uint32_t m = 0;
        bool tail_ok = true;
        if (t < iss.ctx) {
            if (b >= 0 && (long long)b < a.num_blocks) {
                const long long o = ((long long)b * a.P + (t % a.P)) * kKvRowBytes;
                w0 = o & ~15ll;
                m = 4u | (uint32_t)((o >> 2) & 3);
                tail_ok = w0 + kWinBytes <= a.pool_bytes;
            } else {
                atomicOr(a.status, 0x1u);
            }
        }
        const int slot = ki % SG;
        meta[slot * 32 + lane] = (uint8_t)m;
        const uint32_t sb = smem_u32(stg + (uint32_t)slot * kWarpSlotBytes);
#pragma unroll
        for (int qq = 0; qq < 9; ++qq) {
            const int e = qq * 32 + lane;
            const int j = e / 9, ch = e - j * 9;
            const long long wj = __shfl_sync(kFullMask, w0, j);
            const uint32_t mj = __shfl_sync(kFullMask, m, j);
            const bool tj = __shfl_sync(kFullMask, tail_ok, j);
            if (mj & 4u) {
                const uint32_t dst = sb + (uint32_t)j * kWinBytes + (uint32_t)ch * 16u;
                const uint8_t *src = a.kv + wj + ch * 16;
                if (ch < 8 || tj) {
                    cp_async_16_hint(dst, src, pol);
                } else {
                    // last row of the pool: never read past its end
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) {
                        const bool in = wj + 128 + 4 * (q4 + 1) <= a.pool_bytes;
                        cp_async_4(dst + 4 * q4, in ? src + 4 * q4 : a.kv, in ? 4u : 0u, pol);
                    }
                }
            }
        }
        cp_async_commit();
        iss.next(a);
    };

    // prologue: SG - 1 tiles in flight before the first repack. Tile k is this
    // thread's cp.async group k, so tile kk has landed once at most
    // (issued - kk - 1) groups are still pending.
    int ki = 0;
    for (; ki < SG - 1 && ki < count; ++ki)
        issue(ki);
    bool ok = true;
    for (int kk = 0; kk < count; ++kk) {
        if (ki < count) {
            issue(ki);
            ++ki;
        }
        cp_async_wait_upto(ki - kk - 1);
        __syncwarp();
        const int s = kk % a.S;
        if (!mbar_wait(&B.op_empty[s], ((kk / a.S) & 1) ^ 1, &c.abort)) {
            ok = false;
            break;
        }
        const int slot = kk % SG;
        const uint8_t *sb = stg + (uint32_t)slot * kWarpSlotBytes;
        const uint32_t my_m = meta[slot * 32 + lane];
        uint8_t *ob = smem + a.off_op + (uint32_t)s * kStageBytes;
        const uint32_t chunk_off = (uint32_t)(lane & 3) * 4u;
        const uint32_t chunk_id = (uint32_t)lane >> 2;
#pragma unroll 8
        for (int j = 0; j < 32; ++j) {
            const uint32_t mj = __shfl_sync(kFullMask, my_m, j);
            uint32_t v = 0;
            if (mj & 4u)
                v = *reinterpret_cast<const uint32_t *>(sb + j * kWinBytes +
                                                        ((mj & 3u) + (uint32_t)lane) * 4u);
            const uint32_t r = (uint32_t)(pw * 32 + j);
            *reinterpret_cast<uint32_t *>(ob + r * 128u + ((chunk_id ^ (r & 7u)) << 4) +
                                          chunk_off) = v;
        }
        float sc = 0.0f;
        if (my_m & 4u)
            sc = *reinterpret_cast<const float *>(sb + lane * kWinBytes + ((my_m & 3u) + 32u) * 4u);
        sring[(kk % a.RS) * kTileTokens + lane_tok] = sc;
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            mbar_arrive(&B.op_full[s]);
            mbar_arrive(&B.sfull[kk % a.RS]);
        }
    }
    cp_async_wait_all();
    if (!ok)
        raise_abort(a, c);
}

// ---------------------------------------------------------------- MMA issue

static __device__ void mma_role(const MainArgs &a, uint8_t *smem, CtaCtl &c)
{
    const Bars B(a, smem);
    const int N = a.N, count = (int)c.count;
    const uint32_t tbase = c.tmem_base;
    TileIter it;
    it.init(a, c.i0, c.m0);
    uint32_t req = 0;
    bool ok = true;
    for (int kk = 0; kk < count; ++kk) {
        const int s = kk % a.S, b = kk % a.NBUF;
        const uint32_t qs = req % a.QS;
        const bool first = kk == 0 || it.m == 0;
        if (first && !mbar_wait(&B.qfull[qs], (req / a.QS) & 1, &c.abort)) {
            ok = false;
            break;
        }
        if (!mbar_wait(&B.op_full[s], (kk / a.S) & 1, &c.abort) ||
            !mbar_wait(&B.tempty[b], ((kk / a.NBUF) & 1) ^ 1, &c.abort)) {
            ok = false;
            break;
        }
        tc_fence_after_sync();
        const uint32_t abase = smem_u32(smem + a.off_op + (uint32_t)s * kStageBytes);
        const uint32_t bbase = smem_u32(smem + a.off_q + qs * (uint32_t)N * kHeadDim);
#pragma unroll
        for (int k4 = 0; k4 < kHeadDim / 32; ++k4) {
            const uint64_t ad = sw128_kmajor_desc(abase + k4 * 32);
            for (int nc = 0; nc * 256 < N; ++nc) {
                const int nw = min(256, N - nc * 256);
                const uint64_t bd = sw128_kmajor_desc(bbase + nc * 256 * kHeadDim + k4 * 32);
                umma_e4m3(tbase + (uint32_t)(b * a.cols + nc * 256), ad, bd,
                          idesc_e4m3_f32(128, nw), k4 > 0 ? 1u : 0u);
            }
        }
        umma_commit(&B.op_empty[s]);
        umma_commit(&B.tfull[b]);
        if (kk == count - 1 || it.m == it.nt - 1) {
            umma_commit(&B.qempty[qs]);
            ++req;
        }
        it.next(a);
    }
    if (!ok)
        raise_abort(a, c);
    umma_commit(B.done);
    if (!mbar_wait(B.done, 0, nullptr))
        atomicOr(a.status, 0x4u);
}

// ---------------------------------------------------------------- epilogue

// Scores of rows j = g, g + E, ... for this thread's token: TMEM columns
// [j*H, j*H + H) of the buffer. Releases the TMEM buffer after the last load.
template <int H>
__device__ __forceinline__ void epi_rows(uint32_t taddr, const float *wsl, float sc, int g, int E,
                                         int nn, float (&logit)[2], uint64_t *tempty_bar,
                                         int lane)
{
    constexpr int CH = H >= 32 ? 32 : 16;  // columns per chunk
    constexpr int CPR = H / CH;            // chunks per row
    constexpr int MAXC = 2 * CPR;
    const int rows_here = (nn - g + E - 1) / E;  // 1 or 2
    const int nchunks = rows_here * CPR;
    const bool all_pos = __all_sync(kFullMask, !(sc < 0.0f));
    const uint32_t flip = sc < 0.0f ? 0x80000000u : 0u;
    const float mag = fabsf(sc);
    uint32_t buf[2][CH];
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    logit[0] = logit[1] = 0.f;

    auto issue = [&](int c, uint32_t *dst) {
        const int u = c / CPR, part = c % CPR;
        const int j = g + u * E;
        const uint32_t col = (uint32_t)(j * H + part * CH);
#pragma unroll
        for (int q = 0; q < CH / 16; ++q)
            tmem_ld16(taddr + col + q * 16, dst + q * 16);
    };
    issue(0, buf[0]);
    tmem_ld_wait();
#pragma unroll
    for (int q = 0; q < CH / 16; ++q)
        reg_fence16(buf[0] + q * 16);
#pragma unroll
    for (int c = 0; c < MAXC; ++c) {
        if (c >= nchunks)
            break;
        if (c + 1 < nchunks) {
            issue(c + 1, buf[(c + 1) & 1]);
        } else {
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(tempty_bar);
        }
        const int u = c / CPR, part = c % CPR;
        const int j = g + u * E;
        const float4 *w4 = reinterpret_cast<const float4 *>(wsl + j * H + part * CH);
        const uint32_t *x = buf[c & 1];
        if (all_pos) {
#pragma unroll
            for (int h = 0; h < CH; h += 4) {
                const float4 wv = w4[h / 4];
                acc[0] = fmaf(wv.x, fmaxf(__uint_as_float(x[h + 0]), 0.f), acc[0]);
                acc[1] = fmaf(wv.y, fmaxf(__uint_as_float(x[h + 1]), 0.f), acc[1]);
                acc[2] = fmaf(wv.z, fmaxf(__uint_as_float(x[h + 2]), 0.f), acc[2]);
                acc[3] = fmaf(wv.w, fmaxf(__uint_as_float(x[h + 3]), 0.f), acc[3]);
            }
        } else {
#pragma unroll
            for (int h = 0; h < CH; h += 4) {
                const float4 wv = w4[h / 4];
                acc[0] = fmaf(wv.x, fmaxf(__uint_as_float(x[h + 0] ^ flip), 0.f), acc[0]);
                acc[1] = fmaf(wv.y, fmaxf(__uint_as_float(x[h + 1] ^ flip), 0.f), acc[1]);
                acc[2] = fmaf(wv.z, fmaxf(__uint_as_float(x[h + 2] ^ flip), 0.f), acc[2]);
                acc[3] = fmaf(wv.w, fmaxf(__uint_as_float(x[h + 3] ^ flip), 0.f), acc[3]);
            }
        }
        if (part == CPR - 1) {
            const float v = ((acc[0] + acc[1]) + (acc[2] + acc[3])) * mag;
            if (u == 0)
                logit[0] = v;
            else
                logit[1] = v;
            acc[0] = acc[1] = acc[2] = acc[3] = 0.f;
        }
        if (c + 1 < nchunks) {
            tmem_ld_wait();
#pragma unroll
            for (int q = 0; q < CH / 16; ++q)
                reg_fence16(buf[(c + 1) & 1] + q * 16);
        }
    }
}

template <int H>
static __device__ void epilogue_role(const MainArgs &a, uint8_t *smem, CtaCtl &c, int g, int we)
{
    const Bars B(a, smem);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, qd = warp & 3;
    const int r = qd * 32 + lane;  // token row of the tile = TMEM lane
    const int N = a.N, nn = a.nn, E = a.E;
    const float NEG_INF = -__int_as_float(0x7f800000);
    const uint32_t wtid = (uint32_t)(we * 32 + lane);
    const uint32_t bar_id = 1u + (uint32_t)g;
    const bool want_hist = a.hist != nullptr;
    uint32_t *shist = reinterpret_cast<uint32_t *>(smem + a.off_hist) +
                      (uint32_t)g * (uint32_t)a.rpw * kHistBins;
    const uint64_t keep_pol = l2_evict_last_policy();
    const int rows_here = (nn - g + E - 1) / E;

    // -inf beyond the last tile of each row: this CTA's share of every row
    if (a.logits) {
        const int etid = g * 128 + (int)wtid, ethr = E * 128;
        for (int rr = 0; rr < a.bs * nn; ++rr) {
            const int cx = ctx_of(a, rr / nn);
            const long long lo =
                min((long long)(cx + kTileTokens - 1) / kTileTokens * kTileTokens, (long long)a.mml);
            const long long L = a.mml - lo;
            const long long s0 = lo + L * blockIdx.x / gridDim.x;
            const long long s1 = lo + L * (blockIdx.x + 1) / gridDim.x;
            float *row = a.logits + (long long)rr * a.mml;
            for (long long t = s0 + etid; t < s1; t += ethr)
                row[t] = NEG_INF;
        }
    }
    if (want_hist) {
        for (int e = (int)wtid; e < a.rpw * kHistBins; e += 128)
            shist[e] = 0;
        named_bar_sync(bar_id, 128);
    }

    const int count = (int)c.count;
    TileIter it;
    it.init(a, c.i0, c.m0);
    uint32_t req = 0;
    // Waits that fail (abort or time limit) skip the data work but keep the
    // work group's barrier schedule, so no warp is left waiting on another.
    for (int kk = 0; kk < count; ++kk) {
        const int b = kk % a.NBUF;
        const uint32_t qs = req % a.QS;
        const bool first = kk == 0 || it.m == 0;
        bool ok = true;
        if (first)
            ok = mbar_wait(&B.qfull[qs], (req / a.QS) & 1, &c.abort);
        const int sri = kk % a.RS;
        ok = ok && mbar_wait(&B.sfull[sri], (uint32_t)(kk / a.RS) & 1u, &c.abort) &&
             mbar_wait(&B.tfull[b], (kk / a.NBUF) & 1, &c.abort);
        if (ok) {
            tc_fence_after_sync();
            const float sc =
                reinterpret_cast<const float *>(smem + a.off_scale)[sri * kTileTokens + r];
            const int t = it.m * kTileTokens + r;
            const float *wsl =
                reinterpret_cast<const float *>(smem + a.off_w + qs * (uint32_t)N * 4);
            const uint32_t taddr =
                c.tmem_base + ((uint32_t)(qd * 32) << 16) + (uint32_t)(b * a.cols);
            float logit[2];
            epi_rows<H>(taddr, wsl, sc, g, E, nn, logit, &B.tempty[b], lane);
            for (int u = 0; u < rows_here; ++u) {
                const int j = g + u * E;
                const long long row = (long long)it.i * nn + j;
                const bool valid = t < valid_len(it.ctx, nn, j);
                if (a.logits && t < a.mml)
                    a.logits[row * a.mml + t] = valid ? logit[u] : NEG_INF;
                if (a.clogits && valid)
                    st_global_hint(a.clogits + row * a.mml + t, logit[u], keep_pol);
                if (want_hist) {
                    const uint32_t bin = f32_order_key(logit[u]) >> kHistShift;
                    const uint32_t grp =
                        __match_any_sync(kFullMask, valid ? bin : 0x10000u + (uint32_t)lane);
                    if (valid && (__ffs(grp) - 1) == lane)
                        atomicAdd(shist + u * kHistBins + bin, (uint32_t)__popc(grp));
                }
            }
        } else {
            raise_abort(a, c);
        }
        if (kk == count - 1 || it.m == it.nt - 1) {
            if (want_hist) {
                named_bar_sync(bar_id, 128);
                for (int u = 0; u < rows_here; ++u) {
                    const long long row = (long long)it.i * nn + g + u * E;
                    for (int e = (int)wtid; e < kHistBins; e += 128) {
                        const uint32_t v = shist[u * kHistBins + e];
                        if (v) {
                            atomicAdd(a.hist + row * kHistBins + e, v);
                            shist[u * kHistBins + e] = 0;
                        }
                    }
                }
                named_bar_sync(bar_id, 128);
            }
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&B.qempty[qs]);
            ++req;
        }
        it.next(a);
    }
}

// ---------------------------------------------------------------- kernel

constexpr int kMaxThreads = 32 * (kFirstEpiWarp + 8);

template <int H>
__global__ void __launch_bounds__(kMaxThreads, 1)
    pmqa_main_kernel(const __grid_constant__ MainArgs a)
{
    extern __shared__ uint8_t smem_raw[];
    __shared__ CtaCtl ctl;
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int warp = threadIdx.x >> 5;

    if (threadIdx.x == 0) {
        ctl.abort = 0;
        const Bars B(a, smem);
        for (int s = 0; s < a.S; ++s) {
            mbar_init(&B.op_full[s], kPRWarps);
            mbar_init(&B.op_empty[s], 1);
        }
        for (int b = 0; b < a.NBUF; ++b) {
            mbar_init(&B.tfull[b], 1);
            mbar_init(&B.tempty[b], 4 * a.E);
        }
        for (int q = 0; q < a.QS; ++q) {
            mbar_init(&B.qfull[q], 1);
            mbar_init(&B.qempty[q], 1 + 4 * a.E);
        }
        for (int q = 0; q < a.RS; ++q)
            mbar_init(&B.sfull[q], kPRWarps);
        mbar_init(B.done, 1);
        mbar_init_fence();
    }
    __syncwarp();
    if (warp == 0)
        tmem_alloc(&ctl.tmem_base, (uint32_t)a.tmem_cols);

    balance_schedule(
        a.bs, [&](int i) { return (long long)((ctx_of(a, i) + kTileTokens - 1) / kTileTokens); },
        ctl);
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

    if (warp == 0) {
        if ((threadIdx.x & 31) == 0)
            mma_role(a, smem, ctl);
        __syncwarp();
    } else if (warp == 1) {
        if ((threadIdx.x & 31) == 0)
            qload_role(a, smem, ctl);
        __syncwarp();
    } else if (warp < kFirstEpiWarp) {
        gather_role(a, smem, ctl, warp - kFirstPRWarp);
    } else {
        const int e = warp - kFirstEpiWarp;
        epilogue_role<H>(a, smem, ctl, e >> 2, e & 3);
    }

    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    __syncwarp();
    if (warp == 0)
        tmem_dealloc(ctl.tmem_base, (uint32_t)a.tmem_cols);
}

}  // namespace pmqa
