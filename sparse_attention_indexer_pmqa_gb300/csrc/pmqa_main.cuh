// pmqa_main.cuh -- the persistent FP8 paged MQA-logits kernel for sm_103a.
//
// Definition (page "[Bug] aiter ops triton attention pa", section "Minimal
// reproduction", reference function `torch_ref`): for query row r = (i, j) and
// token t, logit = sum_h w[r][h] * relu(s_t * q[i][j][h] . k_t), -inf outside
// t < ctx_i, t <= ctx_i - next_n + j.
//
// One CTA per SM walks a contiguous range of (request, 128-token tile) work
// items, balanced by tile count over all requests. Warp roles:
//   warp 14     lane 0 issues tcgen05.mma (warp 0 allocates TMEM)
//   warp 8      lane 0 loads each request's q (TMA, 128B swizzle) and weights
//               (bulk copy) into a query slot
//   gather warps (0, 1, 4, 5), 32 tokens of every tile each: block-table entries
//               arrive by cp.async a ring-depth ahead; every 132-byte row is
//               fetched as its 16-byte aligned 144-byte window with 16-byte
//               cp.async into the staging ring, whose mbarrier completes when
//               the copies land (several tiles in flight, no blocking)
//   repack warps (2, 3, 6, 7), 32 tokens of every tile each: once a tile has landed,
//               each row's 32 fp8 words (shifted by the row's 0/4/8/12-byte
//               misalignment) go into the 128B-swizzled K-major operand tile
//               and its fp32 scale into a scale ring
//   warps 10..13 the epilogue work group: tcgen05.ld of the fp32 scores (one
//               token per thread, all heads of a row in registers), relu *
//               weight head sum, scale, mask for every draft row; full logits
//               rows and/or the compact logits + an 11-bit key histogram per
//               row for the selection kernel.
// The MMA computes D[token][(j,h)] = K_tile[128 x 128] * Q[(j,h) x 128]^T with
// tokens as M = 128 and N = next_n * heads, fp8 e4m3 in, fp32 accumulate in
// TMEM (NBUF accumulators). All hand-offs are mbarriers; waits are bounded.
// A warp runs on sub-partition warp % 4. Gather and repack warps sit on
// different sub-partitions (gather on 0 and 1, repack on 2 and 3), so each
// sub-partition's instruction cache holds the code of at most two busy roles,
// and the MMA issue (on 2) does not queue behind the gathers' global copies;
// the epilogue needs one warp on every sub-partition (warp w reads TMEM lanes
// 32 * (w % 4) ...). Warps 9 and 15 have no role.
#pragma once

#include <cuda.h>

#include <cstdint>

#include "pmqa_ptx.cuh"

namespace pmqa {

constexpr uint32_t kFullMask = 0xFFFFFFFFu;
constexpr int kTileTokens = 128;
constexpr int kHeadDim = 128;
constexpr int kKvRowBytes = kHeadDim + 4;
constexpr int kGatherWarps = 4;
constexpr int kRepackWarps = 4;
constexpr int kTokPerWarp = kTileTokens / kGatherWarps;    // 32 tokens per gather/repack warp
constexpr int kFirstEpiWarp = 10;
constexpr int kMmaWarp = 14;
constexpr int kQloadWarp = 8;

// Row block (0..3) of a gather warp (0, 1, 4, 5) or a repack warp (2, 3, 6, 7).
__device__ __forceinline__ int row_block_of(int warp) { return (warp & 1) | ((warp >> 2) & 1) << 1; }
constexpr int kMaxRows = 4;                                // draft rows per request
constexpr uint32_t kStageBytes = kTileTokens * kHeadDim;  // 16 KB operand tile
constexpr uint32_t kWinBytes = 144;                        // aligned window of one row
constexpr uint32_t kSlotBytes = kTileTokens * kWinBytes;   // one staging slot (18 KB)
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
    int page_mode;     // block_size % 4 == 0: rows move as page runs by bulk copy
    // shared-memory / pipeline layout, computed on the host
    int N, S, SG, NBUF, QS, RS, cols, tmem_cols;
    int q_box;  // rows per q TMA box: N / ceil(N / 256)
    uint32_t off_op, off_q, off_w, off_scale, off_meta, off_tab, off_bar, off_hist, smem_bytes;
};

constexpr int kCtxCache = 512;  // context lengths of the CTA's first requests, in smem

struct CtaCtl {
    long long red[32];  // per-warp partial sums (up to 32 warps)
    int wsum[32];
    long long start, count;
    int i0, m0;
    int abort;
    uint32_t tmem_base;
    int ctx[kCtxCache];  // clamped context of request i0 + n, n < kCtxCache
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

// Walks (request, tile) pairs in order, skipping empty requests. Context
// lengths come from the CTA's shared-memory cache while it covers them. Every
// field the walk needs is copied out of the kernel parameters at init, so the
// hot loops never re-read parameter memory.
struct TileIter {
    int i, m, nt, ctx;
    int bs, i0, lim;
    const int *cache;  // clamped contexts of requests i0 .. i0 + kCtxCache - 1
    const int32_t *ctx_lens;
    __device__ int ctx_at(int r) const
    {
        const int n = r - i0;
        return (n >= 0 && n < kCtxCache) ? cache[n] : clamp_ctx(__ldg(ctx_lens + r), (long long)lim);
    }
    __device__ void init(const MainArgs &a, const CtaCtl &cc)
    {
        bs = a.bs;
        i0 = cc.i0;
        lim = (int)min((long long)a.mml, (long long)a.W * a.P);
        cache = cc.ctx;
        ctx_lens = a.ctx_lens;
        i = cc.i0;
        m = cc.m0;
        ctx = i < bs ? ctx_at(i) : 0;
        nt = (ctx + kTileTokens - 1) / kTileTokens;
    }
    __device__ void next()
    {
        if (++m < nt)
            return;
        m = 0;
        do {
            if (++i >= bs) {
                nt = 0;
                ctx = 0;
                return;
            }
            ctx = ctx_at(i);
            nt = (ctx + kTileTokens - 1) / kTileTokens;
        } while (nt == 0);
    }
};

// Position in a ring of n slots plus the parity of the current lap.
struct Ring {
    int n, slot;
    uint32_t phase;
    __device__ explicit Ring(int n_) : n(n_), slot(0), phase(0) {}
    __device__ void advance()
    {
        if (++slot == n) {
            slot = 0;
            phase ^= 1u;
        }
    }
};

// mdone[k % RS] completes (one tcgen05.commit) when the MMAs of tile k have
// finished: the epilogue waits for tile k's accumulator there and the repack
// for tile k - S's operand stage. RS = S + NBUF is deep enough that neither
// waiter can see a later phase of the same barrier: the MMA of tile k + RS
// needs the repack of tile k + RS and the epilogue of tile k + S, neither of
// which can have happened while a waiter is still at tile k.
struct Bars {
    uint64_t *op_full, *mdone, *tempty, *qfull, *qempty, *sfull, *gfull, *gempty, *done;
    __device__ Bars(const MainArgs &a, uint8_t *smem)
    {
        op_full = reinterpret_cast<uint64_t *>(smem + a.off_bar);
        mdone = op_full + a.S;
        tempty = mdone + a.RS;
        qfull = tempty + a.NBUF;
        qempty = qfull + a.QS;
        sfull = qempty + a.QS;
        gfull = sfull + a.RS;
        gempty = gfull + a.SG;
        done = gempty + a.SG;
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

// Each role copies the kernel parameters its loop needs into registers before
// the loop: the loops are full of inline-asm memory clobbers, after which any
// field read through the parameter reference would be fetched again.

static __device__ void qload_role(const MainArgs &a, uint8_t *smem, CtaCtl &c)
{
    const Bars B(a, smem);
    const int N = a.N, count = (int)c.count, q_box = a.q_box;
    const uint32_t q_bytes = (uint32_t)N * kHeadDim, w_bytes = (uint32_t)N * 4u;
    const uint32_t q0 = smem_u32(smem + a.off_q), w0 = smem_u32(smem + a.off_w);
    const float *const w = a.w;
    const void *const tmap = &a.tmap_q;
    TileIter it;
    it.init(a, c);
    Ring q(a.QS);
    for (int kk = 0; kk < count; ++kk) {
        if (kk == 0 || it.m == 0) {
            if (!mbar_wait(&B.qempty[q.slot], q.phase ^ 1u, &c.abort)) {
                raise_abort(a, c);
                return;
            }
            mbar_arrive_expect_tx(&B.qfull[q.slot], q_bytes + w_bytes);
            const uint32_t qdst = q0 + (uint32_t)q.slot * q_bytes;
            // boxes of q_box rows tile the request's N rows exactly (N = nbox * q_box)
            for (int nc = 0; nc * q_box < N; ++nc)
                tma_load_2d(qdst + (uint32_t)(nc * q_box * kHeadDim), tmap, 0, it.i * N + nc * q_box,
                            &B.qfull[q.slot]);
            bulk_load(w0 + (uint32_t)q.slot * w_bytes, w + (long long)it.i * N, w_bytes, &B.qfull[q.slot]);
            q.advance();
        }
        it.next();
    }
}

// ---------------------------------------------------------------- gather + repack

// Gather warp gw: rows 32*gw .. 32*gw+31 of every tile. The copies of tile k
// land in staging slot k % SG; gfull[slot] completes when every gather thread
// has published its rows' metadata (release arrive) and its copies have landed
// (cp.async arrive). The block-table entry of tile k travels by cp.async in
// this thread's cp.async group k: groups 0..SG-2 carry only the first entries,
// group SG-1+k carries the entry of tile k+SG-1 and the copies of tile k.
static __device__ void gather_role(const MainArgs &a, uint8_t *smem, CtaCtl &c, int gw)
{
    const Bars B(a, smem);
    const int lane = threadIdx.x & 31;
    const int row = gw * kTokPerWarp + lane;  // this lane's token row in a tile
    const uint64_t pol = a.l2_policy == 0   ? l2_evict_first_policy()
                         : a.l2_policy == 2 ? l2_evict_last_policy()
                                            : l2_evict_normal_policy();
    const uint8_t *const kv = a.kv;
    const int32_t *const bt = a.bt;
    const long long num_blocks = a.num_blocks, pool_bytes = a.pool_bytes;
    const int P = a.P, W = a.W;
    const bool p_pow2 = (P & (P - 1)) == 0;
    const int p_shift = __ffs(P) - 1;
    uint32_t *const status = a.status;
    const int count = (int)c.count, SG = a.SG, DT = a.SG - 1;
    uint8_t *const meta = smem + a.off_meta;                             // [SG][128]
    int32_t *const tring = reinterpret_cast<int32_t *>(smem + a.off_tab);  // [SG][128]
    const uint32_t stage0 = smem_u32(smem) + (uint32_t)(gw * kTokPerWarp) * kWinBytes;
    const uint32_t page0 = smem_u32(smem) + (uint32_t)(gw * kTokPerWarp) * (uint32_t)kKvRowBytes;
    const bool page_mode = a.page_mode != 0;
    auto page_of = [&](int tok) { return p_pow2 ? tok >> p_shift : tok / P; };
    TileIter iss, tab;
    iss.init(a, c);
    tab = iss;
    int tab_slot = 0;
    auto prefetch_table = [&]() {  // entry of tab's tile into ring slot tab_slot
        const int tok = tab.m * kTileTokens + row;
        int32_t *dst = tring + tab_slot * kTileTokens + row;
        if (tab.nt > 0 && tok < tab.ctx)
            cp_async_4(smem_u32(dst), bt + (long long)tab.i * W + page_of(tok), 4u, pol);
        else
            *dst = -1;
        tab.next();
        if (++tab_slot == SG)
            tab_slot = 0;
    };
    for (int kt = 0; kt < DT; ++kt) {
        if (kt < count)
            prefetch_table();
        cp_async_commit();
    }
    Ring g(SG);
    bool ok = true;
    for (int ki = 0; ki < count; ++ki) {
        if (!mbar_wait(&B.gempty[g.slot], g.phase ^ 1u, &c.abort)) {
            ok = false;
            break;
        }
        cp_async_wait_upto(DT - 1);  // group ki: the table entry of tile ki
        const int32_t b = tring[g.slot * kTileTokens + row];
        if (ki + DT < count)
            prefetch_table();
        const int t = iss.m * kTileTokens + row;
        if (page_mode) {
            // Page runs: consecutive rows of one page lie back to back in the
            // pool, so each run goes as one bulk copy (TMA engine, no
            // per-thread copies). Rows land at row * 132 in the slot. A run
            // starts at a multiple of 4 rows of its page (block starts and page
            // starts are), and its length is rounded up to whole 4-row groups
            // inside the same page, so source, destination and size keep the
            // 16-byte rule; the extra rows lie past the context and are masked.
            bool v = false;
            uint32_t tok = 0;
            if (t < iss.ctx) {
                if (b >= 0 && (long long)b < num_blocks) {
                    const int in_page = p_pow2 ? (t & (P - 1)) : t - page_of(t) * P;
                    tok = (uint32_t)((long long)b * P + in_page);
                    v = true;
                } else {
                    atomicOr(status, 0x1u);
                }
            }
            meta[g.slot * kTileTokens + row] = (uint8_t)(v ? 4u | ((uint32_t)row & 3u) : 0u);
            const uint32_t vmask = __ballot_sync(kFullMask, v);
            const uint32_t tprev = __shfl_up_sync(kFullMask, tok, 1);
            const bool start =
                v && (lane == 0 || !((vmask >> (lane - 1)) & 1u) || tok != tprev + 1u);
            const uint32_t smask = __ballot_sync(kFullMask, start);
            uint32_t bytes = 0;
            if (start) {
                const uint32_t later = lane == 31 ? 0u : (smask | ~vmask) & (~0u << (lane + 1));
                const int end = later ? __ffs(later) - 1 : 32;
                bytes = (uint32_t)(((end - lane) + 3) & ~3) * (uint32_t)kKvRowBytes;
            }
            const uint32_t total = __reduce_add_sync(kFullMask, bytes);
            __syncwarp();  // every lane's metadata before the arrive
            if (lane == 0)
                mbar_arrive_expect_tx(&B.gfull[g.slot], total);
            __syncwarp();
            if (start)
                bulk_load(page0 + (uint32_t)g.slot * kSlotBytes + (uint32_t)lane * kKvRowBytes,
                          kv + (unsigned long long)tok * kKvRowBytes, bytes, &B.gfull[g.slot]);
            cp_async_commit();  // keeps the table prefetch group count in step
            iss.next();
            g.advance();
            continue;
        }
        long long w0 = 0;
        uint32_t m = 0;
        uint32_t last = 16;  // bytes of the window's last chunk inside the pool (4..16)
        if (t < iss.ctx) {
            if (b >= 0 && (long long)b < num_blocks) {
                const int in_page = p_pow2 ? (t & (P - 1)) : t - page_of(t) * P;
                const long long o = ((long long)b * P + in_page) * kKvRowBytes;
                w0 = o & ~15ll;
                m = 4u | (uint32_t)((o >> 2) & 3);
                last = (uint32_t)min(16ll, pool_bytes - (w0 + 128));
            } else {
                atomicOr(status, 0x1u);
            }
        }
        meta[g.slot * kTileTokens + row] = (uint8_t)m;
        const uint32_t sb = stage0 + (uint32_t)g.slot * kSlotBytes;
        // 32 windows x 9 chunks = 288 copies: lane -> (token e / 9, chunk e % 9).
        // The window's first 128 bytes start at or before the row, so lie in
        // the pool; its last chunk may pass the end of the pool's last row and
        // then reads only the bytes inside (zero fill for the rest).
#pragma unroll
        for (int qq = 0; qq < 9; ++qq) {
            const int e = qq * 32 + lane;
            const int j = e / 9, ch = e - j * 9;
            const long long wj = __shfl_sync(kFullMask, w0, j);
            const uint32_t mj = __shfl_sync(kFullMask, m, j);
            const uint32_t lj = __shfl_sync(kFullMask, last, j);
            if (mj & 4u)
                cp_async_16_zfill(sb + (uint32_t)j * kWinBytes + (uint32_t)ch * 16u, kv + wj + ch * 16,
                                  ch < 8 ? 16u : lj, pol);
        }
        mbar_arrive(&B.gfull[g.slot]);            // metadata published
        cp_async_arrive_noinc(&B.gfull[g.slot]);  // copies landed
        cp_async_commit();
        iss.next();
        g.advance();
    }
    cp_async_wait_all();
    if (!ok)
        raise_abort(a, c);
}

// Repack warp rw: rows 32*rw .. 32*rw+31 of every tile, staging -> operand.
// Lane l moves row 32*rw + l: its 144-byte window as nine 16-byte loads (rows
// 144 bytes apart: eight lanes of a load phase hit distinct bank groups), a
// shift by the row's misalignment in registers, and eight 16-byte stores into
// the row's 128B-swizzled chunks (again conflict-free per phase).
static __device__ void repack_role(const MainArgs &a, uint8_t *smem, CtaCtl &c, int rw)
{
    const Bars B(a, smem);
    const int lane = threadIdx.x & 31;
    const int count = (int)c.count;
    // This lane's row: lanes 8k..8k+7 of a load/store phase take rows
    // 4a + ((a/2 + k) mod 4), a = 0..7, so the eight 16-byte accesses of a
    // phase hit distinct bank groups both when reading windows (rows 144 or
    // 132 bytes apart) and when writing the swizzled operand rows.
    const uint32_t pa = (uint32_t)lane & 7u, pk = (uint32_t)lane >> 3;
    const uint32_t r = (uint32_t)(rw * kTokPerWarp) + 4u * pa + (((pa >> 1) + pk) & 3u);
    const uint8_t *const meta = smem + a.off_meta + r;
    float *const sring = reinterpret_cast<float *>(smem + a.off_scale) + r;
    uint8_t *const op_row = smem + a.off_op + r * 128u;
    // the row's 16-byte aligned window: its own 144-byte slot, or (page runs)
    // the aligned bytes around row * 132
    const uint8_t *const win0 =
        smem + (a.page_mode ? (r * (uint32_t)kKvRowBytes) & ~15u : r * kWinBytes);
    Ring g(a.SG), st(a.S), sr(a.RS), rel(a.RS);  // rel: tile kk - S (stage release)
    bool ok = true;
    for (int kk = 0; kk < count; ++kk) {
        if (!mbar_wait(&B.gfull[g.slot], g.phase, &c.abort) ||
            (kk >= a.S && !mbar_wait(&B.mdone[rel.slot], rel.phase, &c.abort))) {
            ok = false;
            break;
        }
        if (kk >= a.S)
            rel.advance();
        const uint32_t m = meta[g.slot * kTileTokens];
        const uint4 *win = reinterpret_cast<const uint4 *>(win0 + (uint32_t)g.slot * kSlotBytes);
        uint32_t w[36];
#pragma unroll
        for (int q = 0; q < 9; ++q) {
            const uint4 v = win[q];
            w[4 * q + 0] = v.x;
            w[4 * q + 1] = v.y;
            w[4 * q + 2] = v.z;
            w[4 * q + 3] = v.w;
        }
        // word k of the row is window word k + (m & 3): shift by 1, then by 2
        const bool s1 = (m & 1u) != 0, s2 = (m & 2u) != 0;
#pragma unroll
        for (int k = 0; k < 35; ++k)
            w[k] = s1 ? w[k + 1] : w[k];
#pragma unroll
        for (int k = 0; k < 33; ++k)
            w[k] = s2 ? w[k + 2] : w[k];
        const bool valid = (m & 4u) != 0;
        uint8_t *ob = op_row + (uint32_t)st.slot * kStageBytes;
#pragma unroll
        for (int ch = 0; ch < 8; ++ch) {
            const uint4 v = valid ? make_uint4(w[4 * ch], w[4 * ch + 1], w[4 * ch + 2], w[4 * ch + 3])
                                  : make_uint4(0u, 0u, 0u, 0u);
            *reinterpret_cast<uint4 *>(ob + (((uint32_t)ch ^ (r & 7u)) << 4)) = v;
        }
        sring[sr.slot * kTileTokens] = valid ? __uint_as_float(w[32]) : 0.0f;
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            mbar_arrive(&B.op_full[st.slot]);
            mbar_arrive(&B.sfull[sr.slot]);
            mbar_arrive(&B.gempty[g.slot]);
        }
        g.advance();
        st.advance();
        sr.advance();
    }
    if (!ok)
        raise_abort(a, c);
}

// ---------------------------------------------------------------- MMA issue

static __device__ void mma_role(const MainArgs &a, uint8_t *smem, CtaCtl &c)
{
    const Bars B(a, smem);
    const int N = a.N, count = (int)c.count, cols = a.cols;
    const uint32_t tbase = c.tmem_base;
    const uint32_t op0 = smem_u32(smem + a.off_op), q0 = smem_u32(smem + a.off_q);
    const uint32_t q_bytes = (uint32_t)N * kHeadDim;
    TileIter it;
    it.init(a, c);
    Ring st(a.S), tb(a.NBUF), q(a.QS), md(a.RS);
    bool ok = true;
    for (int kk = 0; kk < count; ++kk) {
        const bool first = kk == 0 || it.m == 0;
        if (first && !mbar_wait(&B.qfull[q.slot], q.phase, &c.abort)) {
            ok = false;
            break;
        }
        if (!mbar_wait(&B.op_full[st.slot], st.phase, &c.abort) ||
            !mbar_wait(&B.tempty[tb.slot], tb.phase ^ 1u, &c.abort)) {
            ok = false;
            break;
        }
        tc_fence_after_sync();
        const uint32_t abase = op0 + (uint32_t)st.slot * kStageBytes;
        const uint32_t bbase = q0 + (uint32_t)q.slot * q_bytes;
        const uint32_t dcol = tbase + (uint32_t)(tb.slot * cols);
        // rolled: the issuing thread's loop stays small in the instruction cache
#pragma unroll 1
        for (int k4 = 0; k4 < kHeadDim / 32; ++k4) {
            const uint64_t ad = sw128_kmajor_desc(abase + k4 * 32);
            for (int nc = 0; nc * 256 < N; ++nc) {
                const int nw = min(256, N - nc * 256);
                const uint64_t bd = sw128_kmajor_desc(bbase + nc * 256 * kHeadDim + k4 * 32);
                umma_e4m3(dcol + (uint32_t)(nc * 256), ad, bd, idesc_e4m3_f32(128, nw),
                          k4 > 0 ? 1u : 0u);
            }
        }
        umma_commit(&B.mdone[md.slot]);
        if (kk == count - 1 || it.m == it.nt - 1) {
            umma_commit(&B.qempty[q.slot]);
            q.advance();
        }
        it.next();
        st.advance();
        tb.advance();
        md.advance();
    }
    if (!ok)
        raise_abort(a, c);
    umma_commit(B.done);
    if (!mbar_wait(B.done, 0, nullptr))
        atomicOr(a.status, 0x4u);
}

// ---------------------------------------------------------------- epilogue

// One epilogue chunk: 16 consecutive TMEM columns of this thread's lane.
__device__ __forceinline__ void epi_load(uint32_t taddr, uint32_t (&buf)[16]) { tmem_ld16(taddr, buf); }

__device__ __forceinline__ void epi_wait(uint32_t (&buf)[16])
{
    tmem_ld_wait();
    reg_fence16(buf);
}

// acc += sum over a 16-column chunk of w[h] * relu(x[h]) (SIGNED: of
// relu(-x[h]) when the thread's scale is negative, flip = its sign bit).
// Packed fp32x2 multiply-adds; the weights come as float4 broadcasts.
template <bool SIGNED>
__device__ __forceinline__ void epi_accumulate(const uint32_t (&x)[16], const float *w, uint32_t flip,
                                               float (&acc)[8])
{
    const float4 *w4 = reinterpret_cast<const float4 *>(w);
#pragma unroll
    for (int h = 0; h < 16; h += 4) {
        const float4 wv = w4[h / 4];
        float v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u)
            v[u] = fmaxf(__uint_as_float(SIGNED ? (x[h + u] ^ flip) : x[h + u]), 0.f);
        // four independent fp32x2 accumulator pairs: short dependency chains
        float *a = acc + ((h / 4) & 1) * 4;
        ffma2(a[0], a[1], wv.x, wv.y, v[0], v[1]);
        ffma2(a[2], a[3], wv.z, wv.w, v[2], v[3]);
    }
}

// All draft rows of one tile for this thread's token (TMEM lane): row j's
// score sum_h w[j][h] * relu(sc * x[j][h]) = |sc| * sum_h w[j][h] *
// relu(+-x[j][h]), x in TMEM columns [j*H, j*H + H), walked as 16-column
// chunks in two register buffers with the next chunk (of this row or the
// next) loading while the current one is reduced. Calls out(j, score) per
// row; arrives on tempty once the last TMEM read has completed.
template <int H, bool SIGNED, class Out>
__device__ __forceinline__ void epi_tile(uint32_t taddr, const float *wsl, uint32_t flip, float mag,
                                         int nn, uint64_t *tempty_bar, int lane, Out &&out)
{
    constexpr int CPR = H / 16;  // chunks per draft row
    uint32_t b0[16], b1[16];
    epi_load(taddr, b0);
    epi_wait(b0);
    for (int j = 0; j < nn; ++j) {
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        const uint32_t tj = taddr + (uint32_t)(j * H);
        const float *wj = wsl + j * H;
        const bool more_rows = j + 1 < nn;
        // b0 holds chunk p of row j (p even) on entry of each pass
#pragma unroll 1
        for (int p = 0; p < CPR; p += 2) {
            const bool has1 = p + 1 < CPR;
            const bool next_here = p + 2 < CPR;
            const bool has_next = next_here || more_rows;
            const uint32_t next_addr = next_here ? tj + (uint32_t)((p + 2) * 16) : tj + (uint32_t)H;
            if (has1) {
                epi_load(tj + (uint32_t)((p + 1) * 16), b1);
                epi_accumulate<SIGNED>(b0, wj + p * 16, flip, acc);
                epi_wait(b1);
                if (has_next)
                    epi_load(next_addr, b0);
                epi_accumulate<SIGNED>(b1, wj + (p + 1) * 16, flip, acc);
            } else {
                epi_accumulate<SIGNED>(b0, wj + p * 16, flip, acc);
                if (has_next)
                    epi_load(next_addr, b0);
            }
            if (has_next)
                epi_wait(b0);
        }
        if (!more_rows) {  // every TMEM read of this buffer has completed
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(tempty_bar);
        }
        out(j, (((acc[0] + acc[1]) + (acc[2] + acc[3])) + ((acc[4] + acc[5]) + (acc[6] + acc[7]))) *
                   mag);
    }
}

template <int H>
static __device__ void epilogue_role(const MainArgs &a, uint8_t *smem, CtaCtl &c, int we)
{
    const Bars B(a, smem);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, qd = warp & 3;
    const int r = qd * 32 + lane;  // token row of the tile = TMEM lane
    const int N = a.N, nn = a.nn, cols = a.cols;
    const long long mml = a.mml;
    float *const logits = a.logits;
    float *const clogits = a.clogits;
    uint32_t *const hist = a.hist;
    const float NEG_INF = -__int_as_float(0x7f800000);
    const uint32_t wtid = (uint32_t)(we * 32 + lane);
    constexpr int kEpiThreads = 128;
    const uint32_t bar_id = 1u;
    const bool want_hist = hist != nullptr;
    uint32_t *const shist = reinterpret_cast<uint32_t *>(smem + a.off_hist);
    const float *const scales = reinterpret_cast<const float *>(smem + a.off_scale) + r;
    const float *const w_smem = reinterpret_cast<const float *>(smem + a.off_w);
    const uint32_t tlane = c.tmem_base + ((uint32_t)(qd * 32) << 16);
    const uint64_t keep_pol = l2_evict_last_policy();

    // -inf beyond the last tile of each row: this CTA's share of every row.
    // Each warp takes 32 rows at a time (one coalesced load of their context
    // lengths), then writes the rows' shares one after another.
    if (logits) {
        const int rows = a.bs * nn;
        for (int base = we * 32; base < rows; base += kEpiThreads) {
            const int my_row = base + lane;
            const int my_cx = my_row < rows ? ctx_of(a, my_row / nn) : 0;
            const int nr = min(32, rows - base);
            for (int u = 0; u < nr; ++u) {
                const int cx = __shfl_sync(kFullMask, my_cx, u);
                const long long lo =
                    min((long long)(cx + kTileTokens - 1) / kTileTokens * kTileTokens, mml);
                const long long L = mml - lo;
                const long long s0 = lo + L * blockIdx.x / gridDim.x;
                const long long s1 = lo + L * (blockIdx.x + 1) / gridDim.x;
                float *row = logits + (long long)(base + u) * mml;
                for (long long t = s0 + lane; t < s1; t += 32)
                    row[t] = NEG_INF;
            }
        }
    }
    if (want_hist) {
        for (int e = (int)wtid; e < nn * kHistBins; e += kEpiThreads)
            shist[e] = 0;
        named_bar_sync(bar_id, kEpiThreads);
    }

    const int count = (int)c.count;
    TileIter it;
    it.init(a, c);
    Ring tb(a.NBUF), q(a.QS), sr(a.RS);
    // Waits that fail (abort or time limit) skip the data work but keep the
    // work group's barrier schedule, so no warp is left waiting on another.
    for (int kk = 0; kk < count; ++kk) {
        const bool first = kk == 0 || it.m == 0;
        bool ok = true;
        if (first)
            ok = mbar_wait(&B.qfull[q.slot], q.phase, &c.abort);
        ok = ok && mbar_wait(&B.sfull[sr.slot], sr.phase, &c.abort) &&
             mbar_wait(&B.mdone[sr.slot], sr.phase, &c.abort);
        // one outcome per warp: the tile body uses warp-wide shuffles and votes
        ok = __all_sync(kFullMask, ok);
        if (ok) {
            tc_fence_after_sync();
            const float sc = scales[sr.slot * kTileTokens];
            const int t = it.m * kTileTokens + r;
            const float *wsl = w_smem + q.slot * N;
            const uint32_t flip = sc < 0.0f ? 0x80000000u : 0u;
            const float mag = fabsf(sc);
            const uint32_t taddr = tlane + (uint32_t)(tb.slot * cols);
            auto out = [&](int j, float lj) {
                const long long row = (long long)it.i * nn + j;
                const bool valid = t < valid_len(it.ctx, nn, j);
                if (logits && t < mml)
                    logits[row * mml + t] = valid ? lj : NEG_INF;
                if (clogits && valid)
                    st_global_hint(clogits + row * mml + t, lj, keep_pol);
                // plain shared-memory atomics: the hardware merges same-bin
                // lanes far more cheaply than a match/vote aggregation
                if (want_hist && valid)
                    atomicAdd(shist + j * kHistBins + (f32_order_key(lj) >> kHistShift), 1u);
            };
            // negative scales are legal but rare: a separate (cold) path
            if (__all_sync(kFullMask, flip == 0u))
                epi_tile<H, false>(taddr, wsl, flip, mag, nn, &B.tempty[tb.slot], lane, out);
            else
                epi_tile<H, true>(taddr, wsl, flip, mag, nn, &B.tempty[tb.slot], lane, out);
        } else {
            raise_abort(a, c);
        }
        if (kk == count - 1 || it.m == it.nt - 1) {
            if (want_hist) {
                named_bar_sync(bar_id, kEpiThreads);
                for (int u = 0; u < nn; ++u) {
                    const long long row = (long long)it.i * nn + u;
                    for (int e = (int)wtid; e < kHistBins; e += kEpiThreads) {
                        const uint32_t v = shist[u * kHistBins + e];
                        if (v) {
                            atomicAdd(hist + row * kHistBins + e, v);
                            shist[u * kHistBins + e] = 0;
                        }
                    }
                }
                named_bar_sync(bar_id, kEpiThreads);
            }
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&B.qempty[q.slot]);
            q.advance();
        }
        it.next();
        tb.advance();
        sr.advance();
    }
}

// ---------------------------------------------------------------- kernel

constexpr int kMaxThreads = 32 * 16;
static_assert(kMaxThreads <= 32 * 32, "CtaCtl holds per-warp sums for at most 32 warps");

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
        for (int s = 0; s < a.S; ++s)
            mbar_init(&B.op_full[s], kRepackWarps);
        for (int g = 0; g < a.SG; ++g) {
            // window copies: a release arrive and a cp.async arrive per gather
            // thread; page runs: one expect-tx arrive per gather warp
            mbar_init(&B.gfull[g], a.page_mode ? kGatherWarps : 2 * 32 * kGatherWarps);
            mbar_init(&B.gempty[g], kRepackWarps);
        }
        for (int b = 0; b < a.NBUF; ++b)
            mbar_init(&B.tempty[b], 4);
        for (int q = 0; q < a.QS; ++q) {
            mbar_init(&B.qfull[q], 1);
            mbar_init(&B.qempty[q], 1 + 4);
        }
        for (int q = 0; q < a.RS; ++q) {
            mbar_init(&B.sfull[q], kRepackWarps);
            mbar_init(&B.mdone[q], 1);
        }
        mbar_init(B.done, 1);
        mbar_init_fence();
    }
    __syncwarp();
    if (warp == 0)
        tmem_alloc(&ctl.tmem_base, (uint32_t)a.tmem_cols);

    balance_schedule(
        a.bs, [&](int i) { return (long long)((ctx_of(a, i) + kTileTokens - 1) / kTileTokens); },
        ctl);
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

    if (warp == kMmaWarp) {
        if ((threadIdx.x & 31) == 0)
            mma_role(a, smem, ctl);
        __syncwarp();
    } else if (warp == kQloadWarp) {
        if ((threadIdx.x & 31) == 0)
            qload_role(a, smem, ctl);
        __syncwarp();
    } else if (warp < kQloadWarp) {
        if ((warp & 2) == 0)
            gather_role(a, smem, ctl, row_block_of(warp));
        else
            repack_role(a, smem, ctl, row_block_of(warp));
    } else if (warp >= kFirstEpiWarp && warp < kFirstEpiWarp + 4) {
        epilogue_role<H>(a, smem, ctl, warp - kFirstEpiWarp);
    }

    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    __syncwarp();
    if (warp == 0)
        tmem_dealloc(ctl.tmem_base, (uint32_t)a.tmem_cols);
}

}  // namespace pmqa
