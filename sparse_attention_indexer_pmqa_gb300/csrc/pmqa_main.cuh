// pmqa_main.cuh -- the persistent FP8 paged MQA-logits kernel for sm_103a.
//
// Definition (page "[Bug] aiter ops triton attention pa", section "Minimal
// reproduction", reference function `torch_ref`): for query row r = (i, j) and
// token t, logit = sum_h w[r][h] * relu(s_t * q[i][j][h] . k_t), -inf outside
// t < ctx_i, t <= ctx_i - next_n + j.
//
// One CTA per SM walks a contiguous range of (request, 128-token tile) work
// items, balanced by tile count over all requests. The CTA's 16 warps form
// four warpgroups; warpgroup g takes the CTA's tiles g, g + 4, g + 8, ... and
// runs each one through every step on its own, so the four tiles in flight
// overlap one another's latencies. Thread (warp w, lane l) of a warpgroup owns
// tile row R = 32 * (w % 4) + l, which is also its TMEM lane. Per tile:
//   1. wait for the tile's rows to land in the warpgroup's staging slot: the
//      16-byte aligned 144-byte window of each 132-byte row, copied with
//      16-byte cp.async (any block size), or, when the block size is a
//      multiple of 4, runs of consecutive rows of a page, one bulk copy each;
//   2. repack row R: its 32 fp8 words, shifted by the row's 0/4/8/12-byte
//      misalignment, into the 128B-swizzled K-major operand tile; its fp32
//      scale stays in a register;
//   3. issue the copies of the warpgroup's next tile (block-table entries for
//      the one after it are already in registers);
//   4. one thread issues tcgen05.mma: D[token][(j,h)] = K_tile[128 x 128] *
//      Q[(j,h) x 128]^T, fp8 e4m3 in, fp32 accumulators in TMEM: the
//      warpgroup's own 128 columns up to next_n * H = 128; for up to 256
//      columns a 256-column half that warpgroups g and g ^ 2 use in turn
//      (each warp hands it on by an mbarrier arrival once it has read its
//      lane); beyond that, passes of 128 columns (whole draft rows);
//   5. each thread reads its lane of the accumulators (tcgen05.ld), forms
//      sum_h w[j][h] * relu(x) per draft row, scales, masks, and writes full
//      logits rows and/or the compact logits plus the per-row key histogram
//      (global atomics) that the selection reads. In a warpgroup's own
//      columns these outputs wait in registers and are written while the
//      next tile's MMA runs.
// At the end of each request the four warpgroups meet at a CTA barrier and
// thread 0 loads the query and weights of the request QS ahead into the slot
// just freed (TMA). Every wait is bounded.
#pragma once

#include <cuda.h>

#include <cstdint>

#include "pmqa_ptx.cuh"

namespace pmqa {

constexpr uint32_t kFullMask = 0xFFFFFFFFu;
constexpr int kTileTokens = 128;
constexpr int kHeadDim = 128;
constexpr int kKvRowBytes = kHeadDim + 4;
constexpr int kGroups = 4;                                 // warpgroups per CTA
constexpr int kNumWarps = 4 * kGroups;
constexpr int kMaxThreads = 32 * kNumWarps;
constexpr int kMaxRows = 4;                                // draft rows per request
constexpr uint32_t kStageBytes = kTileTokens * kHeadDim;  // 16 KB operand tile
constexpr uint32_t kWinBytes = 144;                        // aligned window of one row
constexpr uint32_t kSlotBytes = kTileTokens * kWinBytes;   // one staging slot (18 KB)
constexpr uint32_t kGroupBytes = kSlotBytes + kStageBytes; // a warpgroup's region (34 KB)
constexpr int kPassCols = 128;                             // accumulator columns per MMA pass
constexpr int kHistBins = 2048;                            // top 11 bits of the order key
constexpr int kHistShift = 21;
constexpr uint32_t kCtaBarrier = 5;                        // named barrier of all 512 threads

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
    uint32_t *hist;    // per-row histograms of the top 11 bits of the order keys [rows, 2048], or null
    uint32_t *status;
    int l2_policy;     // KV stream: 0 evict_first, 1 evict_normal, 2 evict_last
    int page_mode;     // block_size % 4 == 0: rows move as page runs by bulk copy
    // a slice [tok_begin[i], tok_end[i]) of every request's tokens, or null
    // for all of them (clamped to [0, ctx_i])
    const int32_t *tok_begin, *tok_end;
    // shared-memory / TMEM layout, computed on the host
    int N, QS, cols, tmem_cols;
    int q_box;  // rows per q TMA box: N / ceil(N / 256)
    uint32_t off_q, off_w, off_grp, off_bar, smem_bytes;
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

// Context lengths of the CTA's requests: from the shared-memory cache while it
// covers them, else from global memory (clamped); and, when SLICED, the slice
// of each request's tokens to score (else all of them: the kernel is compiled
// for each case so the common one carries no slice bounds).
template <bool SLICED>
struct ReqCtx {
    int bs, i0, lim;
    const int *cache;  // clamped contexts of requests i0 .. i0 + kCtxCache - 1
    const int32_t *ctx_lens;
    const int32_t *tok_begin, *tok_end;
    __device__ void init(const MainArgs &a, const CtaCtl &cc)
    {
        bs = a.bs;
        i0 = cc.i0;
        lim = (int)min((long long)a.mml, (long long)a.W * a.P);
        cache = cc.ctx;
        ctx_lens = a.ctx_lens;
        tok_begin = a.tok_begin;
        tok_end = a.tok_end;
    }
    __device__ int ctx_at(int r) const
    {
        const int n = r - i0;
        return (n >= 0 && n < kCtxCache) ? cache[n] : clamp_ctx(__ldg(ctx_lens + r), (long long)lim);
    }
    // tokens [tb, te) of request r (context ctx) are scored
    __device__ void bounds(int r, int ctx, int &tb, int &te) const
    {
        if constexpr (SLICED) {
            tb = clamp_ctx(__ldg(tok_begin + r), (long long)ctx);
            te = max(tb, clamp_ctx(__ldg(tok_end + r), (long long)ctx));
        } else {
            tb = 0;
            te = ctx;
        }
    }
};

// 128-token tiles [mb, nt) that cover tokens [tb, te) (none when te <= tb).
__device__ __forceinline__ void tile_span(int tb, int te, int &mb, int &nt)
{
    if (te > tb) {
        mb = tb / kTileTokens;
        nt = (te + kTileTokens - 1) / kTileTokens;
    } else {
        mb = nt = 0;
    }
}

// Tiles of request i to score (the length of its work item in the schedule).
template <bool SLICED>
__device__ __forceinline__ int tiles_of(const MainArgs &a, int i)
{
    const int ctx = ctx_of(a, i);
    int tb = 0, te = ctx, mb, nt;
    if constexpr (SLICED) {
        tb = clamp_ctx(__ldg(a.tok_begin + i), (long long)ctx);
        te = max(tb, clamp_ctx(__ldg(a.tok_end + i), (long long)ctx));
    }
    tile_span(tb, te, mb, nt);
    return nt - mb;
}

// Position (request i, tile m of the tiles [mb, nt) covering its tokens
// [tb, te), context ctx) in the CTA's walk over (request, tile) pairs;
// requests without tiles are skipped. Without slices mb = tb = 0, te = ctx.
template <bool SLICED>
struct TilePos {
    int i, m, mb, nt, ctx, tb, te;
    __device__ void set_request(const ReqCtx<SLICED> &rc, int r)
    {
        i = r;
        ctx = rc.ctx_at(r);
        if constexpr (SLICED) {
            rc.bounds(r, ctx, tb, te);
            tile_span(tb, te, mb, nt);
        } else {
            tb = mb = 0;
            te = ctx;
            nt = (ctx + kTileTokens - 1) / kTileTokens;
        }
    }
    __device__ void clear()
    {
        m = mb = nt = ctx = tb = te = 0;
    }
    __device__ void init(const ReqCtx<SLICED> &rc, const CtaCtl &cc)
    {
        if (cc.i0 < rc.bs) {
            set_request(rc, cc.i0);
            m = mb + cc.m0;
        } else {
            i = cc.i0;
            clear();
        }
    }
    __device__ void next(const ReqCtx<SLICED> &rc)
    {
        if (++m < nt)
            return;
        do {
            if (i + 1 >= rc.bs) {
                ++i;
                clear();
                return;
            }
            set_request(rc, i + 1);
        } while (nt == 0);
        m = mb;
    }
    __device__ bool last_of_request() const { return m == nt - 1; }
};

// Steps from request to request of the CTA's range: `first` is the CTA tile
// index of the current request's first tile here.
template <bool SLICED>
struct ReqWalk {
    TilePos<SLICED> p;
    int first;
    __device__ void init(const ReqCtx<SLICED> &rc, const CtaCtl &c)
    {
        p.init(rc, c);
        first = 0;
    }
    __device__ bool valid(int count) const { return p.nt > 0 && first < count; }
    __device__ void advance(const ReqCtx<SLICED> &rc)
    {
        first += p.nt - p.m;
        p.m = p.nt - 1;
        p.next(rc);
    }
};

// Shared-memory mbarriers.
//   qfull[QS]     query + weights of a request landed (TMA transaction count)
//   mma[4]        a warpgroup's MMA pass finished (one tcgen05.commit)
//   run[16]       a warp's page runs of its warpgroup's staging slot landed
struct Bars {
    uint64_t *qfull, *mma, *run, *tfree;
    __device__ Bars(const MainArgs &a, uint8_t *smem)
    {
        qfull = reinterpret_cast<uint64_t *>(smem + a.off_bar);
        mma = qfull + a.QS;
        run = mma + kGroups;
        tfree = run + kNumWarps;
    }
};
// tfree[h]: TMEM half h released by the warpgroup that used it last, one arrival per warp (when two
// warpgroups share each 256-column half)
constexpr int kNumBars = kGroups + kNumWarps + 2;  // plus QS

__device__ __forceinline__ void raise_abort(const MainArgs &a, CtaCtl &c)
{
    c.abort = 1;
    atomicOr(a.status, 0x4u);
}

__device__ __forceinline__ bool aborted(const CtaCtl &c)
{
    return *reinterpret_cast<const volatile int *>(&c.abort) != 0;
}

// Query rows (TMA, 128B swizzle) and weights (bulk copy) of request i into
// query slot `slot`; qfull[slot] completes when both have landed.
__device__ __forceinline__ void load_query(const MainArgs &a, uint8_t *smem, const Bars &B, int slot,
                                           int i)
{
    const int N = a.N, q_box = a.q_box;
    const uint32_t q_bytes = (uint32_t)N * kHeadDim, w_bytes = (uint32_t)N * 4u;
    const uint32_t qdst = smem_u32(smem + a.off_q) + (uint32_t)slot * q_bytes;
    mbar_arrive_expect_tx(&B.qfull[slot], q_bytes + w_bytes);
    // boxes of q_box rows tile the request's N rows exactly (N = nbox * q_box)
    for (int nc = 0; nc * q_box < N; ++nc)
        tma_load_2d(qdst + (uint32_t)(nc * q_box * kHeadDim), &a.tmap_q, 0, i * N + nc * q_box,
                    &B.qfull[slot]);
    bulk_load(smem_u32(smem + a.off_w) + (uint32_t)slot * w_bytes, a.w + (long long)i * N, w_bytes,
              &B.qfull[slot]);
}

// ---------------------------------------------------------------- epilogue math

// Over NC consecutive columns: acc[0..3] += w[h] * x[h] and acc[4..7] +=
// w[h] * |x[h]|, packed fp32x2 multiply-adds (two accumulator pairs each).
// relu(x) = (x + |x|) / 2 and relu(-x) = (|x| - x) / 2, so the row's
// sum_h w[h] * relu(+-x[h]) is formed from the two sums in acc_sum without a
// max per column; the thread's scale sign enters there once. The weights come
// as float4 broadcasts from shared memory. FIRST: the chunk starts a row, and
// its products initialise the accumulators instead of adding to them.
template <int NC, bool FIRST = false>
__device__ __forceinline__ void epi_accumulate(const uint32_t (&x)[NC], uint32_t w, float (&acc)[8])
{
#pragma unroll
    for (int h = 0; h < NC; h += 4) {
        const float4 wv = lds128f_nv(w + (uint32_t)(h * 4));
        float v[4], av[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            v[u] = __uint_as_float(x[h + u]);
            av[u] = fabsf(v[u]);
        }
        if (FIRST && h == 0) {
            fmul2(acc[0], acc[1], wv.x, wv.y, v[0], v[1]);
            fmul2(acc[2], acc[3], wv.z, wv.w, v[2], v[3]);
            fmul2(acc[4], acc[5], wv.x, wv.y, av[0], av[1]);
            fmul2(acc[6], acc[7], wv.z, wv.w, av[2], av[3]);
        } else {
            ffma2(acc[0], acc[1], wv.x, wv.y, v[0], v[1]);
            ffma2(acc[2], acc[3], wv.z, wv.w, v[2], v[3]);
            ffma2(acc[4], acc[5], wv.x, wv.y, av[0], av[1]);
            ffma2(acc[6], acc[7], wv.z, wv.w, av[2], av[3]);
        }
    }
}

// The row's sum_h w[h] * relu(x[h]) (SIGNED: relu(-x[h]) when the thread's
// scale is negative, flip = its sign bit) from the signed sum (acc[0..3]) and
// the absolute sum (acc[4..7]): (|sum| part +- signed part) / 2. Where every
// term is clipped the two parts cancel exactly (the same operations on
// negated operands), so the score is exactly 0. The next row's first chunk
// re-initialises the accumulators.
template <bool SIGNED>
__device__ __forceinline__ float acc_sum(float (&acc)[8], uint32_t flip)
{
    fadd2(acc[0], acc[1], acc[2], acc[3]);
    fadd2(acc[4], acc[5], acc[6], acc[7]);
    float s = acc[0] + acc[1];
    if (SIGNED)
        s = __uint_as_float(__float_as_uint(s) ^ flip);
    return 0.5f * (s + (acc[4] + acc[5]));
}

// Draft rows j0 .. j0 + NR - 1 for this thread's token (TMEM lane): row j's
// score is |sc| * sum_h w[j][h] * relu(+-x[j][h]), x in TMEM columns
// [(j - j0) * H, (j - j0) * H + H) from taddr, weights w[j][h] at shared
// address wsl + 4 * ((j - j0) * H + h). The NR * H / 16 chunks of 16 columns
// alternate between two register buffers, the next chunk loading while the
// current one is reduced. Once every TMEM read of the pass has completed (the
// last chunk is in registers) it calls done(): the columns may be reused from
// then on. Then out(j, score) per row.
template <int H, int NR, bool SIGNED, class Out, class Done>
__device__ __forceinline__ void epi_rows(uint32_t taddr, uint32_t wsl, uint32_t flip, float mag,
                                         int j0, Out &&out, Done &&done)
{
    constexpr int NC = 16;
    constexpr int CPR = H / NC;  // chunks per draft row
    constexpr int TOTAL = NR * CPR;
    uint32_t b[2][NC];
    float acc[8];
    float res[NR];
    tmem_ld_cols<NC>(taddr, b[0]);
    tmem_ld_wait();
    reg_fence_cols<NC>(b[0]);
    if (TOTAL == 1)
        done();
#pragma unroll
    for (int ch = 0; ch < TOTAL; ++ch) {
        if (ch + 1 < TOTAL)
            tmem_ld_cols<NC>(taddr + (uint32_t)((ch + 1) * NC), b[(ch + 1) & 1]);
        if (ch % CPR == 0)
            epi_accumulate<NC, true>(b[ch & 1], wsl + (uint32_t)(ch * NC * 4), acc);
        else
            epi_accumulate<NC>(b[ch & 1], wsl + (uint32_t)(ch * NC * 4), acc);
        if ((ch + 1) % CPR == 0)
            res[ch / CPR] = acc_sum<SIGNED>(acc, flip) * mag;
        if (ch + 1 < TOTAL) {
            tmem_ld_wait();
            reg_fence_cols<NC>(b[(ch + 1) & 1]);
            if (ch + 2 == TOTAL)
                done();  // the last chunk is in registers
        }
    }
#pragma unroll
    for (int u = 0; u < NR; ++u)
        out(j0 + u, res[u]);
}


// epi_rows for nr (1 .. RPP) rows, the scale's sign known warp-wide (all_pos)
// or per thread.
template <int H, int RPP, class Out, class Done>
__device__ __forceinline__ void epi_dispatch(int nr, bool all_pos, uint32_t taddr, uint32_t wsl,
                                             uint32_t flip, float mag, int j0, Out &out, Done &done)
{
    if (nr == RPP) {
        if (all_pos)
            epi_rows<H, RPP, false>(taddr, wsl, flip, mag, j0, out, done);
        else
            epi_rows<H, RPP, true>(taddr, wsl, flip, mag, j0, out, done);
    } else if constexpr (RPP > 1) {
        epi_dispatch<H, RPP - 1>(nr, all_pos, taddr, wsl, flip, mag, j0, out, done);
    }
}

// ---------------------------------------------------------------- warpgroup

// Position in the CTA's tile range: `cur` is tile kk. step(n) moves n tiles on
// and counts the request ends it passes (the last tile of a request, and the
// range's last tile).
template <bool SLICED>
struct Walk {
    TilePos<SLICED> cur;
    int kk;
    __device__ int step(const ReqCtx<SLICED> &rc, int n, int count)
    {
        // common case: the n tiles left behind lie inside one request and
        // before the range's last tile
        if (cur.m + n < cur.nt && kk + n < count) {
            cur.m += n;
            kk += n;
            return 0;
        }
        int ends = 0;
        for (int u = 0; u < n; ++u) {
            if (kk < count && (cur.m == cur.nt - 1 || kk == count - 1))
                ++ends;
            cur.next(rc);
            ++kk;
        }
        return ends;
    }
};

// One warpgroup's gather of its own tiles: the block-table entries, the copies
// of a tile's rows into the warpgroup's staging slot, and the repack of this
// thread's row R into the 128B-swizzled K-major operand tile behind the slot.
// PAGE: rows move as page runs by bulk copy (block size a multiple of 4), else
// as 16-byte aligned windows by cp.async, with 32-bit byte offsets when POOL32
// (a pool under 2 GB).
template <bool PAGE, bool POOL32>
struct TileGather {
    const uint8_t *kv;
    const int32_t *bt;
    long long num_blocks, pool_bytes;
    uint32_t *status;
    uint64_t pol;
    int P, W, p_shift;
    bool p_pow2;
    uint32_t R, lane, last9;
    uint32_t stage, win, opx, wstage;
    uint64_t *run_bar;
    uint32_t run_phase;

    __device__ void init(const MainArgs &a, uint32_t stage_addr, uint32_t qd, uint32_t lane_,
                         uint64_t *run_bar_)
    {
        pol = a.l2_policy == 0   ? l2_evict_first_policy()
              : a.l2_policy == 2 ? l2_evict_last_policy()
                                 : l2_evict_normal_policy();
        kv = a.kv;
        bt = a.bt;
        num_blocks = a.num_blocks;
        pool_bytes = a.pool_bytes;
        P = a.P;
        W = a.W;
        p_pow2 = (P & (P - 1)) == 0;
        p_shift = __ffs(P) - 1;
        status = a.status;
        lane = lane_;
        R = qd * 32u + lane;
        stage = stage_addr;
        // window mode: row R's 16-byte aligned window; page runs: the row itself
        win = stage + (PAGE ? R * (uint32_t)kKvRowBytes : R * kWinBytes);
        // operand row R is 128-byte aligned: chunk ch sits at opx ^ (ch << 4)
        opx = (stage + kSlotBytes + R * 128u) ^ ((R & 7u) << 4);
        wstage = stage + qd * 32u * kWinBytes;  // this warp's 32 windows
        run_bar = run_bar_;
        run_phase = 0;
        // copy e = qq * 32 + lane of a warp's 288 window chunks: window e / 9,
        // chunk e % 9; bit qq of last9 marks chunk 8 (the window's last)
        last9 = 0;
#pragma unroll
        for (int qq = 0; qq < 9; ++qq)
            last9 |= (((uint32_t)(qq * 32) + lane) % 9u == 8u ? 1u : 0u) << qq;
    }

    __device__ int page_of(int tok) const { return p_pow2 ? tok >> p_shift : tok / P; }

    // Block-table entry of this thread's row in tile p (-1 past the context).
    template <bool SLICED>
    __device__ int32_t table_entry(const TilePos<SLICED> &p) const
    {
        const int tok = p.m * kTileTokens + (int)R;
        const bool in = SLICED ? (tok >= p.tb && tok < p.te) : tok < p.ctx;
        return (p.nt > 0 && in) ? __ldg(bt + (long long)p.i * W + page_of(tok)) : -1;
    }

    // Copies of this warp's 32 rows of tile p (this row's table entry b) into
    // the staging slot; returns the row's repack metadata: 4 | misalignment / 4
    // when the row is valid, else 0.
    template <bool SLICED>
    __device__ uint32_t issue(const TilePos<SLICED> &p, int32_t b)
    {
        const int t = p.m * kTileTokens + (int)R;
        bool v = false;
        long long o = 0;  // byte offset of the row in the pool
        if (SLICED ? (t >= p.tb && t < p.te) : t < p.ctx) {
            if (b >= 0 && (long long)b < num_blocks) {
                const int in_page = p_pow2 ? (t & (P - 1)) : t - page_of(t) * P;
                o = ((long long)b * P + in_page) * kKvRowBytes;
                v = true;
            } else {
                atomicOr(status, 0x1u);
            }
        }
        if constexpr (PAGE) {
            // A run of consecutive valid rows moves as one bulk copy of whole
            // 4-row groups: its start is rounded down, and its length up, to
            // group boundaries. A group's 4 tokens are t = 4u .. 4u + 3 (the
            // warp's rows start at a multiple of 32), so they sit in one page
            // (P % 4 == 0) at in-page positions 4v .. 4v + 3: the copy is
            // 16-byte aligned (4 rows = 528 bytes) in the pool and in the slot,
            // reads only rows of the run's pages and stays inside the warp's
            // 32 rows. Rows copied outside the run are masked. Runs start at
            // the warp's first row, a page start, the first row after a bad
            // page, or the first row of the request's scored slice; valid rows
            // never resume inside a group once they stop, so runs do not share
            // a group.
            const uint32_t tok = (uint32_t)(o / kKvRowBytes);
            const uint32_t vmask = __ballot_sync(kFullMask, v);
            const uint32_t tprev = __shfl_up_sync(kFullMask, tok, 1);
            const bool start = v && (lane == 0 || !((vmask >> (lane - 1)) & 1u) || tok != tprev + 1u);
            const uint32_t smask = __ballot_sync(kFullMask, start);
            const uint32_t back = lane & 3u;  // rows from the group's first row
            uint32_t bytes = 0;
            if (start) {
                const uint32_t later = lane == 31 ? 0u : (smask | ~vmask) & (~0u << (lane + 1));
                const int end = later ? __ffs(later) - 1 : 32;
                bytes = (uint32_t)(((end - (int)(lane - back)) + 3) & ~3) * (uint32_t)kKvRowBytes;
            }
            const uint32_t total = __reduce_add_sync(kFullMask, bytes);
            if (lane == 0)
                mbar_arrive_expect_tx(run_bar, total);
            __syncwarp();
            if (start)
                bulk_load(stage + (R - back) * (uint32_t)kKvRowBytes, kv + (o - (long long)back * kKvRowBytes),
                          bytes, run_bar);
            return v ? 4u : 0u;
        }
        // Window j of the warp starts at wstage + 144 j = wstage + 16 (9 j),
        // so copy e lands at wstage + 16 e and reads kv + (w0_j - 144 j) + 16 e.
        // One instruction covers about 3.5 whole windows. A window's first
        // 128 bytes start at or before its row, so lie in the pool; its last
        // chunk may pass the end of the pool and then reads only the bytes
        // inside.
        const long long w0 = o & ~15ll;
        const uint32_t last = v ? (uint32_t)min(16ll, pool_bytes - (w0 + 128)) : 0u;
        const uint32_t ml = (v ? 0x100u : 0u) | last;
        if constexpr (POOL32) {
            const int wrel = (int)w0 - (int)kWinBytes * (int)lane;
#pragma unroll
            for (int qq = 0; qq < 9; ++qq) {
                const uint32_t e = (uint32_t)(qq * 32) + lane;
                const int j = (int)((e * 7282u) >> 16);  // e / 9 for e < 288
                const int wj = __shfl_sync(kFullMask, wrel, j);
                const uint32_t mj = __shfl_sync(kFullMask, ml, j);
                if (mj & 0x100u)
                    cp_async_16_zfill(wstage + 16u * e, kv + (uint32_t)(wj + 16 * (int)e),
                                      ((last9 >> qq) & 1u) ? (mj & 0xFFu) : 16u, pol);
            }
        } else {
            const long long wrel = w0 - (long long)kWinBytes * lane;
#pragma unroll
            for (int qq = 0; qq < 9; ++qq) {
                const uint32_t e = (uint32_t)(qq * 32) + lane;
                const int j = (int)((e * 7282u) >> 16);
                const long long wj = __shfl_sync(kFullMask, wrel, j);
                const uint32_t mj = __shfl_sync(kFullMask, ml, j);
                if (mj & 0x100u)
                    cp_async_16_zfill(wstage + 16u * e, kv + (wj + 16ll * e),
                                      ((last9 >> qq) & 1u) ? (mj & 0xFFu) : 16u, pol);
            }
        }
        return v ? 4u | ((uint32_t)(o >> 2) & 3u) : 0u;
    }

    // Wait until the rows of the tile in the staging slot have landed: window
    // copies per thread, page runs on the warp's mbarrier.
    __device__ bool wait_rows(const int *abort_flag)
    {
        bool ok = true;
        if constexpr (PAGE) {
            ok = mbar_wait(run_bar, run_phase, abort_flag);
            run_phase ^= 1u;
        } else {
            cp_async_wait_group<0>();
        }
        __syncwarp();
        return ok;
    }

    // Repack row R into the operand; returns its scale (0 for an invalid row).
    // Rows past the context keep whatever the slot holds: their scores are
    // masked.
    __device__ float repack(uint32_t meta) const
    {
        float sc;
        if constexpr (PAGE) {
            // rows 132 bytes apart: word k of the 32 lanes' rows sits in bank
            // (R + k) mod 32, so 4-byte loads are conflict-free
#pragma unroll
            for (int ch = 0; ch < 8; ++ch)
                sts128(opx ^ ((uint32_t)ch << 4), lds32(win + 16u * ch), lds32(win + 16u * ch + 4u),
                       lds32(win + 16u * ch + 8u), lds32(win + 16u * ch + 12u));
            sc = (meta & 4u) ? __uint_as_float(lds32(win + 128u)) : 0.0f;
        } else {
            uint32_t wv[36];
#pragma unroll
            for (int q = 0; q < 9; ++q) {
                const uint4 x = lds128(win + 16u * q);
                wv[4 * q + 0] = x.x;
                wv[4 * q + 1] = x.y;
                wv[4 * q + 2] = x.z;
                wv[4 * q + 3] = x.w;
            }
            // row word k is window word k + (meta & 3): shift by 1, then by 2
            const bool s1 = (meta & 1u) != 0, s2 = (meta & 2u) != 0;
#pragma unroll
            for (int k = 0; k < 35; ++k)
                wv[k] = s1 ? wv[k + 1] : wv[k];
#pragma unroll
            for (int k = 0; k < 33; ++k)
                wv[k] = s2 ? wv[k + 2] : wv[k];
#pragma unroll
            for (int ch = 0; ch < 8; ++ch)
                sts128(opx ^ ((uint32_t)ch << 4), wv[4 * ch], wv[4 * ch + 1], wv[4 * ch + 2], wv[4 * ch + 3]);
            sc = (meta & 4u) ? __uint_as_float(wv[32]) : 0.0f;
        }
        __syncwarp();  // every lane has read its row before the slot is refilled
        return sc;
    }
};

// Query slots. Request n of the CTA's range (counting only requests with
// tokens) sits in slot n % QS; at each request end every warpgroup meets the
// others (a CTA barrier), then thread 0 loads the query of the request QS
// ahead into the slot just freed.
template <bool SLICED>
struct QuerySlots {
    int slot;        // slot of this warpgroup's current request
    uint32_t phase;  // parity of that slot's fill
    bool have;       // the warpgroup has waited for its current request's slot
    int loads;       // query loads issued (thread 0)
    ReqWalk<SLICED> nxt;  // next request whose query is to be loaded (thread 0)

    __device__ void init(const MainArgs &a, uint8_t *smem, const Bars &B, const ReqCtx<SLICED> &rc,
                         const CtaCtl &c, int count)
    {
        slot = 0;
        phase = 0;
        have = false;
        loads = 0;
        nxt.init(rc, c);
        if (threadIdx.x == 0)
            for (int n = 0; n < a.QS; ++n) {
                if (nxt.valid(count)) {
                    load_query(a, smem, B, n, nxt.p.i);
                    ++loads;
                }
                nxt.advance(rc);
            }
    }
    __device__ void pass_ends(const MainArgs &a, uint8_t *smem, const Bars &B,
                              const ReqCtx<SLICED> &rc, const CtaCtl &c, int count, int ends)
    {
        for (int u = 0; u < ends; ++u) {
            named_bar_sync(kCtaBarrier, kMaxThreads);
            if (threadIdx.x == 0) {
                if (nxt.valid(count) && !aborted(c)) {
                    load_query(a, smem, B, slot, nxt.p.i);
                    ++loads;
                }
                nxt.advance(rc);
            }
            if (++slot == a.QS) {
                slot = 0;
                phase ^= 1u;
            }
            have = false;
        }
    }
    // after an abort, query loads nobody consumed land before the CTA exits (bounded)
    __device__ void drain(const Bars &B, int QS) const
    {
        if (threadIdx.x == 0)
            for (int u = loads > QS ? loads - QS : 0; u < loads; ++u)
                mbar_wait(&B.qfull[u % QS], (uint32_t)(u / QS) & 1u, nullptr);
    }
};

// The epilogue's output of one token for draft row j: the full logits row
// and/or the compact logits plus the row's key histogram.
struct TokenOut {
    float *logits, *clogits;
    uint32_t *hrow;
    long long obase, mml;
    int t, lim0;
    bool in_slice;  // t inside the request's scored tokens [tb, te)
    uint64_t keep_pol;
    __device__ void operator()(int j, float lj) const
    {
        const bool vj = in_slice && t < lim0 + j;
        const long long o = obase + (long long)j * mml;
        if (logits && t < mml)
            logits[o] = vj ? lj : -__int_as_float(0x7f800000);
        if (clogits && vj)
            st_global_hint(clogits + o, lj, keep_pol);
        if (hrow && vj)
            atomicAdd(hrow + j * kHistBins + (f32_order_key(lj) >> kHistShift), 1u);
    }
};

template <bool SLICED>
__device__ __forceinline__ TokenOut token_out(const MainArgs &a, const TilePos<SLICED> &it,
                                              uint32_t R, uint64_t keep_pol)
{
    TokenOut o;
    o.logits = a.logits;
    o.clogits = a.clogits;
    o.mml = a.mml;
    o.t = it.m * kTileTokens + (int)R;
    o.lim0 = it.ctx - a.nn + 1;  // draft row j admits t < lim0 + j
    // without slices every token below ctx is in range: the window test
    // (t < lim0 + j <= ctx) already bounds it
    o.in_slice = SLICED ? (o.t >= it.tb && o.t < it.te) : true;
    o.obase = (long long)it.i * a.nn * o.mml + o.t;
    o.hrow = a.hist ? a.hist + (long long)it.i * a.nn * kHistBins : nullptr;
    o.keep_pol = keep_pol;
    return o;
}

// Warpgroup g, warp quadrant qd (warp % 4): CTA tiles g, g + 4, g + 8, ...,
// each carried through every step by this warpgroup alone. Shared memory is
// addressed through 32-bit shared addresses throughout.
template <int H, int NN, bool SLICED, bool PAGE, bool POOL32>
static __device__ void group_role(const MainArgs &a, uint8_t *smem, CtaCtl &c, int g, int qd)
{
    const Bars B(a, smem);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint32_t R = (uint32_t)(qd * 32 + lane);  // tile row = TMEM lane
    const bool elected = qd == 0 && lane == 0;
    const uint32_t wg_bar = 1u + (uint32_t)g;
    const int count = (int)c.count;
    const uint32_t tmem_base = c.tmem_base;
    const int N = a.N, QS = a.QS;
    const uint32_t sbase = smem_u32(smem);
    const uint32_t stage = sbase + a.off_grp + (uint32_t)g * kGroupBytes;
    TileGather<PAGE, POOL32> G;
    G.init(a, stage, (uint32_t)qd, (uint32_t)lane, &B.run[warp]);
    const uint32_t w_base = sbase + a.off_w;
    const uint32_t w_slot_bytes = (uint32_t)N * 4u;
    // TMEM: this warp's lane quadrant, the group's columns
    // next_n * H in (128, 256]: one MMA pass of N = next_n * H per tile into a
    // 256-column TMEM half that warpgroups g and g ^ 2 use in turn (tile order
    // alternates between them); else passes of at most 128 columns in the
    // warpgroup's own columns
    constexpr bool kShare = NN * H > kPassCols && NN * H <= 2 * kPassCols;
    const uint32_t dcol = tmem_base + (uint32_t)(kShare ? (g & 1) * 2 * kPassCols : g * a.cols);
    const uint32_t tacc = dcol + ((uint32_t)(qd * 32) << 16);
    // MMA operands; passes of at most 128 accumulator columns (whole draft rows)
    const uint64_t adesc = sw128_kmajor_desc(stage + kSlotBytes);
    const uint64_t bdesc0 = sw128_kmajor_desc(sbase + a.off_q);
    const uint32_t q_units = (uint32_t)N * kHeadDim >> 4;
    constexpr int kRpp = kShare ? NN : (kPassCols / H < kMaxRows ? kPassCols / H : kMaxRows);  // rows per pass
    constexpr int npass = (NN + kRpp - 1) / kRpp;
    const uint64_t keep_pol = l2_evict_last_policy();

    ReqCtx<SLICED> rc;
    rc.init(a, c);
    QuerySlots<SLICED> qs;
    qs.init(a, smem, B, rc, c, count);

    Walk<SLICED> w;  // the group's current tile
    w.cur.init(rc, c);
    w.kk = 0;
    qs.pass_ends(a, smem, B, rc, c, count, w.step(rc, g, count));
    Walk<SLICED> nx = w;  // the group's next tile to gather
    uint32_t meta = 0;
    if (w.kk < count)
        meta = G.issue(w.cur, G.table_entry(w.cur));
    cp_async_commit();
    nx.step(rc, kGroups, count);
    int32_t b_nx = nx.kk < count ? G.table_entry(nx.cur) : -1;
    uint32_t mma_phase = 0;
    uint32_t use = (uint32_t)(g >> 1);  // kShare: this tile's use of the half, counting both users
    // one pass per tile: the previous tile's scores and where they go
    struct Pending {
        TokenOut out;
        float v[kRpp];
        __device__ void keep(int j, float x)
        {
#pragma unroll
            for (int u = 0; u < kRpp; ++u)
                if (j == u)
                    v[u] = x;
        }
        __device__ void flush() const
        {
#pragma unroll
            for (int u = 0; u < NN && u < kRpp; ++u)
                out(u, v[u]);
        }
    } pend;
    int pend_n = 0;

    while (w.kk < count) {
        // 1. the tile's rows have landed; 2. repack row R, scale -> register
        bool ok = G.wait_rows(&c.abort);
        const float sc = G.repack(meta);
        // 3. the group's next tile: copies now, table entries of the one after
        if (nx.kk < count)
            meta = G.issue(nx.cur, b_nx);
        cp_async_commit();
        nx.step(rc, kGroups, count);
        b_nx = nx.kk < count ? G.table_entry(nx.cur) : -1;
        // operand visible to the tensor core; the previous tile's TMEM reads done
        fence_proxy_async_smem();
        tc_fence_before_sync();
        named_bar_sync(wg_bar, 128);
        tc_fence_after_sync();
        const int q_slot = qs.slot;
        if (!qs.have) {
            ok = mbar_wait(&B.qfull[q_slot], qs.phase, &c.abort) && ok;
            qs.have = true;
        }
        // weights of the request: valid after the query-slot wait above
        const uint32_t wsl = launder_u32(w_base + (uint32_t)q_slot * w_slot_bytes);
        const TokenOut out = token_out(a, w.cur, R, keep_pol);
        const uint32_t flip = sc < 0.0f ? 0x80000000u : 0u;
        const float mag = fabsf(sc);
        const bool all_pos = __all_sync(kFullMask, flip == 0u);
        // a shared half goes to the other warpgroup once each of the four
        // warps has read its lanes (one arrival per warp, no warpgroup
        // barrier), before the tile's outputs; an arrival even after a
        // failed wait keeps the phases in step
        auto release = [&]() {
            if constexpr (kShare) {
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&B.tfree[g & 1]);
            }
        };
        if constexpr (npass == 1) {
            // one pass in the warpgroup's own columns: the tile's outputs are
            // written during the next tile's MMA (the scores wait in
            // registers). With a shared half they are written at once (the
            // half's wait leaves nothing to hide them behind, and deferring
            // them measured slower).
            bool mma_ok = true;
            if (elected) {
                // a shared half: the other warpgroup's previous tile has read it
                if (kShare && use > 0)
                    mma_ok = mbar_wait(&B.tfree[g & 1], (use - 1u) & 1u, &c.abort);
                if (mma_ok) {
                    tc_fence_after_sync();
                    const uint64_t bd = bdesc0 + (uint64_t)((uint32_t)q_slot * q_units);
                    const uint32_t idesc = idesc_e4m3_f32(128, NN * H);
#pragma unroll
                    for (int k4 = 0; k4 < kHeadDim / 32; ++k4)
                        umma_e4m3(dcol, adesc + 2u * k4, bd + 2u * k4, idesc, k4 > 0 ? 1u : 0u);
                    umma_commit(&B.mma[g]);
                }
            }
            if (pend_n) {
                pend.flush();
                pend_n = 0;
            }
            // the elected thread waits for the MMAs; the rest of the group
            // sleeps on the named barrier meanwhile
            if (elected && mma_ok)
                mma_ok = mbar_wait(&B.mma[g], mma_phase, &c.abort);
            mma_phase ^= 1u;
            ok = named_bar_and(wg_bar, 128, mma_ok) && ok;
            tc_fence_after_sync();
            // one outcome per warp: the tile body uses warp-wide votes
            if (__all_sync(kFullMask, ok)) {
                if constexpr (kShare) {
                    epi_dispatch<H, kRpp>(NN, all_pos, tacc, wsl, flip, mag, 0, out, release);
                } else {
                    pend.out = out;
                    auto keep = [&](int j, float v) { pend.keep(j, v); };
                    epi_dispatch<H, kRpp>(NN, all_pos, tacc, wsl, flip, mag, 0, keep, release);
                    pend_n = NN;
                }
            } else {
                release();
                raise_abort(a, c);
            }
        } else {
            // passes of at most 128 columns (next_n * H above 256): each pass
            // reuses the columns once all four warps have read the last
            // (a warpgroup barrier), outputs at once
#pragma unroll
            for (int p = 0; p < npass; ++p) {
                const int j0 = p * kRpp, nr = min(kRpp, NN - j0);
                bool mma_ok = true;
                if (elected) {
                    tc_fence_after_sync();
                    const uint64_t bd = bdesc0 + (uint64_t)((uint32_t)q_slot * q_units +
                                                            ((uint32_t)(j0 * H * kHeadDim) >> 4));
                    const uint32_t idesc = idesc_e4m3_f32(128, nr * H);
#pragma unroll
                    for (int k4 = 0; k4 < kHeadDim / 32; ++k4)
                        umma_e4m3(dcol, adesc + 2u * k4, bd + 2u * k4, idesc, k4 > 0 ? 1u : 0u);
                    umma_commit(&B.mma[g]);
                    mma_ok = mbar_wait(&B.mma[g], mma_phase, &c.abort);
                }
                mma_phase ^= 1u;
                ok = named_bar_and(wg_bar, 128, mma_ok) && ok;
                tc_fence_after_sync();
                if (__all_sync(kFullMask, ok)) {
                    const uint32_t wj0 = wsl + (uint32_t)(j0 * H * 4);
                    epi_dispatch<H, kRpp>(nr, all_pos, tacc, wj0, flip, mag, j0, out, release);
                } else {
                    raise_abort(a, c);
                }
                if (p + 1 < npass) {  // the next pass reuses the columns
                    tc_fence_before_sync();
                    named_bar_sync(wg_bar, 128);
                    tc_fence_after_sync();
                }
            }
        }
        if constexpr (kShare)
            use += 2u;
        qs.pass_ends(a, smem, B, rc, c, count, w.step(rc, kGroups, count));
    }
    if (pend_n)
        pend.flush();
    cp_async_wait_all();
    qs.drain(B, QS);
}

}  // namespace pmqa
