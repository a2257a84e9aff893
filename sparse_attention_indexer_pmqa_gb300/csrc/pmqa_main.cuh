// pmqa_main.cuh -- the persistent FP8 paged MQA-logits kernel for sm_103a.
//
// Definition (page "[Bug] aiter ops triton attention pa", section "Minimal
// reproduction", reference function `torch_ref`): for query row r = (i, j) and
// token t, logit = sum_h w[r][h] * relu(s_t * q[i][j][h] . k_t), -inf outside
// t < ctx_i, t <= ctx_i - next_n + j.
//
// One CTA per SM walks a contiguous range of (request, 128-token tile) work
// items, balanced by tile count over all requests. Warp roles:
//   warp 0        allocates TMEM; lane 0 issues tcgen05.mma
//   warps 1..4    gather: block-table lookup, then per token one warp-wide
//                 4-byte cp.async of the 128 fp8 bytes straight into the
//                 128B-swizzled K-major operand tile, plus the fp32 scale
//   warps 5..     epilogue work groups (1 or 2 x 4 warps): tcgen05.ld of the
//                 fp32 scores (one token per thread, all heads of a row in
//                 registers), relu * weight head sum, scale, mask, store;
//                 optionally the streaming top-k of pmqa_topk_wg.cuh.
// The MMA computes D[token][(j,h)] = K_tile[128 x 128] * Q[(j,h) x 128]^T with
// tokens as M = 128 and N = next_n * heads, fp8 e4m3 in, fp32 accumulate in
// TMEM. Pipelines: S shared-memory K stages, NBUF TMEM accumulators, QS query
// slots, a scale ring of S + NBUF entries; all handshakes are mbarriers.
#pragma once

#include <cstdint>

#include "pmqa_ptx.cuh"
#include "pmqa_topk_wg.cuh"

namespace pmqa {

constexpr int kTileTokens = 128;
constexpr int kHeadDim = 128;
constexpr int kKvRowBytes = kHeadDim + 4;
constexpr int kProducerWarps = 4;
constexpr int kFirstEpiWarp = 1 + kProducerWarps;
constexpr uint32_t kStageBytes = kTileTokens * kHeadDim;  // 16 KB

struct MainArgs {
    const uint8_t *q;
    const uint8_t *kv;
    const float *w;
    const int32_t *ctx_lens;
    const int32_t *bt;
    long long num_blocks;
    int bs, nn, P, W, mml;
    float *logits;  // may be null in the fused kernel
    int k;
    int32_t *out_idx;
    float *out_vals;
    TopkWs ws;
    // shared-memory / pipeline layout, computed on the host
    int N, S, NBUF, QS, RS, cols, tmem_cols, E, rpw, cap;
    uint32_t off_q, off_w, off_scale, off_bar, off_cand, smem_bytes;
};

struct CtaCtl {
    long long red[16];
    int wsum[16];
    long long start, count;
    int i0, m0;
    int abort;
    uint32_t tmem_base;
};

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

// Split `total` units (per-item counts given by len_of) evenly over the grid.
// Every thread calls it; results land in c.start/c.count/c.i0/c.m0.
template <class LenFn>
static __device__ void balance_schedule(int n_items, LenFn len_of, CtaCtl &c)
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

// sfull: the scale ring slot of a tile has landed. The epilogue reads the
// scales written by the gather warps, so it acquires them from those warps'
// own barrier rather than through the MMA thread.
struct Bars {
    uint64_t *full, *empty, *tfull, *tempty, *qfull, *qempty, *sfull, *done;
    __device__ Bars(const MainArgs &a, uint8_t *smem)
    {
        full = reinterpret_cast<uint64_t *>(smem + a.off_bar);
        empty = full + a.S;
        tfull = empty + a.S;
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
    default: cp_async_wait_group<5>(); break;
    }
}

__device__ __forceinline__ void raise_abort(const MainArgs &a, CtaCtl &c)
{
    c.abort = 1;
    atomicOr(a.ws.status, 0x4u);
}

// ---------------------------------------------------------------- gather

static __device__ void producer_role(const MainArgs &a, uint8_t *smem, CtaCtl &c, int pw)
{
    const Bars B(a, smem);
    const int lane = threadIdx.x & 31, ptid = pw * 32 + lane;
    const uint64_t pol = l2_evict_first_policy();
    const int N = a.N, lag = a.S - 1;
    const int count = (int)c.count;
    TileIter it;
    it.init(a, c.i0, c.m0);
    uint32_t req = 0, hist_first = 0, hist_qs = 0;
    int kk = 0;
    bool ok = true;
    for (; kk < count; ++kk) {
        const int s = kk % a.S;
        if (!mbar_wait(&B.empty[s], ((kk / a.S) & 1) ^ 1, &c.abort)) {
            ok = false;
            break;
        }
        const bool first = kk == 0 || it.m == 0;
        uint32_t qs = 0;
        if (first) {
            qs = req % a.QS;
            if (!mbar_wait(&B.qempty[qs], ((req / a.QS) & 1) ^ 1, &c.abort)) {
                ok = false;
                break;
            }
            // q rows (j, h) of request i into the swizzled B-operand slot
            const uint8_t *qsrc = a.q + (long long)it.i * N * kHeadDim;
            const uint32_t qdst = smem_u32(smem + a.off_q + qs * (uint32_t)N * kHeadDim);
            for (int ch = ptid; ch < N * 8; ch += 128) {
                const int n = ch >> 3, cc = ch & 7;
                cp_async_16(qdst + (n >> 3) * 1024 + (n & 7) * 128 + ((cc ^ (n & 7)) << 4),
                            qsrc + n * kHeadDim + cc * 16);
            }
            const float *wsrc = a.w + (long long)it.i * N;
            const uint32_t wdst = smem_u32(smem + a.off_w + qs * (uint32_t)N * 4);
            for (int ch = ptid; ch < N / 4; ch += 128)
                cp_async_16(wdst + ch * 16, wsrc + ch * 4);
            ++req;
        }
        // this warp's 32 tokens of the tile
        const int t = it.m * kTileTokens + pw * 32 + lane;
        const uint8_t *rowp = a.kv;
        uint32_t nb = 0;
        if (t < it.ctx) {
            const int blk = t / a.P;
            const int off = t - blk * a.P;
            const int b = __ldg(a.bt + (long long)it.i * a.W + blk);
            if (b >= 0 && (long long)b < a.num_blocks) {
                rowp = a.kv + ((long long)b * a.P + off) * kKvRowBytes;
                nb = 4;
            } else {
                atomicOr(a.ws.status, 0x1u);
            }
        }
        const uint32_t sbase = smem_u32(smem + (uint32_t)s * kStageBytes);
        const uint32_t chunk_off = (uint32_t)(lane & 3) * 4;
        const uint32_t chunk_id = (uint32_t)lane >> 2;
#pragma unroll 8
        for (int jj = 0; jj < 32; ++jj) {
            const uint8_t *src = reinterpret_cast<const uint8_t *>(
                __shfl_sync(kFullMask, reinterpret_cast<unsigned long long>(rowp), jj));
            const uint32_t n = __shfl_sync(kFullMask, nb, jj);
            const uint32_t r = (uint32_t)(pw * 32 + jj);
            cp_async_4(sbase + r * 128 + ((chunk_id ^ (r & 7)) << 4) + chunk_off, src + lane * 4,
                       n, pol);
        }
        const int sri = kk % a.RS;
        cp_async_4(smem_u32(smem + a.off_scale + sri * 512 + (pw * 32 + lane) * 4),
                   rowp + kHeadDim, nb, pol);
        cp_async_commit();
        hist_first = (hist_first << 1) | (first ? 1u : 0u);
        hist_qs = (hist_qs << 1) | qs;
        if (kk >= lag) {
            cp_async_wait_upto(lag);
            fence_proxy_async_smem();
            mbar_arrive(&B.full[(kk - lag) % a.S]);
            mbar_arrive(&B.sfull[(kk - lag) % a.RS]);
            if ((hist_first >> lag) & 1u)
                mbar_arrive(&B.qfull[(hist_qs >> lag) & 1u]);
        }
        it.next(a);
    }
    cp_async_wait_all();
    fence_proxy_async_smem();
    if (!ok) {
        raise_abort(a, c);
        return;
    }
    for (int d = lag - 1; d >= 0; --d) {
        const int kd = kk - 1 - d;
        if (kd < 0)
            continue;
        mbar_arrive(&B.full[kd % a.S]);
        mbar_arrive(&B.sfull[kd % a.RS]);
        if ((hist_first >> d) & 1u)
            mbar_arrive(&B.qfull[(hist_qs >> d) & 1u]);
    }
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
        if (!mbar_wait(&B.full[s], (kk / a.S) & 1, &c.abort) ||
            !mbar_wait(&B.tempty[b], ((kk / a.NBUF) & 1) ^ 1, &c.abort)) {
            ok = false;
            break;
        }
        tc_fence_after_sync();
        const uint32_t abase = smem_u32(smem + (uint32_t)s * kStageBytes);
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
        umma_commit(&B.empty[s]);
        umma_commit(&B.tfull[b]);
        if (kk == count - 1 || it.m == it.nt - 1) {
            umma_commit(&B.qempty[qs]);
            ++req;
        }
        it.next(a);
    }
    if (!ok)
        raise_abort(a, c);
    // all MMAs issued by this thread have completed once `done` flips
    umma_commit(B.done);
    if (!mbar_wait(B.done, 0, nullptr))
        atomicOr(a.ws.status, 0x4u);
}

// ---------------------------------------------------------------- epilogue

// Scores of rows j = g, g + E, ... for this thread's token: TMEM columns
// [j*H, j*H + H) of buffer b. Releases the TMEM buffer after the last load.
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

// Wait on an mbarrier for a whole work group and agree on the outcome.
__device__ __forceinline__ bool wg_wait(uint64_t *bar, uint32_t parity, CtaCtl &c, const Wg &g)
{
    if (g.warp == 0) {
        const bool ok = mbar_wait(bar, parity, &c.abort);
        if (g.lane == 0)
            g.scr->flag = ok ? 1u : 0u;
    }
    g.sync();
    const bool ok = g.scr->flag != 0;
    g.sync();
    return ok;
}

template <int H, bool FUSED>
static __device__ void epilogue_role(const MainArgs &a, uint8_t *smem, CtaCtl &c, int g, int we)
{
    const Bars B(a, smem);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, qd = warp & 3;
    const int r = qd * 32 + lane;  // token row of the tile = TMEM lane
    const int N = a.N, nn = a.nn, E = a.E;
    const float NEG_INF = -__int_as_float(0x7f800000);

    // per-work-group top-k state
    uint8_t *cbase = smem + a.off_cand +
                     (uint32_t)g * ((uint32_t)a.rpw * (uint32_t)a.cap * 8u + 64u +
                                    (uint32_t)sizeof(WgScratch));
    Wg wg;
    wg.tid = (uint32_t)(we * 32 + lane);
    wg.lane = (uint32_t)lane;
    wg.warp = (uint32_t)we;
    wg.bar = 1u + (uint32_t)g;
    wg.scr = reinterpret_cast<WgScratch *>(cbase + (uint32_t)a.rpw * a.cap * 8u + 64u);
    CandBuf cb[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
        cb[u].key = reinterpret_cast<uint32_t *>(cbase) + (uint32_t)u * a.cap;
        cb[u].pos = reinterpret_cast<int32_t *>(cbase + (uint32_t)a.rpw * a.cap * 4u) +
                    (uint32_t)u * a.cap;
        cb[u].count = reinterpret_cast<uint32_t *>(cbase + (uint32_t)a.rpw * a.cap * 8u) + 2 * u;
        cb[u].thresh = cb[u].count + 1;
        cb[u].cap = (uint32_t)a.cap;
    }
    const int rows_here = (nn - g + E - 1) / E;

    // -inf beyond the last tile of each row: this CTA's share of every row
    if (a.logits) {
        const int etid = g * 128 + we * 32 + lane, ethr = E * 128;
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
    if constexpr (FUSED) {
        // requests with no tokens: no segment will ever merge their rows
        if (blockIdx.x == 0 && g == 0) {
            for (int rr = 0; rr < a.bs * nn; ++rr) {
                if (ctx_of(a, rr / nn) > 0)
                    continue;
                for (int e = wg.tid; e < a.k; e += 128) {
                    a.out_idx[(long long)rr * a.k + e] = -1;
                    if (a.out_vals)
                        a.out_vals[(long long)rr * a.k + e] = NEG_INF;
                }
            }
        }
        for (int u = 0; u < rows_here; ++u)
            cand_reset(cb[u], wg);
    }

    const int count = (int)c.count;
    TileIter it;
    it.init(a, c.i0, c.m0);
    uint32_t req = 0, seg_tiles = 0;
    for (int kk = 0; kk < count; ++kk) {
        const int b = kk % a.NBUF;
        const uint32_t qs = req % a.QS;
        const bool first = kk == 0 || it.m == 0;
        if (first) {
            seg_tiles = 0;
            bool ok;
            if constexpr (FUSED)
                ok = wg_wait(&B.qfull[qs], (req / a.QS) & 1, c, wg);
            else
                ok = mbar_wait(&B.qfull[qs], (req / a.QS) & 1, &c.abort);
            if (!ok) {
                raise_abort(a, c);
                break;
            }
        }
        const int sri = kk % a.RS;
        const uint32_t sph = (uint32_t)(kk / a.RS) & 1u;
        bool ok;
        if constexpr (FUSED)
            ok = wg_wait(&B.sfull[sri], sph, c, wg) &&
                 wg_wait(&B.tfull[b], (kk / a.NBUF) & 1, c, wg);
        else
            ok = mbar_wait(&B.sfull[sri], sph, &c.abort) &&
                 mbar_wait(&B.tfull[b], (kk / a.NBUF) & 1, &c.abort);
        if (!ok) {
            raise_abort(a, c);
            break;
        }
        tc_fence_after_sync();
        const float sc =
            reinterpret_cast<const float *>(smem + a.off_scale)[sri * kTileTokens + r];
        const int t = it.m * kTileTokens + r;
        const float *wsl = reinterpret_cast<const float *>(smem + a.off_w + qs * (uint32_t)N * 4);
        const uint32_t taddr = c.tmem_base + ((uint32_t)(qd * 32) << 16) + (uint32_t)(b * a.cols);
        float logit[2];
        epi_rows<H>(taddr, wsl, sc, g, E, nn, logit, &B.tempty[b], lane);

        for (int u = 0; u < rows_here; ++u) {
            const int j = g + u * E;
            const bool valid = t < valid_len(it.ctx, nn, j);
            if (a.logits && t < a.mml)
                a.logits[((long long)it.i * nn + j) * a.mml + t] = valid ? logit[u] : NEG_INF;
            if constexpr (FUSED) {
                const uint32_t key = f32_order_key(logit[u]);
                cand_append(cb[u], wg, key, t, valid && key >= *cb[u].thresh);
            }
        }
        ++seg_tiles;
        if constexpr (FUSED) {
            for (int u = 0; u < rows_here; ++u)
                cand_make_room(cb[u], (uint32_t)a.k, wg);
        }
        if (kk == count - 1 || it.m == it.nt - 1) {
            if constexpr (FUSED) {
                for (int u = 0; u < rows_here; ++u) {
                    const int j = g + u * E;
                    const uint32_t vl = (uint32_t)valid_len(it.ctx, nn, j);
                    const uint32_t k_eff = vl < (uint32_t)a.k ? vl : (uint32_t)a.k;
                    segment_finish(cb[u], a.ws, (long long)it.i * nn + j, seg_tiles,
                                   (uint32_t)it.nt, (uint32_t)a.k, k_eff, a.out_idx, a.out_vals,
                                   wg);
                }
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

template <int H, bool FUSED>
__global__ void __launch_bounds__(32 * (kFirstEpiWarp + 8), 1)
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
            mbar_init(&B.full[s], 32 * kProducerWarps);
            mbar_init(&B.empty[s], 1);
        }
        for (int b = 0; b < a.NBUF; ++b) {
            mbar_init(&B.tfull[b], 1);
            mbar_init(&B.tempty[b], 4 * a.E);
        }
        for (int q = 0; q < a.QS; ++q) {
            mbar_init(&B.qfull[q], 32 * kProducerWarps);
            mbar_init(&B.qempty[q], 1 + 4 * a.E);
        }
        for (int q = 0; q < a.RS; ++q)
            mbar_init(&B.sfull[q], 32 * kProducerWarps);
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
                atomicOr(a.ws.status, 0x2u);
        }
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();

    if (warp == 0) {
        if ((threadIdx.x & 31) == 0)
            mma_role(a, smem, ctl);
        __syncwarp();
    } else if (warp < kFirstEpiWarp) {
        producer_role(a, smem, ctl, warp - 1);
    } else {
        const int e = warp - kFirstEpiWarp;
        epilogue_role<H, FUSED>(a, smem, ctl, e >> 2, e & 3);
    }

    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    __syncwarp();
    if (warp == 0)
        tmem_dealloc(ctl.tmem_base, (uint32_t)a.tmem_cols);
}

}  // namespace pmqa
