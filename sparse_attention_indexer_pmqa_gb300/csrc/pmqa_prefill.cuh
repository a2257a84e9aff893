// pmqa_prefill.cuh -- the non-paged (prefill) FP8 MQA-logits kernel for sm_103a.
//
// Definition (page "[Bug] aiter ops triton attention pa", section "Observations
// while narrowing it down", which names the prefill indexer `fp8_mqa_logits`
// beside the paged decode kernel; its arithmetic is the decode one of section
// "Minimal reproduction" with the paging removed): for query row r and key n,
// logit = sum_h w[r][h] * relu(s_n * q[r][h] . k_n) for ks[r] <= n < ke[r],
// -inf elsewhere.
//
// A CTA works on super-groups of 4 * G query rows (G = 128 / heads, so one
// warpgroup's G rows fill 128 accumulator columns) and walks a contiguous,
// tile-balanced range of (super-group, 128-key tile) items. Each key tile is
// loaded once by TMA, already in the 128B-swizzled K-major operand layout, into
// a ring of S stages that all four warpgroups read: warpgroup g multiplies it
// by the Q rows of its G query rows, D[key][(row, h)] in its own 128 TMEM
// columns, and reduces its accumulators with the same epilogue as the paged
// kernel (thread = key = TMEM lane). The last warpgroup whose MMA on a stage
// completes refills that stage with the tile S items ahead. Query rows and
// weights of the super-group QS ahead are loaded at super-group ends, as in the
// paged kernel. Every wait is bounded.
#pragma once

#include "pmqa_main.cuh"

namespace pmqa {

constexpr int kPfMaxStages = 4;

struct PfArgs {
    CUtensorMap tmap_q;  // q as [m * heads rows, 128 bytes], 128B swizzle, box [128, q_box]
    CUtensorMap tmap_k;  // k as [n rows, 128 bytes], 128B swizzle, box [128, 128]
    const float *k_scale;
    const float *w;
    const int32_t *ks, *ke;
    float *logits;  // [m, n]
    uint32_t *status;
    int m, n;
    int G;     // query rows per warpgroup (128 / heads)
    int SGR;   // query rows per super-group (4 * G)
    int n_sg;  // super-groups: ceil(m / SGR)
    int S, QS, q_box;
    uint32_t off_k, off_q, off_w, off_bar, smem_bytes;
};

// Tile range [lo, lo + nt) of super-group sg: the union of its rows' key ranges.
struct PfRange {
    int lo, nt;
};

__device__ __forceinline__ PfRange pf_range(const PfArgs &a, int sg)
{
    int lo = 0x7FFFFFFF, hi = 0;
    const int r0 = sg * a.SGR, r1 = min(r0 + a.SGR, a.m);
    for (int r = r0; r < r1; ++r) {
        const int s = max(__ldg(a.ks + r), 0), e = min(__ldg(a.ke + r), a.n);
        if (e > s) {
            lo = min(lo, s);
            hi = max(hi, e);
        }
    }
    PfRange R;
    if (hi == 0) {
        R.lo = 0;
        R.nt = 0;
    } else {
        R.lo = lo / kTileTokens;
        R.nt = (hi + kTileTokens - 1) / kTileTokens - R.lo;
    }
    return R;
}

// Position (super-group sg, tile m of nt, first tile lo) in a CTA's walk over
// (super-group, tile) items; empty super-groups are skipped.
struct PfPos {
    int sg, m, nt, lo;
    __device__ void at(const PfArgs &a, int g, int mm)
    {
        sg = g;
        m = mm;
        if (sg < a.n_sg) {
            const PfRange R = pf_range(a, sg);
            nt = R.nt;
            lo = R.lo;
        } else {
            nt = 0;
            lo = 0;
        }
    }
    __device__ void next(const PfArgs &a)
    {
        if (++m < nt)
            return;
        m = 0;
        do {
            if (++sg >= a.n_sg) {
                nt = 0;
                return;
            }
            const PfRange R = pf_range(a, sg);
            nt = R.nt;
            lo = R.lo;
        } while (nt == 0);
    }
    __device__ int tile() const { return lo + m; }
};

// Shared-memory mbarriers of the prefill kernel, and the per-stage counters of
// warpgroups done with a stage.
//   kfull[S]   a key tile landed in stage s
//   qfull[QS]  query rows + weights of a super-group landed
//   mma[4]     a warpgroup's MMA finished
struct PfBars {
    uint64_t *kfull, *qfull, *mma;
    int *done;
    __device__ PfBars(const PfArgs &a, uint8_t *smem)
    {
        kfull = reinterpret_cast<uint64_t *>(smem + a.off_bar);
        qfull = kfull + a.S;
        mma = qfull + a.QS;
        done = reinterpret_cast<int *>(mma + kGroups);
    }
};

__device__ __forceinline__ void pf_load_k(const PfArgs &a, uint32_t kbase, const PfBars &B, int s,
                                          int tile)
{
    mbar_arrive_expect_tx(&B.kfull[s], kStageBytes);
    tma_load_2d(kbase + (uint32_t)s * kStageBytes, &a.tmap_k, 0, tile * kTileTokens, &B.kfull[s]);
}

// Query rows (TMA boxes; rows past m read as zeros) and the weights of the
// super-group's rows that exist (bulk copy) into query slot `slot`.
__device__ __forceinline__ void pf_load_query(const PfArgs &a, uint8_t *smem, const PfBars &B,
                                              int slot, int sg, int heads)
{
    const int N = a.SGR * heads;
    const uint32_t q_bytes = (uint32_t)N * kHeadDim, w_bytes_slot = (uint32_t)N * 4u;
    const int rows = min(a.SGR, a.m - sg * a.SGR);
    const uint32_t w_bytes = (uint32_t)(rows * heads) * 4u;
    const uint32_t qdst = smem_u32(smem + a.off_q) + (uint32_t)slot * q_bytes;
    mbar_arrive_expect_tx(&B.qfull[slot], q_bytes + w_bytes);
    for (int nc = 0; nc * a.q_box < N; ++nc)
        tma_load_2d(qdst + (uint32_t)(nc * a.q_box * kHeadDim), &a.tmap_q, 0,
                    sg * N + nc * a.q_box, &B.qfull[slot]);
    bulk_load(smem_u32(smem + a.off_w) + (uint32_t)slot * w_bytes_slot,
              a.w + (long long)sg * N, w_bytes, &B.qfull[slot]);
}

// Warpgroup g, warp quadrant qd: every item of the CTA's range, query rows
// g * G .. g * G + G - 1 of each super-group.
template <int H>
static __device__ void pf_group_role(const PfArgs &a, uint8_t *smem, CtaCtl &c, int g, int qd)
{
    constexpr int G = kPassCols / H;
    const PfBars B(a, smem);
    const int lane = threadIdx.x & 31;
    const uint32_t R = (uint32_t)(qd * 32 + lane);  // key of the tile = TMEM lane
    const bool elected = qd == 0 && lane == 0;
    const uint32_t wg_bar = 1u + (uint32_t)g;
    const int count = (int)c.count;
    const int S = a.S, QS = a.QS, SGR = a.SGR, m = a.m, n = a.n;
    const uint32_t sbase = smem_u32(smem);
    const uint32_t kbase = sbase + a.off_k;
    const uint32_t q_slot_bytes = (uint32_t)(SGR * H * kHeadDim);
    const uint32_t w_slot_bytes = (uint32_t)(SGR * H * 4);
    // this warpgroup's G query rows inside a query slot
    const uint32_t q_off = (uint32_t)(g * G * H * kHeadDim);
    const uint32_t w_off = (uint32_t)(g * G * H * 4);
    const uint32_t dcol = c.tmem_base + (uint32_t)(g * kPassCols);
    const uint32_t tacc = dcol + ((uint32_t)(qd * 32) << 16);
    const uint32_t idesc = idesc_e4m3_f32(128, G * H);
    float *const logits = a.logits;
    const float NEG_INF = -__int_as_float(0x7f800000);

    int q_slot = 0;
    uint32_t q_phase = 0;
    bool have_q = false;
    int loads = 0;  // query loads issued (thread 0)
    PfPos nxt;      // next super-group whose query is to be loaded (thread 0)
    nxt.at(a, c.i0, c.m0);
    int nxt_first = 0;  // CTA item index of nxt's current tile
    auto nxt_valid = [&]() { return nxt.nt > 0 && nxt_first < count; };
    auto nxt_advance = [&]() {
        nxt_first += nxt.nt - nxt.m;
        nxt.m = nxt.nt - 1;
        nxt.next(a);
    };
    if (threadIdx.x == 0) {
        for (int u = 0; u < QS; ++u) {
            if (nxt_valid()) {
                pf_load_query(a, smem, B, u, nxt.sg, H);
                ++loads;
            }
            nxt_advance();
        }
    }
    // key tiles: thread 0 fills the first S stages; afterwards the last
    // warpgroup done with a stage refills it (pre = the tile S items ahead)
    PfPos pre;
    pre.at(a, c.i0, c.m0);
    if (threadIdx.x == 0)
        for (int s = 0; s < S && s < count; ++s) {
            pf_load_k(a, kbase, B, s, pre.tile());
            pre.next(a);
        }
    else if (elected)
        for (int s = 0; s < S && s < count; ++s)
            pre.next(a);

    PfPos cur;
    cur.at(a, c.i0, c.m0);
    int rks[G], rke[G];  // key ranges of this warpgroup's rows in the current super-group
    int r0 = 0, nr = 0;
    uint32_t mma_phase = 0;
    for (int kk = 0; kk < count; ++kk) {
        const int s = kk % S;
        const uint32_t kphase = (uint32_t)(kk / S) & 1u;
        const int tile = cur.tile();
        const int t = tile * kTileTokens + (int)R;
        const float sc = t < n ? __ldg(a.k_scale + t) : 0.0f;
        if (!have_q) {
            r0 = cur.sg * SGR + g * G;
            nr = max(0, min(G, m - r0));
#pragma unroll
            for (int j = 0; j < G; ++j) {
                rks[j] = j < nr ? __ldg(a.ks + r0 + j) : 0;
                rke[j] = j < nr ? __ldg(a.ke + r0 + j) : 0;
            }
        }
        // the previous epilogue's TMEM reads are done before the MMA overwrites
        tc_fence_before_sync();
        named_bar_sync(wg_bar, 128);
        tc_fence_after_sync();
        bool ok = true;
        if (!have_q) {
            ok = mbar_wait(&B.qfull[q_slot], q_phase, &c.abort);
            have_q = true;
        }
        bool mma_ok = true;
        if (elected) {
            mma_ok = mbar_wait(&B.kfull[s], kphase, &c.abort) && ok;
            if (mma_ok) {
                tc_fence_after_sync();
                const uint64_t ad = sw128_kmajor_desc(kbase + (uint32_t)s * kStageBytes);
                const uint64_t bd = sw128_kmajor_desc(sbase + a.off_q + (uint32_t)q_slot * q_slot_bytes +
                                                      q_off);
#pragma unroll
                for (int k4 = 0; k4 < kHeadDim / 32; ++k4)
                    umma_e4m3(dcol, ad + 2u * k4, bd + 2u * k4, idesc, k4 > 0 ? 1u : 0u);
                umma_commit(&B.mma[g]);
                mma_ok = mbar_wait(&B.mma[g], mma_phase, &c.abort);
            }
            // the stage is free once all four warpgroups' MMAs on it completed;
            // the fourth to get here refills it
            const int done = atomicAdd(&B.done[s], 1) + 1;
            if ((done & 3) == 0 && kk + S < count && !aborted(c))
                pf_load_k(a, kbase, B, s, pre.tile());
            if (kk + S < count)
                pre.next(a);
        }
        mma_phase ^= 1u;
        ok = named_bar_and(wg_bar, 128, mma_ok) && ok;
        tc_fence_after_sync();
        if (__all_sync(kFullMask, ok)) {
            if (nr > 0) {
                const uint32_t wsl =
                    launder_u32(sbase + a.off_w + (uint32_t)q_slot * w_slot_bytes + w_off);
                const uint32_t flip = sc < 0.0f ? 0x80000000u : 0u;
                const float mag = fabsf(sc);
                const bool all_pos = __all_sync(kFullMask, flip == 0u);
                float *const orow = logits + (long long)r0 * n + t;
                auto out = [&](int j, float v) {
                    if (t < n && j < nr)
                        orow[(long long)j * n] = (t >= rks[j] && t < rke[j]) ? v : NEG_INF;
                };
                epi_dispatch<H, G>(nr, all_pos, tacc, wsl, flip, mag, 0, out);
            }
        } else {
            c.abort = 1;
            atomicOr(a.status, 0x4u);
        }
        // super-group end: all warpgroups meet, thread 0 loads the query of
        // the super-group QS ahead into the freed slot
        const bool last_of_sg = cur.m == cur.nt - 1 || kk == count - 1;
        cur.next(a);
        if (last_of_sg) {
            named_bar_sync(kCtaBarrier, kMaxThreads);
            if (threadIdx.x == 0) {
                if (nxt_valid() && !aborted(c)) {
                    pf_load_query(a, smem, B, q_slot, nxt.sg, H);
                    ++loads;
                }
                nxt_advance();
            }
            if (++q_slot == QS) {
                q_slot = 0;
                q_phase ^= 1u;
            }
            have_q = false;
        }
    }
    // after an abort, copies nobody consumed land before the CTA exits (bounded)
    if (threadIdx.x == 0)
        for (int u = loads > QS ? loads - QS : 0; u < loads; ++u)
            mbar_wait(&B.qfull[u % QS], (uint32_t)(u / QS) & 1u, nullptr);
}

template <int H>
__global__ void __launch_bounds__(kMaxThreads, 1) pmqa_prefill_kernel(const __grid_constant__ PfArgs a)
{
    extern __shared__ uint8_t smem_raw[];
    __shared__ CtaCtl ctl;
    uint8_t *const smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const int warp = threadIdx.x >> 5;

    if (threadIdx.x == 0) {
        ctl.abort = 0;
        const PfBars B(a, smem);
        for (int s = 0; s < a.S; ++s) {
            mbar_init(&B.kfull[s], 1);
            B.done[s] = 0;
        }
        for (int q = 0; q < a.QS; ++q)
            mbar_init(&B.qfull[q], 1);
        for (int g = 0; g < kGroups; ++g)
            mbar_init(&B.mma[g], 1);
        mbar_init_fence();
    }
    __syncwarp();
    if (warp == 0)
        tmem_alloc(&ctl.tmem_base, (uint32_t)(kGroups * kPassCols));

    balance_schedule(a.n_sg, [&](int sg) { return (long long)pf_range(a, sg).nt; }, ctl);
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();

    // -inf outside the tiles each row's super-group covers: CTA b takes rows
    // b, b + grid, ...; its 16 warps stride over each row's two segments.
    {
        const long long n = a.n;
        for (int r = blockIdx.x; r < a.m; r += gridDim.x) {
            const PfRange Rg = pf_range(a, r / a.SGR);
            const long long c0 = Rg.nt > 0 ? (long long)Rg.lo * kTileTokens : n;
            const long long c1 =
                Rg.nt > 0 ? min((long long)(Rg.lo + Rg.nt) * kTileTokens, n) : n;
            float *row = a.logits + (long long)r * n;
            const float NEG_INF = -__int_as_float(0x7f800000);
            for (long long x = threadIdx.x; x < c0; x += blockDim.x)
                row[x] = NEG_INF;
            for (long long x = c1 + threadIdx.x; x < n; x += blockDim.x)
                row[x] = NEG_INF;
        }
    }

    pf_group_role<H>(a, smem, ctl, warp >> 2, warp & 3);

    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    if (warp == 0)
        tmem_dealloc(ctl.tmem_base, (uint32_t)(kGroups * kPassCols));
}

}  // namespace pmqa
