// pmqa_prefill.cuh -- the non-paged (prefill) FP8 MQA-logits kernel for sm_103a.
//
// Definition (page "[Bug] aiter ops triton attention pa", section "Observations
// while narrowing it down", which names the prefill indexer `fp8_mqa_logits`
// beside the paged decode kernel; its arithmetic is the decode one of section
// "Minimal reproduction" with the paging removed): for query row r and key n,
// logit = sum_h w[r][h] * relu(s_n * q[r][h] . k_n) for ks[r] <= n < ke[r],
// -inf elsewhere.
//
// Two launches. The prep kernel reduces each super-group's rows (SGR = 4 G
// query rows, G = 128 / heads) to the range of 128-key tiles their key ranges
// touch, and writes -inf outside it. The main kernel, one CTA per SM, walks a
// contiguous, tile-balanced range of (super-group, key tile) items. Warp 16 is
// the control warp: its lane 0 loads every key tile (TMA, already in the
// 128B-swizzled K-major operand layout, a ring of S stages) and every query
// slot, and issues every MMA: per item, one N = 256 MMA per warpgroup pair p,
// D[key][(row, h)] = K_tile * Q^T for the 2 G rows of warpgroups 2p and 2p + 1,
// into TMEM columns [256 p, 256 p + 256). Warps 0-15 are four warpgroups;
// warpgroup g reduces columns [128 g, 128 g + 128), its G rows (thread = key =
// TMEM lane): sum_h w[row][h] * relu(s_key * x), masked to the row's key
// range. The pairs run independently of each other, each handing its columns
// back to the control warp through an mbarrier, so one pair's reduction
// overlaps the other pair's MMA. Every wait is bounded.
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
    int2 *ranges;   // per super-group: first key tile, tile count (written by the prep kernel)
    int m, n;
    int SGR;   // query rows per super-group: 4 warpgroups x 128 / heads
    int n_sg;  // super-groups: ceil(m / SGR)
    int S, QS, q_box;
    uint32_t off_k, off_q, off_w, off_bar, smem_bytes;
};

// ---------------------------------------------------------------- prep kernel

// One CTA per super-group (grid-strided): the tile range [lo, lo + nt) that
// covers the union of its rows' key ranges, and -inf in every entry of its
// rows outside those tiles (the main kernel writes the entries inside).
#ifdef PMQA_PREFILL_PREP
__global__ void __launch_bounds__(256) pmqa_prefill_prep_kernel(const __grid_constant__ PfArgs a)
{
    __shared__ int2 rng;
    const int tid = threadIdx.x, lane = tid & 31;
    // the main kernel may start launching; it waits for this grid before it
    // reads the ranges
    griddep_launch_dependents();
    const float NEG_INF = -__int_as_float(0x7f800000);
    for (int sg = blockIdx.x; sg < a.n_sg; sg += gridDim.x) {
        if (tid < 32) {
            const int r = sg * a.SGR + lane;
            int lo = 0x7FFFFFFF, hi = 0;
            if (lane < a.SGR && r < a.m) {
                const int s = max(__ldg(a.ks + r), 0), e = min(__ldg(a.ke + r), a.n);
                if (e > s) {
                    lo = s;
                    hi = e;
                }
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                lo = min(lo, __shfl_xor_sync(kFullMask, lo, o));
                hi = max(hi, __shfl_xor_sync(kFullMask, hi, o));
            }
            if (lane == 0) {
                int2 R = make_int2(0, 0);
                if (hi > 0) {
                    R.x = lo / kTileTokens;
                    R.y = (hi + kTileTokens - 1) / kTileTokens - R.x;
                }
                a.ranges[sg] = R;
                rng = R;
            }
        }
        __syncthreads();
        const int2 R = rng;
        const long long n = a.n;
        const long long c0 = R.y > 0 ? (long long)R.x * kTileTokens : n;
        const long long c1 = R.y > 0 ? min((long long)(R.x + R.y) * kTileTokens, n) : n;
        const int r1 = min(a.SGR, a.m - sg * a.SGR);
        // [x0, x1) of a row to -inf: scalar stores up to a 16-byte boundary,
        // then 16-byte stores, then the scalar tail
        auto fill = [&](float *row, long long x0, long long x1) {
            const long long mis = (long long)((reinterpret_cast<uintptr_t>(row + x0) >> 2) & 3u);
            const long long head = min(x1 - x0, mis ? 4 - mis : 0);
            if (tid < head)
                row[x0 + tid] = NEG_INF;
            const long long v0 = x0 + head, nv = (x1 - v0) >> 2;
            float4 *rv = reinterpret_cast<float4 *>(row + v0);
            const float4 ninf = make_float4(NEG_INF, NEG_INF, NEG_INF, NEG_INF);
            for (long long x = tid; x < nv; x += blockDim.x)
                rv[x] = ninf;
            for (long long x = v0 + 4 * nv + tid; x < x1; x += blockDim.x)
                row[x] = NEG_INF;
        };
        for (int j = 0; j < r1; ++j) {
            float *row = a.logits + (long long)(sg * a.SGR + j) * n;
            if (c0 > 0)
                fill(row, 0, c0);
            if (c1 < n)
                fill(row, c1, n);
        }
        __syncthreads();  // rng is rewritten for the next super-group
    }
}
#endif  // PMQA_PREFILL_PREP

// ---------------------------------------------------------------- main kernel

// Position (super-group sg, tile m of nt, first tile lo) in a CTA's walk over
// (super-group, tile) items; empty super-groups are skipped.
struct PfPos {
    int sg, m, nt, lo;
    __device__ void load(const PfArgs &a)
    {
        if (sg < a.n_sg) {
            const int2 R = a.ranges[sg];
            lo = R.x;
            nt = R.y;
        } else {
            lo = 0;
            nt = 0;
        }
    }
    __device__ void at(const PfArgs &a, int g, int mm)
    {
        sg = g;
        m = mm;
        load(a);
    }
    __device__ void next(const PfArgs &a)
    {
        if (++m < nt)
            return;
        m = 0;
        do {
            ++sg;
            load(a);
        } while (nt == 0 && sg < a.n_sg);
    }
    __device__ int tile() const { return lo + m; }
};

// Shared-memory mbarriers of the prefill kernel.
//   kfull[S]    a key tile landed in stage s
//   qfull[QS]   query rows + weights of a super-group landed
//   acc[2]      pair p's MMA finished (TMEM columns [256 p, 256 p + 256): warpgroups 2 p, 2 p + 1)
//   bufree[2]   both warpgroups of pair p have read their columns (8 arrivals:
//               one per warp, as soon as its last chunk is in registers)
struct PfBars {
    uint64_t *kfull, *qfull, *acc, *bufree;
    __device__ PfBars(const PfArgs &a, uint8_t *smem)
    {
        kfull = reinterpret_cast<uint64_t *>(smem + a.off_bar);
        qfull = kfull + a.S;
        acc = qfull + a.QS;
        bufree = acc + 2;
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

constexpr int kPfWarps = 4 * kGroups + 1;  // four reducing warpgroups and the control warp
constexpr int kPfThreads = 32 * kPfWarps;
// Register bound of the kernel: 5 of the 17 warps share one SM sub-partition
// (16K registers), so at most 96 registers per thread.
constexpr int kPfBoundThreads = 640;

// Lane 0 of the control warp: every load and every MMA of the CTA's range.
// For item k it issues pair p's MMA (N = 256: the 2 G query rows of
// warpgroups 2 p and 2 p + 1 against the key tile) once both have read their
// columns of item k - 1.
template <int H>
static __device__ void pf_control(const PfArgs &a, uint8_t *smem, CtaCtl &c, int &kloads, int &qloads)
{
    const PfBars B(a, smem);
    const int count = (int)c.count;
    const int S = a.S, QS = a.QS;
    const uint32_t sbase = smem_u32(smem);
    const uint32_t kbase = sbase + a.off_k;
    const uint32_t q_slot_bytes = (uint32_t)(a.SGR * H * kHeadDim);
    const uint32_t idesc = idesc_e4m3_f32(128, 2 * kPassCols);

    // query slots: super-group n of the range in slot n % QS
    PfPos nxt;
    nxt.at(a, c.i0, c.m0);
    int nxt_first = 0;  // CTA item index of nxt's current tile
    auto nxt_valid = [&]() { return nxt.nt > 0 && nxt_first < count; };
    auto nxt_advance = [&]() {
        nxt_first += nxt.nt - nxt.m;
        nxt.m = nxt.nt - 1;
        nxt.next(a);
    };
    for (int u = 0; u < QS; ++u) {
        if (nxt_valid()) {
            pf_load_query(a, smem, B, u, nxt.sg, H);
            ++qloads;
        }
        nxt_advance();
    }
    // key tiles: items 0 .. S - 1 now; item k - 1 + S once item k - 1 is done
    PfPos kp;
    kp.at(a, c.i0, c.m0);
    for (int s = 0; s < S && s < count; ++s) {
        pf_load_k(a, kbase, B, s, kp.tile());
        ++kloads;
        kp.next(a);
    }

    PfPos ip;
    ip.at(a, c.i0, c.m0);
    int islot = 0, prev_slot = 0;
    uint32_t iqphase = 0;
    bool prev_last = false, ok = true, have_q = false;
    // item k's key stage s = k % S and that stage's fill parity, kept as
    // counters (no division on the issuing thread's path)
    int s = 0, s_prev = 0;
    uint32_t s_phase = 0;
    for (int k = 0; k < count; ++k) {
        const bool last = ip.m == ip.nt - 1 || k == count - 1;
        ok = ok && mbar_wait(&B.kfull[s], s_phase, &c.abort);
        if (!have_q) {
            ok = ok && mbar_wait(&B.qfull[islot], iqphase, &c.abort);
            have_q = true;
        }
        const uint64_t ad = sw128_kmajor_desc(kbase + (uint32_t)s * kStageBytes);
        const uint64_t bd0 = sw128_kmajor_desc(sbase + a.off_q + (uint32_t)islot * q_slot_bytes);
#pragma unroll
        for (int p = 0; p < 2; ++p) {
            // both warpgroups of pair p have read their columns of item k - 1
            if (k > 0)
                ok = ok && mbar_wait(&B.bufree[p], (uint32_t)(k - 1) & 1u, &c.abort);
            if (ok) {
                tc_fence_after_sync();
                const uint64_t bd = bd0 + (uint64_t)((uint32_t)(p * 2 * kPassCols * kHeadDim) >> 4);
#pragma unroll
                for (int k4 = 0; k4 < kHeadDim / 32; ++k4)
                    umma_e4m3(c.tmem_base + (uint32_t)(p * 2 * kPassCols), ad + 2u * k4, bd + 2u * k4,
                              idesc, k4 > 0 ? 1u : 0u);
            } else if (!aborted(c)) {
                c.abort = 1;
                atomicOr(a.status, 0x4u);
            }
            // committed even when nothing was issued: the waiters' phases stay in step
            umma_commit(&B.acc[p]);
        }
        if (k > 0 && ok) {
            // every MMA of item k - 1 has completed (the warpgroups read their
            // results): its key stage takes item k - 1 + S, and if it ended a
            // super-group, that super-group's query slot takes the one QS ahead
            if (k - 1 + S < count) {
                pf_load_k(a, kbase, B, s_prev, kp.tile());
                ++kloads;
                kp.next(a);
            }
            if (prev_last) {
                if (nxt_valid()) {
                    pf_load_query(a, smem, B, prev_slot, nxt.sg, H);
                    ++qloads;
                }
                nxt_advance();
            }
        }
        prev_last = last;
        prev_slot = islot;
        s_prev = s;
        if (++s == S) {
            s = 0;
            s_phase ^= 1u;
        }
        if (last) {
            if (++islot == QS) {
                islot = 0;
                iqphase ^= 1u;
            }
            have_q = false;
        }
        ip.next(a);
    }
}

// Warpgroup g, warp quadrant qd: the reductions of every item of the CTA's
// range for query rows g * G .. g * G + G - 1 of each super-group (TMEM
// columns 128 g .. 128 g + 127, thread = key = TMEM lane).
template <int H>
static __device__ void pf_reduce_role(const PfArgs &a, uint8_t *smem, CtaCtl &c, int g, int qd)
{
    constexpr int G = kPassCols / H;
    const PfBars B(a, smem);
    const int lane = threadIdx.x & 31;
    const uint32_t R = (uint32_t)(qd * 32 + lane);
    const int count = (int)c.count;
    const int QS = a.QS, SGR = a.SGR, m = a.m, n = a.n;
    const uint32_t w_slot_bytes = (uint32_t)(SGR * H * 4);
    const uint32_t wbase = smem_u32(smem) + a.off_w + (uint32_t)(g * kPassCols * 4);
    const uint32_t tacc = c.tmem_base + (uint32_t)(g * kPassCols) + ((uint32_t)(qd * 32) << 16);
    float *const logits = a.logits;
    const float NEG_INF = -__int_as_float(0x7f800000);

    PfPos cur;
    cur.at(a, c.i0, c.m0);
    int q_slot = 0;
    uint32_t q_phase = 0;
    bool have_q = false;
    int r0 = 0, nr = 0;  // first row of this warpgroup in the super-group, rows that exist
    int rks[G], rke[G];  // their key ranges
    // key scales are loaded one item ahead
    int t = count > 0 ? cur.tile() * kTileTokens + (int)R : 0;
    float sc = count > 0 && t < n ? __ldg(a.k_scale + t) : 0.0f;
    for (int kk = 0; kk < count; ++kk) {
        PfPos nx = cur;
        nx.next(a);
        const int t_next = kk + 1 < count ? nx.tile() * kTileTokens + (int)R : 0;
        const float sc_next = kk + 1 < count && t_next < n ? __ldg(a.k_scale + t_next) : 0.0f;
        bool ok = true;
        if (!have_q) {
            r0 = cur.sg * SGR + g * G;
            nr = max(0, min(G, m - r0));
#pragma unroll
            for (int j = 0; j < G; ++j) {
                rks[j] = j < nr ? __ldg(a.ks + r0 + j) : 0;
                rke[j] = j < nr ? __ldg(a.ke + r0 + j) : 0;
            }
            ok = mbar_wait(&B.qfull[q_slot], q_phase, &c.abort);
            have_q = true;
        }
        const uint32_t wsl = launder_u32(wbase + (uint32_t)q_slot * w_slot_bytes);
        const uint32_t flip = sc < 0.0f ? 0x80000000u : 0u;
        const float mag = fabsf(sc);
        // every thread waits for the pair's MMA itself
        ok = mbar_wait(&B.acc[g >> 1], (uint32_t)kk & 1u, &c.abort) && ok;
        tc_fence_after_sync();
        // this warp has read its lanes: once every warp of the pair has, the
        // control warp may reuse the columns (one arrival per warp per item,
        // before the outputs; also when the warp had nothing to read)
        auto done = [&]() {
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&B.bufree[g >> 1]);
        };
        if (__all_sync(kFullMask, ok)) {
            const bool all_pos = __all_sync(kFullMask, flip == 0u);
            float *const orow = logits + (long long)r0 * n + t;
            auto out = [&](int j, float v) {
                if (t < n)
                    orow[(long long)j * n] = (t >= rks[j] && t < rke[j]) ? v : NEG_INF;
            };
            if (nr > 0)
                epi_dispatch<H, G>(nr, all_pos, tacc, wsl, flip, mag, 0, out, done);
            else
                done();
        } else {
            done();
            if (lane == 0 && !aborted(c)) {
                c.abort = 1;
                atomicOr(a.status, 0x4u);
            }
        }
        if (cur.m == cur.nt - 1 || kk == count - 1) {
            if (++q_slot == QS) {
                q_slot = 0;
                q_phase ^= 1u;
            }
            have_q = false;
        }
        cur = nx;
        t = t_next;
        sc = sc_next;
    }
}

template <int H>
__global__ void __launch_bounds__(kPfBoundThreads, 1) pmqa_prefill_kernel(const __grid_constant__ PfArgs a)
{
    extern __shared__ uint8_t smem_raw[];
    __shared__ CtaCtl ctl;
    uint8_t *const smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const PfBars B(a, smem);

    if (threadIdx.x == 0) {
        ctl.abort = 0;
        for (int s = 0; s < a.S; ++s)
            mbar_init(&B.kfull[s], 1);
        for (int q = 0; q < a.QS; ++q)
            mbar_init(&B.qfull[q], 1);
        for (int p = 0; p < 2; ++p) {
            mbar_init(&B.acc[p], 1);
            mbar_init(&B.bufree[p], 8);
        }
        mbar_init_fence();
    }
    __syncwarp();
    if (warp == 0)
        tmem_alloc(&ctl.tmem_base, (uint32_t)(kGroups * kPassCols));

    // launched as a dependent of the prep kernel: the ranges are complete
    // and visible after this
    griddep_wait();
    balance_schedule(a.n_sg, [&](int sg) { return (long long)a.ranges[sg].y; }, ctl);
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();

    int kloads = 0, qloads = 0;  // loads issued by the control warp (item i into stage i % S)
    if (warp < 4 * kGroups)
        pf_reduce_role<H>(a, smem, ctl, warp >> 2, warp & 3);
    else if (lane == 0)
        pf_control<H>(a, smem, ctl, kloads, qloads);
    __syncwarp();  // the control warp's lanes meet again before the CTA barrier

    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    if (warp == 4 * kGroups && lane == 0) {
        // loads still in flight after an abort land before the CTA exits (bounded)
        for (int s = 0; s < a.S && s < kloads; ++s) {
            const int uses = (kloads - s + a.S - 1) / a.S;  // loads into stage s
            mbar_wait(&B.kfull[s], (uint32_t)(uses - 1) & 1u, nullptr);
        }
        for (int u = qloads > a.QS ? qloads - a.QS : 0; u < qloads; ++u)
            mbar_wait(&B.qfull[u % a.QS], (uint32_t)(u / a.QS) & 1u, nullptr);
    }
    if (warp == 0)
        tmem_dealloc(ctl.tmem_base, (uint32_t)(kGroups * kPassCols));
}

}  // namespace pmqa
