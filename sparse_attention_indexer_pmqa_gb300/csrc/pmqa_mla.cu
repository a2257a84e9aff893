// pmqa_mla.cu -- sparse MLA decode over the indexer's top-k positions, and its
// C ABI (pmqa_sparse_mla_decode, pmqa_sparse_mla_workspace_bytes).
//
// What is computed. Sources: the page "[Bug] aiter ops triton attention pa",
// section "Downstream impact" (the sparse MLA attention of a decode step
// attends to the positions the indexer's top-k selected); the page
// "[Bug][ROCm]: ROCM_AITER_MLA can select an aiter MLA decode kernel that
// silently returns uncorrelated output" (chat-gpts.plus summary: fp8 Q and fp8
// KV, 16 query heads per latent KV head, 1..4 query rows per request, an LSE
// output for decode context parallelism); the page "[Bugfix][Hardware][AMD] Fix
// last_page_len calculation in AITER MLA decode", section "The Bug" (pages of
// one token). For query row r and head h, over the row's listed positions t:
//   out[r][h] = sum_t softmax_t(sm_scale * q_h . k_t) * v_t,   v_t = k_t[0..511]
//   lse[r][h] = ln sum_t exp(sm_scale * q_h . k_t)
// with q and k_t the fp8 codes times their per-tensor scales.
//
// One persistent CTA per SM walks a contiguous range of the flattened
// (row, 128-position tile) sequence. Per tile:
//   * one warp looks up the 128 listed positions in the block table (two
//     tiles ahead) and moves each latent row (576 bytes) with one 1-D bulk
//     copy; the rows of 8 positions land back to back in a 5120-byte group;
//   * four warps permute each group in place into the operand layout: five
//     1024-byte blocks of 8 rows x 128 bytes in the 128-byte swizzle (four
//     blocks of value columns, one of rotary columns, half used), groups 5120
//     bytes apart, so every swizzle atom stays 1024-byte aligned;
//   * one thread issues S^T = K . Q^T on the tensor cores (M = 128 positions,
//     N = 16 heads, K = 576) into TMEM;
//   * 128 softmax threads (one TMEM lane = one position each) take the tile's
//     per-head maximum, keep a running reference maximum that moves only when
//     it would be exceeded by more than 2^8, form p = 2^(x - m) and write it
//     as two fp8 terms p_hi = e4m3(p), p_lo = e4m3(16 (p - p_hi)) into a
//     K-major operand of 32 rows (16 hi + 16 lo heads);
//   * the thread issues O^T += V^T . P^T (M = 128 value columns per block, four
//     blocks, N = 32, K = 128 positions), reading the SAME tile as an
//     MN-major operand, into four TMEM accumulators of 32 columns.
// With at most as many rows as SMs every row gets the same number of CTAs
// (one keeps it whole); with more, the tiles split evenly over the CTAs. A
// CTA that holds part of a row writes the unnormalised part (O, m, l) to the
// workspace and a second kernel combines the parts.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>

#include "../../include/pmqa.h"
#include "pmqa_mla_ptx.cuh"

namespace pmqa {
namespace mla {

constexpr int kDim = 576;    // latent row: 512 value columns + 64 rotary columns
constexpr int kVDim = 512;   // value columns
constexpr int kHeads = 16;   // query heads per latent KV head
constexpr int kTile = 128;   // listed positions per tile (the first product's M)
constexpr int kChunks = kDim / 16;
constexpr uint32_t kVGroup = 4u * 1024u;          // 8 rows x 4 value blocks of 128 bytes
constexpr uint32_t kVStage = 16u * kVGroup;       // 128 rows of value columns (64 KB)
constexpr uint32_t kRGroup = 512u;                // 8 rows x 64 rotary bytes
constexpr uint32_t kRStage = 16u * kRGroup;       // 128 rows of rotary columns (8 KB)
constexpr int kVStages = 3;                       // value ring
constexpr int kRStages = 2;                       // rotary ring (free once the scores are done)
constexpr uint32_t kPBytes = 32u * 128u;          // 32 rows (hi, lo) x 128 positions
constexpr int kProducers = 128;                   // warps 0-3
constexpr int kSoftmax = 128;                     // warps 4-7
constexpr int kMmaWarp = 8;
constexpr int kThreads = 288;
constexpr int kMaxCtas = 256;                     // workspace parts: 2 per CTA
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kColS = 0;                     // 2 x 16 score columns
constexpr uint32_t kColO = 128;                   // 4 x 32 output columns
constexpr float kLoScale = 16.0f;                 // p_lo holds 16 (p - p_hi)
constexpr float kRescaleSlack = 8.0f;             // p <= 2^8 before the maximum moves
#ifndef PMQA_MLA_MIN_TILES
#define PMQA_MLA_MIN_TILES 2                      // fewest tiles a CTA takes (small problems)
#endif

// Shared memory (the dynamic base is 1024-byte aligned; checked at entry).
constexpr uint32_t kOffV = 0;
constexpr uint32_t kOffR = kOffV + kVStages * kVStage;
constexpr uint32_t kOffQV = kOffR + kRStages * kRStage;      // 16 query heads, value part
constexpr uint32_t kOffQR = kOffQV + 2u * kVGroup;           // 16 query heads, rotary part
constexpr uint32_t kOffP = kOffQR + 2u * kRGroup;
constexpr uint32_t kOffFlags = kOffP + 2u * kPBytes;
constexpr uint32_t kOffRed = kOffFlags + kVStages * kTile;   // [2][4 warps][16] floats
constexpr uint32_t kOffLred = kOffRed + 2u * 4u * 16u * 4u;  // [4 warps][16] floats
constexpr uint32_t kOffBar = kOffLred + 4u * 16u * 4u;
enum {
    kBarFlags = 0,     // [3] tile position flags written: one arrival per producer warp
    kBarReady = 3,     // [3] tile (and query) rows landed: 128 producer cp.async arrivals
    kBarVEmpty = 6,    // [3] value columns read by the output update: MMA commit
    kBarREmpty = 9,    // [2] rotary columns read by the scores: MMA commit
    kBarSFull = 11,    // [2] scores in TMEM: MMA commit
    kBarSFree = 13,    // [2] scores read: one arrival per softmax warp
    kBarPFull = 15,    // [2] P written (and O rescaled): one arrival per softmax warp
    kBarPEmpty = 17,   // [2] P read by the output update: MMA commit
    kBarQEmpty = 19,   // query buffer read: MMA commit after a row's last tile
    kBarDrain = 20,    // MMAs drained before TMEM is freed
    kNumBars = 21
};
constexpr uint32_t kOffMisc = kOffBar + kNumBars * 8u;  // tmem base, abort flag
constexpr uint32_t kSmemBytes = kOffMisc + 16u;
static_assert(kSmemBytes <= 232448, "shared memory budget");
static_assert(kOffR % 1024 == 0 && kOffQV % 1024 == 0 && kOffP % 1024 == 0, "atom alignment");

constexpr uint32_t kIdescQK = idesc_e4m3_f32(128, kHeads);
constexpr uint32_t kIdescPV = idesc_e4m3_f32(128, 2 * kHeads) | kIdescAMnMajor;

// Byte offset of value chunk c (0..31) of row t: groups of 8 rows 4096 bytes
// apart, four 1024-byte blocks of 8 rows x 128 bytes, 128-byte swizzle.
__host__ __device__ constexpr uint32_t v_offset(int t, int c)
{
    return (uint32_t)(t >> 3) * kVGroup + (uint32_t)(c >> 3) * 1024u + (uint32_t)(t & 7) * 128u +
           ((uint32_t)((c & 7) ^ (t & 7)) << 4);
}

// Byte offset of rotary chunk c (0..3) of row t: groups of 8 rows x 64 bytes,
// 64-byte swizzle (chunk c of row r at c ^ (r >> 1)).
__host__ __device__ constexpr uint32_t r_offset(int t, int c)
{
    return (uint32_t)(t >> 3) * kRGroup + (uint32_t)(t & 7) * 64u +
           ((uint32_t)((c ^ ((t & 7) >> 1)) & 3) << 4);
}

struct Args {
    const uint8_t *q;     // [R, 16, 576]
    const uint8_t *kv;    // [num_blocks * P, 576]
    const int32_t *idx;   // [R, topk]
    const int32_t *bt;    // [bs, W]
    float c_log2;         // sm_scale * q_scale * kv_scale * log2(e)
    float kv_scale;
    int next_n, topk, T, P, W;
    int p_shift;          // log2(P) when P is a power of two, else -1
    long long num_blocks;
    long long N;          // R * T tiles
    int G;                // CTAs
    uint16_t *out;        // bf16 [R, 16, 512]
    float *lse;           // [R, 16] or null
    const int32_t *tok_begin;  // [bs] or null: only positions in [tok_begin_i, tok_end_i)
    const int32_t *tok_end;
    uint32_t *status;
    float *ml;            // [2 G][16][2] (m, l) of each part
    float *part;          // [2 G][16][512] unnormalised output of each part
};

__device__ __forceinline__ long long tile_start(const Args &a, int b)
{
    return (long long)b * a.N / a.G;
}

// The CTA whose range holds tile x.
__device__ __forceinline__ int cta_of(const Args &a, long long x)
{
    return (int)(((x + 1) * (long long)a.G - 1) / a.N);
}

// Row r, tile j of the row and request i = r / next_n of the flattened tile x,
// moved on one tile at a time without a division.
struct TileCursor {
    long long r;
    int j;
    long long i;
    int jn;
    __device__ void init(const Args &a, long long x)
    {
        r = x / a.T;
        j = (int)(x - r * a.T);
        i = r / a.next_n;
        jn = (int)(r - i * a.next_n);
    }
    __device__ void next(const Args &a)
    {
        if (++j == a.T) {
            j = 0;
            ++r;
            if (++jn == a.next_n) {
                jn = 0;
                ++i;
            }
        }
    }
};

// Reduce 16 per-lane values over the warp; lane returns the result for head
// (lane >> 1) & 15 (halves exchanged by lane bits 4, 3, 2, 1, then bit 0).
template <bool MAX>
__device__ __forceinline__ float warp_reduce_scatter16(const float (&v)[16], int lane)
{
    constexpr uint32_t kFull = 0xFFFFFFFFu;
    auto op = [](float x, float y) { return MAX ? fmaxf(x, y) : x + y; };
    float a8[8], a4[4], a2[2];
    const bool u16 = (lane & 16) != 0, u8 = (lane & 8) != 0, u4 = (lane & 4) != 0,
               u2 = (lane & 2) != 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float send = u16 ? v[i] : v[i + 8];
        const float keep = u16 ? v[i + 8] : v[i];
        a8[i] = op(keep, __shfl_xor_sync(kFull, send, 16));
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float send = u8 ? a8[i] : a8[i + 4];
        const float keep = u8 ? a8[i + 4] : a8[i];
        a4[i] = op(keep, __shfl_xor_sync(kFull, send, 8));
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const float send = u4 ? a4[i] : a4[i + 2];
        const float keep = u4 ? a4[i + 2] : a4[i];
        a2[i] = op(keep, __shfl_xor_sync(kFull, send, 4));
    }
    const float send = u2 ? a2[0] : a2[1];
    const float keep = u2 ? a2[1] : a2[0];
    const float a1 = op(keep, __shfl_xor_sync(kFull, send, 2));
    return op(a1, __shfl_xor_sync(kFull, a1, 1));
}

// v[i] for a run-time i < 16 without indexing the array (which would move it
// to local memory).
__device__ __forceinline__ float pick16(const float (&v)[16], int i)
{
    float r = v[0];
#pragma unroll
    for (int h = 1; h < 16; ++h)
        r = i == h ? v[h] : r;
    return r;
}

// Byte offset of (row n, position s) in a P buffer: K-major, 128-byte swizzle.
__device__ __forceinline__ uint32_t p_offset(int n, int s)
{
    return (uint32_t)((n >> 3) * 1024 + (n & 7) * 128 + ((((s >> 4) ^ (n & 7)) & 7) << 4) +
                      (s & 15));
}

__device__ __forceinline__ void st_shared_u8(uint32_t addr, uint32_t v)
{
    asm volatile("st.shared.u8 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

__device__ __forceinline__ float ld_cg(const float *p)
{
    return __ldcg(p);
}

__global__ void __launch_bounds__(kThreads, 1) sparse_mla_kernel(const Args a)
{
    extern __shared__ __align__(1024) uint8_t smem[];
    const uint32_t sbase = smem_u32(smem);
    if (sbase & 1023u) {
        // the operand layouts need 1024-byte aligned atoms
        if (threadIdx.x == 0)
            atomicOr(a.status, (uint32_t)PMQA_DEV_INTERNAL);
        return;
    }
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + kOffBar);
    uint32_t *misc = reinterpret_cast<uint32_t *>(smem + kOffMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(misc + 1);
    uint8_t *flags = smem + kOffFlags;
    float *red = reinterpret_cast<float *>(smem + kOffRed);
    float *lred = reinterpret_cast<float *>(smem + kOffLred);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) {
        for (int i = 0; i < kVStages; ++i) {
            mbar_init(&bar[kBarFlags + i], kProducers / 32);
            mbar_init(&bar[kBarReady + i], kProducers);
            mbar_init(&bar[kBarVEmpty + i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bar[kBarREmpty + i], 1);
            mbar_init(&bar[kBarSFull + i], 1);
            mbar_init(&bar[kBarSFree + i], kSoftmax / 32);
            mbar_init(&bar[kBarPFull + i], kSoftmax / 32);
            mbar_init(&bar[kBarPEmpty + i], 1);
        }
        mbar_init(&bar[kBarQEmpty], 1);
        mbar_init(&bar[kBarDrain], 1);
        misc[1] = 0;
        mbar_init_fence();
    }
    if (warp == kMmaWarp)
        tmem_alloc(misc, kTmemCols);
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = misc[0];

    const long long x0 = tile_start(a, blockIdx.x), x1 = tile_start(a, blockIdx.x + 1);
    auto fail = [&]() {
        atomicOr(a.status, (uint32_t)PMQA_DEV_TIMEOUT);
        *abort_flag = 1;
    };

    if (warp < kProducers / 32) {
        // ------------------------------------------------------------ producer
        // Thread tok owns position tok of every tile; warp w copies the rows
        // of positions 32w .. 32w+31, one row per instruction (lane = 16-byte
        // chunk), straight into the operand layout. Lookups run ahead of the
        // copies: the listed position of tile it + 3 and the block table
        // entry of tile it + 2 load while tile it is issued.
        const int pw = warp, tok = tid;
        const long long wp = (long long)a.W * a.P;
        auto load_pos = [&](long long x, const TileCursor &c) -> int {
            if (x >= x1)
                return -1;
            const int e = c.j * kTile + tok;
            return e < a.topk ? __ldg(a.idx + c.r * a.topk + e) : -1;
        };
        auto page_of = [&](int pos) -> int { return a.p_shift >= 0 ? pos >> a.p_shift : pos / a.P; };
        auto load_page = [&](long long x, const TileCursor &c, int pos) -> int {
            if (x >= x1 || pos < 0 || (long long)pos >= wp)
                return -1;
            return __ldg(a.bt + c.i * a.W + page_of(pos));
        };
        // pool row of a looked-up position, -1 for none (bad entries recorded)
        auto row_of = [&](int pos, int page, const TileCursor &c) -> long long {
            if (pos < 0)
                return -1;
            if (a.tok_begin) {
                // a slice of the request's tokens: other positions are not this call's
                if (pos < __ldg(a.tok_begin + c.i) || pos >= __ldg(a.tok_end + c.i))
                    return -1;
            }
            if ((long long)pos >= wp) {
                atomicOr(a.status, (uint32_t)PMQA_DEV_BAD_CONTEXT);
                return -1;
            }
            if (page < 0 || (long long)page >= a.num_blocks) {
                atomicOr(a.status, (uint32_t)PMQA_DEV_BAD_BLOCK_ID);
                return -1;
            }
            return (long long)page * a.P + (pos - page_of(pos) * a.P);
        };
        // cursors at tiles x, x + 1, x + 2 and x + 3
        TileCursor c0, c1, c2, c3;
        c0.init(a, x0);
        c1 = c0;
        c1.next(a);
        c2 = c1;
        c2.next(a);
        c3 = c2;
        c3.next(a);
        int pos0 = load_pos(x0, c0), pos1 = load_pos(x0 + 1, c1), pos2 = load_pos(x0 + 2, c2);
        int page0 = load_page(x0, c0, pos0), page1 = load_page(x0 + 1, c1, pos1);
        int seg = -1, vs = 0;
        uint32_t vph = 0;
        for (long long x = x0; x < x1; ++x) {
            const int it = (int)(x - x0), rs = it & 1;
            const uint32_t rph = (uint32_t)(it >> 1) & 1u;
            const long long r = c0.r;
            const bool first = x == x0 || c0.j == 0;
            if (first)
                ++seg;
            const int pos3 = load_pos(x + 3, c3);
            const int page2 = load_page(x + 2, c2, pos2);
            const long long srow = row_of(pos0, page0, c0);
            pos0 = pos1;
            page0 = page1;
            pos1 = pos2;
            page1 = page2;
            pos2 = pos3;
            if (first) {
                // one query buffer: free once the scores of the previous
                // segment's last tile are done
                if (!__all_sync(0xFFFFFFFFu, mbar_wait(&bar[kBarQEmpty], ((uint32_t)seg & 1u) ^ 1u,
                                                        abort_flag))) {
                    fail();
                    break;
                }
                const uint8_t *qsrc = a.q + r * (long long)(kHeads * kDim);
                for (int c = tid; c < kHeads * kChunks; c += kProducers) {
                    const int h = c / kChunks, ch = c - h * kChunks;
                    const uint32_t dst = ch < 32 ? sbase + kOffQV + v_offset(h, ch)
                                                 : sbase + kOffQR + r_offset(h, ch - 32);
                    cp_async_16(dst, qsrc + h * kDim + ch * 16, 16u);
                }
            }
            // the value slot is free once the output update of tile it - 3 read
            // it, the rotary slot once the scores of tile it - 2 did
            if (!__all_sync(0xFFFFFFFFu,
                            mbar_wait(&bar[kBarVEmpty + vs], vph ^ 1u, abort_flag) &&
                                mbar_wait(&bar[kBarREmpty + rs], rph ^ 1u, abort_flag))) {
                fail();
                break;
            }
            flags[vs * kTile + tok] = srow >= 0 ? 1 : 0;
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&bar[kBarFlags + vs]);
            const uint32_t vdst = sbase + kOffV + (uint32_t)vs * kVStage;
            const uint32_t rdst = sbase + kOffR + (uint32_t)rs * kRStage;
            // value columns: one row per instruction, lane = 16-byte chunk
#pragma unroll 4
            for (int tt = 0; tt < 32; ++tt) {
                const long long sr = __shfl_sync(0xFFFFFFFFu, srow, tt);
                const int t = pw * 32 + tt;
                cp_async_16(vdst + v_offset(t, lane), a.kv + (sr >= 0 ? sr : 0ll) * kDim + 16 * lane,
                            sr >= 0 ? 16u : 0u);
            }
            // rotary columns: 4 chunks per row, 8 rows per instruction
#pragma unroll
            for (int g = 0; g < 4; ++g) {
                const int tt = g * 8 + (lane >> 2), cc = lane & 3;
                const long long sr = __shfl_sync(0xFFFFFFFFu, srow, tt);
                const int t = pw * 32 + tt;
                cp_async_16(rdst + r_offset(t, cc), a.kv + (sr >= 0 ? sr : 0ll) * kDim + kVDim + 16 * cc,
                            sr >= 0 ? 16u : 0u);
            }
            cp_async_arrive_noinc(&bar[kBarReady + vs]);
            if (++vs == kVStages) {
                vs = 0;
                vph ^= 1u;
            }
            c0 = c1;
            c1 = c2;
            c2 = c3;
            c3.next(a);
        }
        cp_async_wait_all();
    } else if (warp >= 4 && warp < 8) {
        // ------------------------------------------------------------ softmax
        // Exits are uniform over the 128 threads: a failed wait only clears
        // `ok`, and the group leaves together at its next barrier (bar.red.and).
        const int s = tid - kProducers, w4 = s >> 5;
        const uint32_t lane_off = (uint32_t)(w4 * 32) << 16;
        const int hsel = (lane >> 1) & 15;
        float m[kHeads], l[kHeads];
        int seg = -1, vs = -1;
        uint32_t vph = 1;
        bool ok = true;
        TileCursor cx;
        cx.init(a, x0);
        for (long long x = x0; x < x1; ++x, cx.next(a)) {
            const int it = (int)(x - x0), stage = it & 1;
            const uint32_t kph = (uint32_t)(it >> 1) & 1u;
            if (++vs == kVStages || it == 0) {
                vs = 0;
                vph ^= 1u;
            }
            const long long r = cx.r;
            const int j = cx.j;
            const bool first = x == x0 || j == 0;
            const bool last = x == x1 - 1 || j == a.T - 1;
            if (first) {
                ++seg;
#pragma unroll
                for (int h = 0; h < kHeads; ++h) {
                    m[h] = -INFINITY;
                    l[h] = 0.0f;
                }
            }
            // scores and flags of the tile; the P buffer free once the output
            // update of tile it - 2 has read it
            ok = ok && mbar_wait(&bar[kBarSFull + stage], kph, abort_flag) &&
                 mbar_wait(&bar[kBarFlags + vs], vph, abort_flag) &&
                 mbar_wait(&bar[kBarPEmpty + stage], kph ^ 1u, abort_flag);
            ok = __all_sync(0xFFFFFFFFu, ok);
            uint32_t sr[16];
            if (ok) {
                tc_fence_after_sync();
                tmem_ld16(tmem + kColS + (uint32_t)stage * kHeads + lane_off, sr);
                tmem_ld_wait();
                reg_fence16(sr);
                tc_fence_before_sync();
            } else {
#pragma unroll
                for (int h = 0; h < kHeads; ++h)
                    sr[h] = 0u;
            }
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&bar[kBarSFree + stage]);
            const bool valid = flags[vs * kTile + s] != 0;
            float xs[kHeads];
#pragma unroll
            for (int h = 0; h < kHeads; ++h)
                xs[h] = valid ? __uint_as_float(sr[h]) * a.c_log2 : -INFINITY;
            // the tile's maximum per head over the 128 positions
            // The running maximum moves only where a position exceeds it by
            // more than the slack (at a segment's first tile, always): one
            // barrier tells whether any thread saw that (or a failed wait);
            // only then is the tile's maximum per head exchanged.
            bool exceed = !ok;
#pragma unroll
            for (int h = 0; h < kHeads; ++h)
                exceed |= xs[h] > m[h] + kRescaleSlack;
            float alpha[kHeads];
#pragma unroll
            for (int h = 0; h < kHeads; ++h)
                alpha[h] = 1.0f;
            bool resc = false;
            if (named_bar_or(1, kSoftmax, exceed)) {
                const float wmax = warp_reduce_scatter16<true>(xs, lane);
                float *rs = red + stage * 64;
                if ((lane & 1) == 0)
                    rs[w4 * 16 + hsel] = wmax;
                if (!named_bar_and(1, kSoftmax, ok)) {
                    fail();
                    break;
                }
#pragma unroll
                for (int h = 0; h < kHeads; ++h) {
                    const float tmax =
                        fmaxf(fmaxf(rs[h], rs[16 + h]), fmaxf(rs[32 + h], rs[48 + h]));
                    if (tmax > m[h] + kRescaleSlack) {
                        if (m[h] != -INFINITY) {
                            alpha[h] = ex2_approx(m[h] - tmax);
                            resc = true;
                        }
                        m[h] = tmax;
                    }
                }
            }
            float p[kHeads];
#pragma unroll
            for (int h = 0; h < kHeads; ++h) {
                p[h] = ex2_approx(xs[h] - (m[h] == -INFINITY ? 0.0f : m[h]));
                l[h] = l[h] * alpha[h] + p[h];
            }
            const uint32_t pb = sbase + kOffP + (uint32_t)stage * kPBytes;
#pragma unroll
            for (int h = 0; h < kHeads; h += 2) {
                const uint32_t hi = f32x2_to_e4m3x2(p[h], p[h + 1]);
                float b0, b1;
                e4m3x2_to_f32x2(hi, b0, b1);
                const uint32_t lo =
                    f32x2_to_e4m3x2((p[h] - b0) * kLoScale, (p[h + 1] - b1) * kLoScale);
                st_shared_u8(pb + p_offset(h, s), hi & 0xFFu);
                st_shared_u8(pb + p_offset(h + 1, s), hi >> 8);
                st_shared_u8(pb + p_offset(kHeads + h, s), lo & 0xFFu);
                st_shared_u8(pb + p_offset(kHeads + h + 1, s), lo >> 8);
            }
            if (resc && !first) {
                // O holds the segment's earlier tiles: wait for the product of
                // tile it - 1, then scale every column by its head's alpha
                ok = ok && mbar_wait(&bar[kBarPEmpty + (stage ^ 1)], (uint32_t)((it - 1) >> 1) & 1u,
                                     abort_flag);
                ok = __all_sync(0xFFFFFFFFu, ok);
                if (ok) {
                    tc_fence_after_sync();
#pragma unroll 1
                    for (int kb = 0; kb < 4; ++kb) {
                        uint32_t o[32];
                        const uint32_t ta = tmem + kColO + (uint32_t)kb * 32u + lane_off;
                        tmem_ld32(ta, o);
                        tmem_ld_wait();
                        reg_fence16(o);
                        reg_fence16(o + 16);
#pragma unroll
                        for (int c = 0; c < 32; ++c)
                            o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha[c & 15]);
                        tmem_st32(ta, o);
                    }
                    tmem_st_wait();
                }
            }
            fence_proxy_async_smem();
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&bar[kBarPFull + stage]);
            if (!last)
                continue;

            // ---------------------------------------------- segment epilogue
            ok = ok && mbar_wait(&bar[kBarPEmpty + stage], kph, abort_flag);
            ok = __all_sync(0xFFFFFFFFu, ok);
            const float wl = warp_reduce_scatter16<false>(l, lane);
            if ((lane & 1) == 0)
                lred[w4 * 16 + hsel] = wl;
            if (!named_bar_and(1, kSoftmax, ok)) {
                fail();
                break;
            }
            tc_fence_after_sync();
            float L[kHeads];
#pragma unroll
            for (int h = 0; h < kHeads; ++h)
                L[h] = (lred[h] + lred[16 + h]) + (lred[32 + h] + lred[48 + h]);
            const long long row0 = r * a.T;
            const int bfirst = cta_of(a, row0);
            const int nseg = cta_of(a, row0 + a.T - 1) - bfirst + 1;
            const float ln2 = 0.69314718055994531f;
            if (nseg == 1) {
#pragma unroll 1
                for (int kb = 0; kb < 4; ++kb) {
                    uint32_t o[32];
                    tmem_ld32(tmem + kColO + (uint32_t)kb * 32u + lane_off, o);
                    tmem_ld_wait();
                    reg_fence16(o);
                    reg_fence16(o + 16);
#pragma unroll
                    for (int h = 0; h < kHeads; ++h) {
                        const float v = __uint_as_float(o[h]) +
                                        __uint_as_float(o[kHeads + h]) * (1.0f / kLoScale);
                        const float y = L[h] > 0.0f ? v * (a.kv_scale / L[h]) : 0.0f;
                        a.out[(r * kHeads + h) * kVDim + kb * 128 + s] =
                            __bfloat16_as_ushort(__float2bfloat16_rn(y));
                    }
                }
                if (a.lse && s < kHeads) {
                    const float Ls = pick16(L, s), ms = pick16(m, s);
                    a.lse[r * kHeads + s] = Ls > 0.0f ? (ms + log2f(Ls)) * ln2 : -INFINITY;
                }
            } else {
                const int slot = 2 * (int)blockIdx.x + (seg == 0 ? 0 : 1);
                float *pp = a.part + (long long)slot * kHeads * kVDim;
#pragma unroll 1
                for (int kb = 0; kb < 4; ++kb) {
                    uint32_t o[32];
                    tmem_ld32(tmem + kColO + (uint32_t)kb * 32u + lane_off, o);
                    tmem_ld_wait();
                    reg_fence16(o);
                    reg_fence16(o + 16);
#pragma unroll
                    for (int h = 0; h < kHeads; ++h)
                        __stcg(pp + h * kVDim + kb * 128 + s,
                               __uint_as_float(o[h]) +
                                   __uint_as_float(o[kHeads + h]) * (1.0f / kLoScale));
                }
                if (s < kHeads) {
                    __stcg(a.ml + (slot * kHeads + s) * 2, pick16(m, s));
                    __stcg(a.ml + (slot * kHeads + s) * 2 + 1, pick16(L, s));
                }
                // combined by the second kernel
            }
        }
    } else if (warp == kMmaWarp && lane == 0) {
        // ------------------------------------------------------------ MMA issue
        // Two streams of products, each issued as soon as its inputs are
        // ready (polled without suspending): the scores of tile nq (its rows
        // in operand layout, its score buffer read, the row's query landed)
        // and the output update of tile np (its P written). Issuing the
        // update without waiting for the next tile frees a staging slot as
        // early as possible.
        const int n = (int)(x1 - x0);
        int nq = 0, np = 0, seg = -1, idle = 0;
        TileCursor cq, cp;  // tiles x0 + nq and x0 + np
        cq.init(a, x0);
        cp = cq;
        int qv = 0, pv = 0;              // value slots of tiles nq and np
        uint32_t qvph = 0;
        uint64_t idle_since = 0;
        bool ok = true;
        while (np < n) {
            bool prog = false;
            // the output update first: it frees a staging slot
            if (np < nq) {
                const int sb = np & 1;
                if (mbar_test(&bar[kBarPFull + sb], (uint32_t)(np >> 1) & 1u)) {
                    const long long x = x0 + np;
                    const bool pfirst = x == x0 || cp.j == 0;
                    tc_fence_after_sync();
                    const uint32_t vb = sbase + kOffV + (uint32_t)pv * kVStage;
                    const uint32_t pb = sbase + kOffP + (uint32_t)sb * kPBytes;
#pragma unroll
                    for (int kb = 0; kb < 4; ++kb)
#pragma unroll
                        for (int ks = 0; ks < 4; ++ks)
                            umma_e4m3(tmem + kColO + (uint32_t)kb * 32u,
                                      sw128_mnmajor_desc(vb + (uint32_t)kb * 1024u + (uint32_t)ks * 4u * kVGroup,
                                                         1024u, kVGroup),
                                      sw128_kmajor_desc(pb + (uint32_t)ks * 32u), kIdescPV,
                                      (pfirst && ks == 0) ? 0u : 1u);
                    umma_commit(&bar[kBarVEmpty + pv]);
                    umma_commit(&bar[kBarPEmpty + sb]);
                    if (++pv == kVStages)
                        pv = 0;
                    ++np;
                    cp.next(a);
                    prog = true;
                }
            }
            if (nq < n) {
                const int sb = nq & 1;
                const uint32_t ph = (uint32_t)(nq >> 1) & 1u;
                if (mbar_test(&bar[kBarReady + qv], qvph) && mbar_test(&bar[kBarSFree + sb], ph ^ 1u)) {
                    const long long x = x0 + nq;
                    const int j = cq.j;
                    if (x == x0 || j == 0)
                        ++seg;
                    fence_proxy_async_smem();  // cp.async writes -> tensor-core reads
                    tc_fence_after_sync();
                    const uint32_t vb = sbase + kOffV + (uint32_t)qv * kVStage;
                    const uint32_t rb = sbase + kOffR + (uint32_t)sb * kRStage;
                    const uint32_t qvb = sbase + kOffQV, qrb = sbase + kOffQR;
                    const uint32_t dS = tmem + kColS + (uint32_t)sb * kHeads;
#pragma unroll
                    for (int kb = 0; kb < 4; ++kb)
#pragma unroll
                        for (int ks = 0; ks < 4; ++ks)
                            umma_e4m3(dS, sw128_kmajor_desc_sbo(vb + (uint32_t)kb * 1024u + (uint32_t)ks * 32u, kVGroup),
                                      sw128_kmajor_desc_sbo(qvb + (uint32_t)kb * 1024u + (uint32_t)ks * 32u, kVGroup),
                                      kIdescQK, (kb | ks) != 0 ? 1u : 0u);
#pragma unroll
                    for (int ks = 0; ks < 2; ++ks)
                        umma_e4m3(dS, sw64_kmajor_desc(rb + (uint32_t)ks * 32u, kRGroup),
                                  sw64_kmajor_desc(qrb + (uint32_t)ks * 32u, kRGroup), kIdescQK, 1u);
                    umma_commit(&bar[kBarSFull + sb]);
                    umma_commit(&bar[kBarREmpty + sb]);
                    if (x == x1 - 1 || j == a.T - 1)
                        umma_commit(&bar[kBarQEmpty]);
                    if (++qv == kVStages) {
                        qv = 0;
                        qvph ^= 1u;
                    }
                    ++nq;
                    cq.next(a);
                    prog = true;
                }
            }
            if (prog) {
                idle = 0;
                idle_since = 0;
                continue;
            }
            // nothing ready: every 64 empty polls, check the abort flag and
            // how long nothing has been ready
            if (++idle < 64)
                continue;
            idle = 0;
            const uint64_t now = global_timer_ns();
            if (idle_since == 0) {
                idle_since = now;
            } else if (*abort_flag || now - idle_since > kWaitLimitNs) {
                ok = false;
                break;
            }
        }
        if (!ok)
            fail();
        umma_commit(&bar[kBarDrain]);
        if (!mbar_wait(&bar[kBarDrain], 0u, nullptr))
            atomicOr(a.status, (uint32_t)PMQA_DEV_TIMEOUT);
    }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// The parts of every row split over several CTAs, combined: block (r, y)
// takes heads HB y .. HB y + HB - 1 of row r (HB = 16 for many rows, 1 for
// few, so that there are enough blocks), thread d value column d. Rows held by
// a single CTA were written by the first kernel. Launched as a programmatic
// dependent of the first kernel: it waits for that grid's results. The parts'
// (m, l) load in parallel over (part, head), HB threads turn them into weights
// in shared memory, and each thread then has HB x parts independent output
// loads in flight.
template <int HB>
__global__ void __launch_bounds__(kVDim) sparse_mla_combine_kernel(const Args a)
{
    // a row's parts come from distinct CTAs: at most kMaxCtas of them
    __shared__ int s_slot[kMaxCtas];
    __shared__ float s_m[kMaxCtas][HB];  // m of (part, head), then its weight
    __shared__ float s_l[kMaxCtas][HB];
    __shared__ float s_M[HB], s_L[HB];
    griddep_wait();
    const long long r = blockIdx.x;
    const int h0 = (int)blockIdx.y * HB;
    const long long row0 = r * a.T;
    const int bfirst = cta_of(a, row0);
    const int nseg = cta_of(a, row0 + a.T - 1) - bfirst + 1;
    if (nseg == 1)
        return;
    const int d = threadIdx.x;
    // part q of the row is slot 2 b + (the row starts inside CTA b's range ? 0 : 1)
    for (int q = d; q < nseg; q += kVDim) {
        const int bb = bfirst + q;
        s_slot[q] = 2 * bb + (tile_start(a, bb) >= row0 ? 0 : 1);
    }
    __syncthreads();
    for (int t = d; t < nseg * HB; t += kVDim) {
        const int q = t / HB, h = t - q * HB;
        s_m[q][h] = a.ml[(s_slot[q] * kHeads + h0 + h) * 2];
        s_l[q][h] = a.ml[(s_slot[q] * kHeads + h0 + h) * 2 + 1];
    }
    __syncthreads();
    if (d < HB) {
        float M = -INFINITY;
        for (int q = 0; q < nseg; ++q)
            M = fmaxf(M, s_m[q][d]);
        float L = 0.0f;
        for (int q = 0; q < nseg; ++q) {
            const float w = s_m[q][d] == -INFINITY ? 0.0f : ex2_approx(s_m[q][d] - M);
            s_m[q][d] = w;
            L += w * s_l[q][d];
        }
        s_M[d] = M;
        s_L[d] = L;
    }
    __syncthreads();
    float acc[HB];
#pragma unroll
    for (int h = 0; h < HB; ++h)
        acc[h] = 0.0f;
#pragma unroll 2
    for (int q = 0; q < nseg; ++q) {
        const float *pp = a.part + ((long long)s_slot[q] * kHeads + h0) * kVDim + d;
#pragma unroll
        for (int h = 0; h < HB; ++h)
            acc[h] += s_m[q][h] * pp[h * kVDim];
    }
#pragma unroll
    for (int h = 0; h < HB; ++h) {
        const float L = s_L[h];
        const float y = L > 0.0f ? acc[h] * (a.kv_scale / L) : 0.0f;
        a.out[(r * kHeads + h0 + h) * kVDim + d] = __bfloat16_as_ushort(__float2bfloat16_rn(y));
    }
    if (a.lse && d < HB)
        a.lse[r * kHeads + h0 + d] =
            s_L[d] > 0.0f ? (s_M[d] + log2f(s_L[d])) * 0.69314718055994531f : -INFINITY;
}

// Workspace: status word | (m, l) of each part | the parts' unnormalised
// outputs.
struct WsLayout {
    size_t ml, part, total;
};

bool ws_layout(long long rows, WsLayout *L)
{
    if (rows < 0)
        return false;
    auto up = [](size_t v) { return (v + 255) / 256 * 256; };
    L->ml = 256;
    L->part = L->ml + up((size_t)2 * kMaxCtas * kHeads * 2 * 4);
    L->total = L->part + (size_t)2 * kMaxCtas * kHeads * kVDim * 4;
    return true;
}

}  // namespace mla
}  // namespace pmqa

using namespace pmqa::mla;

extern "C" size_t pmqa_sparse_mla_workspace_bytes(int32_t rows)
{
    WsLayout L;
    if (!ws_layout(rows, &L))
        return 0;
    return L.total;
}

static int sparse_mla_call(const pmqa_mla_problem *p, const int32_t *tok_begin,
                           const int32_t *tok_end, void *out, float *lse, void *ws,
                           size_t ws_bytes, pmqa_stream_t stream)
{
    auto aligned = [](const void *ptr, uintptr_t al) {
        return (reinterpret_cast<uintptr_t>(ptr) % al) == 0;
    };
    if (!p || p->bs < 0 || p->next_n < 1 || p->topk < 0 || p->block_size < 1 ||
        p->max_blocks_per_seq < 1 || p->num_blocks < 1 || p->heads < 1 || p->head_dim < 1 ||
        p->v_head_dim < 1)
        return PMQA_ERR_INVALID_ARG;
    if (p->heads != kHeads || p->head_dim != kDim || p->v_head_dim != kVDim)
        return PMQA_ERR_UNSUPPORTED;
    if (!(std::isfinite(p->q_scale) && std::isfinite(p->kv_scale) && std::isfinite(p->sm_scale)))
        return PMQA_ERR_INVALID_ARG;
    const long long rows = (long long)p->bs * p->next_n;
    WsLayout L;
    if (!ws_layout(rows, &L))
        return PMQA_ERR_INVALID_ARG;
    if (!ws || !aligned(ws, 256))
        return PMQA_ERR_INVALID_ARG;
    if (ws_bytes < L.total)
        return PMQA_ERR_WORKSPACE;
    if (rows == 0)
        return PMQA_OK;
    if (!p->q || !p->kv_cache || !p->indices || !p->block_tables || !out)
        return PMQA_ERR_INVALID_ARG;
    if (!aligned(p->q, 16) || !aligned(p->kv_cache, 16) || !aligned(p->indices, 4) ||
        !aligned(p->block_tables, 4) || !aligned(out, 4) || (lse && !aligned(lse, 4)))
        return PMQA_ERR_INVALID_ARG;
    if ((tok_begin != nullptr) != (tok_end != nullptr) ||
        (tok_begin && (!aligned(tok_begin, 4) || !aligned(tok_end, 4))))
        return PMQA_ERR_INVALID_ARG;
    const long long T = std::max<long long>(1, (p->topk + kTile - 1) / kTile);
    if (rows * T > (1ll << 40))
        return PMQA_ERR_UNSUPPORTED;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return PMQA_ERR_CUDA;
    Args a{};
    a.q = static_cast<const uint8_t *>(p->q);
    a.kv = static_cast<const uint8_t *>(p->kv_cache);
    a.idx = p->indices;
    a.bt = p->block_tables;
    a.c_log2 = (float)((double)p->sm_scale * (double)p->q_scale * (double)p->kv_scale *
                       1.4426950408889634);
    a.kv_scale = p->kv_scale;
    a.next_n = p->next_n;
    a.topk = p->topk;
    a.T = (int)T;
    a.P = p->block_size;
    a.p_shift = (a.P & (a.P - 1)) == 0 ? __builtin_ctz((unsigned)a.P) : -1;
    a.W = p->max_blocks_per_seq;
    a.num_blocks = p->num_blocks;
    a.N = rows * T;
    const int ctas = std::min(sms, kMaxCtas);
    if (rows <= ctas) {
        // the same number of CTAs for every row, so CTA ranges start at row
        // starts: rows * per CTAs, per = 1 keeps every row whole (no combine)
        const long long per = std::max<long long>(
            1, std::min<long long>(T / PMQA_MLA_MIN_TILES, ctas / rows));
        a.G = (int)(rows * per);
    } else {
        const long long want = (a.N + PMQA_MLA_MIN_TILES - 1) / PMQA_MLA_MIN_TILES;
        a.G = (int)std::min<long long>(want, ctas);
    }
    uint8_t *wsb = static_cast<uint8_t *>(ws);
    a.tok_begin = tok_begin;
    a.tok_end = tok_end;
    a.out = static_cast<uint16_t *>(out);
    a.lse = lse;
    a.status = reinterpret_cast<uint32_t *>(wsb);
    a.ml = reinterpret_cast<float *>(wsb + L.ml);
    a.part = reinterpret_cast<float *>(wsb + L.part);
    if (cudaFuncSetAttribute(sparse_mla_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kSmemBytes) != cudaSuccess)
        return PMQA_ERR_CUDA;
    const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    sparse_mla_kernel<<<a.G, kThreads, kSmemBytes, st>>>(a);
    if (cudaGetLastError() != cudaSuccess)
        return PMQA_ERR_CUDA;
    if (a.T > 1 && a.G != rows) {
        // rows may be split over CTAs: the combining kernel, its launch
        // overlapping the first kernel's end (rows held whole return at once)
        cudaLaunchConfig_t cfg = {};
        cfg.stream = st;
        cfg.blockDim = dim3(kVDim);
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        // a block per (row, head) for few rows (enough blocks), per row for many
        const bool few = rows <= 32;
        cfg.gridDim = dim3((unsigned)rows, few ? kHeads : 1);
        const cudaError_t e = few ? cudaLaunchKernelEx(&cfg, sparse_mla_combine_kernel<1>, a)
                                  : cudaLaunchKernelEx(&cfg, sparse_mla_combine_kernel<kHeads>, a);
        if (e != cudaSuccess)
            return PMQA_ERR_CUDA;
    }
    return cudaGetLastError() == cudaSuccess ? PMQA_OK : PMQA_ERR_CUDA;
}

namespace pmqa {
namespace mla {

// Merge of G partial decodes of the same rows (one per slice of the listed
// positions): out = sum_g w_g out_g / sum_g w_g and lse = M + ln sum_g w_g with
// w_g = exp(lse_g - M), M = max_g lse_g; a part with lse = -inf has weight 0.
// Block (r, h): thread d value column d.
__global__ void __launch_bounds__(kVDim) sparse_mla_merge_kernel(const uint16_t *outs,
                                                                 const float *lses, int G,
                                                                 long long rows, uint16_t *out,
                                                                 float *lse)
{
    const long long r = blockIdx.x;
    const int h = (int)blockIdx.y, d = (int)threadIdx.x;
    const long long rh = r * kHeads + h;
    const long long part_stride = rows * kHeads;  // (row, head) pairs per part
    float M = -INFINITY;
    for (int g = 0; g < G; ++g)
        M = fmaxf(M, __ldg(lses + g * part_stride + rh));
    float L = 0.0f, acc = 0.0f;
    for (int g = 0; g < G; ++g) {
        const float lg = __ldg(lses + g * part_stride + rh);
        if (lg == -INFINITY)
            continue;
        const float w = expf(lg - M);
        L += w;
        const uint16_t b = __ldg(outs + (g * part_stride + rh) * kVDim + d);
        acc += w * __bfloat162float(__ushort_as_bfloat16(b));
    }
    const float y = L > 0.0f ? acc / L : 0.0f;
    out[rh * kVDim + d] = __bfloat16_as_ushort(__float2bfloat16_rn(y));
    if (lse && d == 0)
        lse[rh] = L > 0.0f ? M + logf(L) : -INFINITY;
}

}  // namespace mla
}  // namespace pmqa

extern "C" int pmqa_sparse_mla_decode(const pmqa_mla_problem *p, void *out, float *lse, void *ws,
                                      size_t ws_bytes, pmqa_stream_t stream)
{
    return sparse_mla_call(p, nullptr, nullptr, out, lse, ws, ws_bytes, stream);
}

extern "C" int pmqa_sparse_mla_decode_range(const pmqa_mla_problem *p,
                                            const int32_t *token_begin,
                                            const int32_t *token_end, void *out, float *lse,
                                            void *ws, size_t ws_bytes, pmqa_stream_t stream)
{
    if (!token_begin || !token_end)
        return PMQA_ERR_INVALID_ARG;
    return sparse_mla_call(p, token_begin, token_end, out, lse, ws, ws_bytes, stream);
}

extern "C" int pmqa_sparse_mla_merge(const void *outs, const float *lses, int32_t parts,
                                     int32_t rows, int32_t heads, void *out, float *lse,
                                     pmqa_stream_t stream)
{
    auto aligned = [](const void *ptr, uintptr_t al) {
        return (reinterpret_cast<uintptr_t>(ptr) % al) == 0;
    };
    if (parts < 1 || rows < 0 || heads < 1)
        return PMQA_ERR_INVALID_ARG;
    if (heads != kHeads)
        return PMQA_ERR_UNSUPPORTED;
    if (rows == 0)
        return PMQA_OK;
    if (!outs || !lses || !out || !aligned(outs, 4) || !aligned(lses, 4) || !aligned(out, 4) ||
        (lse && !aligned(lse, 4)))
        return PMQA_ERR_INVALID_ARG;
    if ((long long)rows > 0x7FFFFFFFll)
        return PMQA_ERR_UNSUPPORTED;
    sparse_mla_merge_kernel<<<dim3((unsigned)rows, kHeads), kVDim, 0,
                              reinterpret_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint16_t *>(outs), lses, parts, rows, static_cast<uint16_t *>(out), lse);
    return cudaGetLastError() == cudaSuccess ? PMQA_OK : PMQA_ERR_CUDA;
}
