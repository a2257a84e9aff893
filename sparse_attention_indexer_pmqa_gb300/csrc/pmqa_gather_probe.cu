// pmqa_gather_probe.cu -- how fast this GPU reads a list of random
// fixed-pitch rows, by three ways of issuing the reads. A measurement aid that
// stands beside the decode path (it computes nothing of the method): the
// indexer's KV pass reads random 132-byte token rows (the row layout of the
// "[Bug] aiter ops triton attention pa" page, Minimal reproduction) and the
// sparse MLA decode random 576-byte latent rows, and the read rate this probe
// reaches on the same rows is the ceiling those kernels' gathers work under.
//
// Every row is read as its 16-byte aligned window (144 bytes for a pitch of
// 132, the row itself for 576), as the decode kernels read them:
//   method 0  16-byte loads into registers, folded into a running XOR;
//   method 1  16-byte cp.async into a per-warp ring of shared-memory slots;
//   method 2  one bulk copy (cp.async.bulk) per row window into the same ring,
//             completion counted on an mbarrier per slot.
// Persistent grids, one CTA per SM. out[0] collects status bits (a skipped row,
// a wait that ran out), out[1] the XOR of every 32-bit word read (method 0) or
// of each window's first word (methods 1 and 2), so a host can check that the
// right bytes were read.

#include <cuda_runtime.h>

#include <cstdint>

#include "pmqa.h"
#include "pmqa_mla_ptx.cuh"
#include "pmqa_ptx.cuh"

using namespace pmqa;

namespace {

constexpr int kLdThreads = 768;
constexpr int kAsyncWarps = 4;
constexpr unsigned long long kNone = ~0ull;

struct ProbeArgs {
    const uint8_t *pool;
    unsigned long long pool_bytes;
    const int32_t *rows;
    long long n;
    int pitch;
    uint32_t *out;
};

// Start of row r's 16-byte aligned window of `win` bytes, or kNone for a
// negative row or a window that would pass the end of the pool.
__device__ __forceinline__ unsigned long long window_start(const ProbeArgs &a, int r, int win)
{
    if (r < 0)
        return kNone;
    const unsigned long long s = ((unsigned long long)r * (unsigned)a.pitch) & ~15ull;
    return s + (unsigned)win <= a.pool_bytes ? s : kNone;
}

__device__ __forceinline__ uint4 ldg_stream(const void *p)
{
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ void sts32(uint32_t addr, uint32_t v)
{
    asm volatile("st.shared.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

__device__ __forceinline__ void finish(const ProbeArgs &a, uint32_t acc, uint32_t status)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        acc ^= __shfl_xor_sync(0xFFFFFFFFu, acc, o);
        status |= __shfl_xor_sync(0xFFFFFFFFu, status, o);
    }
    if ((threadIdx.x & 31) == 0) {
        atomicXor(a.out + 1, acc);
        if (status)
            atomicOr(a.out, status);
    }
}

// A warp takes 32 rows at a time; lane l reads chunks l, l + 32, ... of the
// batch's 32 * C chunks (chunk e is chunk e % C of row e / C), nine loads in
// flight per thread.
template <int C>
__global__ void __launch_bounds__(kLdThreads, 1) gather_probe_ld(ProbeArgs a)
{
    static_assert(C % 9 == 0, "chunks per window in steps of nine");
    const int lane = threadIdx.x & 31;
    const long long gw = ((long long)blockIdx.x * kLdThreads + threadIdx.x) >> 5;
    const long long nw = (long long)gridDim.x * (kLdThreads / 32);
    const long long batches = (a.n + 31) / 32;
    uint32_t acc = 0, status = 0;
    for (long long b = gw; b < batches; b += nw) {
        const long long i = b * 32 + lane;
        unsigned long long s = kNone;
        if (i < a.n) {
            s = window_start(a, __ldg(a.rows + i), C * 16);
            if (s == kNone)
                status |= PMQA_DEV_BAD_CONTEXT;
        }
#pragma unroll 1
        for (int k0 = 0; k0 < C; k0 += 9) {
            uint4 v[9];
#pragma unroll
            for (int u = 0; u < 9; ++u) {
                const int e = lane + 32 * (k0 + u), j = e / C, c = e - j * C;
                const unsigned long long sj = __shfl_sync(0xFFFFFFFFu, s, j);
                v[u] = sj != kNone ? ldg_stream(a.pool + sj + 16 * c) : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int u = 0; u < 9; ++u)
                acc ^= v[u].x ^ v[u].y ^ v[u].z ^ v[u].w;
        }
    }
    finish(a, acc, status);
}

// cp.async: warp w owns S slots of 32 windows; batch k of the warp goes to
// slot k % S once batch k - S has landed (S - 1 batches stay in flight while
// the next is issued). Chunk e of a batch lands at slot + 16 e, so window j
// starts at slot + j * 16 C.
template <int C, int S>
__global__ void __launch_bounds__(kAsyncWarps * 32, 1) gather_probe_cp_async(ProbeArgs a)
{
    extern __shared__ __align__(1024) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    constexpr uint32_t kSlot = 32u * C * 16u;
    const uint32_t base = smem_u32(smem) + (uint32_t)warp * S * kSlot;
    const long long gw = (long long)blockIdx.x * kAsyncWarps + warp;
    const long long nw = (long long)gridDim.x * kAsyncWarps;
    const long long batches = (a.n + 31) / 32;
    uint32_t acc = 0, status = 0;
    long long k = 0;
    for (long long b = gw; b < batches; b += nw, ++k) {
        const uint32_t slot = base + (uint32_t)(k % S) * kSlot;
        if (k >= S) {
            cp_async_wait_group<S - 1>();
            __syncwarp();
            acc ^= lds32(slot + (uint32_t)lane * C * 16u);
            __syncwarp();
        }
        const long long i = b * 32 + lane;
        unsigned long long s = kNone;
        if (i < a.n) {
            s = window_start(a, __ldg(a.rows + i), C * 16);
            if (s == kNone)
                status |= PMQA_DEV_BAD_CONTEXT;
        }
#pragma unroll
        for (int u = 0; u < C; ++u) {
            const int e = lane + 32 * u, j = e / C, c = e - j * C;
            const unsigned long long sj = __shfl_sync(0xFFFFFFFFu, s, j);
            // a skipped row is zero-filled, so its first word adds nothing
            cp_async_16(slot + 16u * e, a.pool + (sj != kNone ? sj + 16 * c : 0ull),
                        sj != kNone ? 16u : 0u);
        }
        cp_async_commit();
    }
    cp_async_wait_all();
    __syncwarp();
    for (long long kk = k > S ? k - S : 0; kk < k; ++kk)
        acc ^= lds32(base + (uint32_t)(kk % S) * kSlot + (uint32_t)lane * C * 16u);
    finish(a, acc, status);
}

// Bulk copies: the same ring; lane j copies window j of the batch with one
// cp.async.bulk, and the slot's mbarrier counts the batch's bytes.
template <int C, int S>
__global__ void __launch_bounds__(kAsyncWarps * 32, 1) gather_probe_bulk(ProbeArgs a)
{
    extern __shared__ __align__(1024) uint8_t smem[];
    __shared__ __align__(8) uint64_t bars[kAsyncWarps][S];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    constexpr uint32_t kWin = C * 16u, kSlot = 32u * kWin;
    const uint32_t base = smem_u32(smem) + (uint32_t)warp * S * kSlot;
    if (lane == 0) {
        for (int s = 0; s < S; ++s)
            mbar_init(&bars[warp][s], 1);
        mbar_init_fence();
    }
    __syncwarp();
    const long long gw = (long long)blockIdx.x * kAsyncWarps + warp;
    const long long nw = (long long)gridDim.x * kAsyncWarps;
    const long long batches = (a.n + 31) / 32;
    uint32_t acc = 0, status = 0;
    long long k = 0;
    // reads the first word of this lane's window in slot kk % S once that
    // batch has landed; a wait that runs out is recorded and the word skipped
    auto collect = [&](long long kk) {
        const int sl = (int)(kk % S);
        const uint32_t parity = (uint32_t)(kk / S) & 1u;
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(&bars[warp][sl], parity, nullptr))) {
            status |= PMQA_DEV_TIMEOUT;
            return;
        }
        acc ^= lds32(base + (uint32_t)sl * kSlot + (uint32_t)lane * kWin);
    };
    for (long long b = gw; b < batches; b += nw, ++k) {
        const int sl = (int)(k % S);
        const uint32_t slot = base + (uint32_t)sl * kSlot;
        if (k >= S)
            collect(k - S);
        if (__any_sync(0xFFFFFFFFu, status & PMQA_DEV_TIMEOUT))
            break;
        __syncwarp();
        const long long i = b * 32 + lane;
        unsigned long long s = kNone;
        if (i < a.n) {
            s = window_start(a, __ldg(a.rows + i), (int)kWin);
            if (s == kNone)
                status |= PMQA_DEV_BAD_CONTEXT;
        }
        const uint32_t valid = __ballot_sync(0xFFFFFFFFu, s != kNone);
        if (s == kNone)
            sts32(slot + (uint32_t)lane * kWin, 0u);  // nothing lands here this round
        // the slot's earlier reads and writes come before the copies that refill it
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0)
            mbar_arrive_expect_tx(&bars[warp][sl], (uint32_t)__popc(valid) * kWin);
        __syncwarp();
        if (s != kNone)
            bulk_load(slot + (uint32_t)lane * kWin, a.pool + s, kWin, &bars[warp][sl]);
    }
    // every batch still in flight lands before the CTA leaves (each wait bounded)
    for (long long kk = k > S ? k - S : 0; kk < k; ++kk)
        collect(kk);
    finish(a, acc, status);
}

int sm_count()
{
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return 0;
    return sms;
}

template <int C, int S>
int launch_async(const ProbeArgs &a, int method, int sms, cudaStream_t st)
{
    const size_t smem = (size_t)kAsyncWarps * S * 32 * C * 16;
    if (method == 1) {
        if (cudaFuncSetAttribute(gather_probe_cp_async<C, S>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem) != cudaSuccess)
            return PMQA_ERR_CUDA;
        gather_probe_cp_async<C, S><<<sms, kAsyncWarps * 32, smem, st>>>(a);
    } else {
        if (cudaFuncSetAttribute(gather_probe_bulk<C, S>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem) != cudaSuccess)
            return PMQA_ERR_CUDA;
        gather_probe_bulk<C, S><<<sms, kAsyncWarps * 32, smem, st>>>(a);
    }
    return PMQA_OK;
}

}  // namespace

extern "C" int pmqa_gather_probe(const void *pool, uint64_t pool_bytes, const int32_t *rows,
                                 int64_t n, int32_t row_pitch, int32_t method, uint32_t *out,
                                 pmqa_stream_t stream)
{
    if (n < 0 || method < 0 || method > 2)
        return PMQA_ERR_INVALID_ARG;
    if (row_pitch != 132 && row_pitch != 576)
        return PMQA_ERR_UNSUPPORTED;
    if (n == 0)
        return PMQA_OK;
    if (!pool || !rows || !out || (reinterpret_cast<uintptr_t>(pool) & 15) ||
        (reinterpret_cast<uintptr_t>(rows) & 3) || (reinterpret_cast<uintptr_t>(out) & 3))
        return PMQA_ERR_INVALID_ARG;
    const int sms = sm_count();
    if (sms <= 0)
        return PMQA_ERR_CUDA;
    const ProbeArgs a{static_cast<const uint8_t *>(pool), (unsigned long long)pool_bytes, rows,
                      (long long)n, row_pitch, out};
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    int rc = PMQA_OK;
    if (method == 0) {
        if (row_pitch == 132)
            gather_probe_ld<9><<<sms, kLdThreads, 0, st>>>(a);
        else
            gather_probe_ld<36><<<sms, kLdThreads, 0, st>>>(a);
    } else if (row_pitch == 132) {
        rc = launch_async<9, 8>(a, method, sms, st);     // 144-byte windows: 8 slots of 4.5 KB
    } else {
        rc = launch_async<36, 2>(a, method, sms, st);    // 576-byte rows: 2 slots of 18 KB
    }
    if (rc != PMQA_OK)
        return rc;
    return cudaGetLastError() == cudaSuccess ? PMQA_OK : PMQA_ERR_CUDA;
}
