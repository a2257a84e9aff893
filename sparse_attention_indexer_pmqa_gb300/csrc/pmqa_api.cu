// pmqa_api.cu -- the C ABI of include/pmqa.h: argument checks, workspace and
// shared-memory layout, kernel launches. No allocation, no synchronisation
// (except pmqa_read_device_status), no state kept between calls.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>

#include "../../include/pmqa.h"
#include "pmqa_main.cuh"
#include "pmqa_topk_kernel.cuh"

namespace pmqa {
cudaError_t launch_main_h16(const MainArgs &, bool, int, int, cudaStream_t);
cudaError_t launch_main_h32(const MainArgs &, bool, int, int, cudaStream_t);
cudaError_t launch_main_h64(const MainArgs &, bool, int, int, cudaStream_t);
cudaError_t launch_main_h128(const MainArgs &, bool, int, int, cudaStream_t);
}  // namespace pmqa

using namespace pmqa;

namespace {

constexpr int kVersion = 100;          // 0.1.0
constexpr uint32_t kMaxDynSmem = 232448 - 1024;
constexpr uint32_t kMinMainSmem = 120 * 1024;  // > half an SM: one CTA per SM
constexpr size_t kWsAlign = 256;

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

struct WsLayout {
    size_t arrive, cand_cnt, cand, total;
};

bool ws_layout(long long rows, long long mml, int op, WsLayout *L)
{
    if (rows < 0 || mml < 1)
        return false;
    L->arrive = kWsAlign;
    if (op == PMQA_OP_LOGITS) {
        L->cand_cnt = L->cand = L->total = kWsAlign;
        return true;
    }
    L->cand_cnt = L->arrive + align_up((size_t)rows * 4, kWsAlign);
    L->cand = L->cand_cnt + align_up((size_t)rows * 4, kWsAlign);
    L->total = L->cand + (size_t)rows * (size_t)mml * 8;
    return true;
}

TopkWs ws_view(void *ws, const WsLayout &L, long long mml)
{
    uint8_t *b = static_cast<uint8_t *>(ws);
    TopkWs w;
    w.status = reinterpret_cast<uint32_t *>(b);
    w.arrive = reinterpret_cast<uint32_t *>(b + L.arrive);
    w.cand_cnt = reinterpret_cast<uint32_t *>(b + L.cand_cnt);
    w.cand = reinterpret_cast<uint2 *>(b + L.cand);
    w.row_cap = mml;
    return w;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int sm_count(int *n)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return PMQA_ERR_CUDA;
    if (cudaDeviceGetAttribute(n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return PMQA_ERR_CUDA;
    return PMQA_OK;
}

bool supported_heads(int h) { return h == 16 || h == 32 || h == 64 || h == 128; }

int check_problem(const pmqa_problem *p)
{
    if (!p)
        return PMQA_ERR_INVALID_ARG;
    if (p->bs < 0 || p->next_n < 1 || p->heads < 1 || p->head_dim < 1 || p->block_size < 1 ||
        p->max_blocks_per_seq < 1 || p->max_model_len < 1 || p->num_blocks < 1)
        return PMQA_ERR_INVALID_ARG;
    if (p->head_dim != kHeadDim || !supported_heads(p->heads) || p->next_n > 4)
        return PMQA_ERR_UNSUPPORTED;
    if (p->bs == 0)
        return PMQA_OK;
    if (!p->q || !p->kv_cache || !p->weights || !p->context_lens || !p->block_tables)
        return PMQA_ERR_INVALID_ARG;
    if (!aligned(p->q, 16) || !aligned(p->weights, 16) || !aligned(p->kv_cache, 4) ||
        !aligned(p->context_lens, 4) || !aligned(p->block_tables, 4))
        return PMQA_ERR_INVALID_ARG;
    return PMQA_OK;
}

// Shared-memory and pipeline layout of the main kernel.
bool main_layout(int heads, int nn, bool fused, int k, MainArgs &a)
{
    const int N = heads * nn;
    a.N = N;
    a.E = nn >= 2 ? 2 : 1;
    a.rpw = (nn + a.E - 1) / a.E;
    int cols = 32;
    while (cols < N)
        cols <<= 1;
    if (cols > 512)
        return false;
    a.cols = cols;
    a.NBUF = std::min(8, 512 / cols);
    a.tmem_cols = a.NBUF * cols;
    for (int S = 4; S >= 2; --S) {
        for (int QS = 2; QS >= 1; --QS) {
            uint32_t off = (uint32_t)S * kStageBytes;
            a.off_q = off;
            off += (uint32_t)(QS * N * kHeadDim);
            a.off_w = off;
            off += (uint32_t)(QS * N * 4);
            off = (uint32_t)align_up(off, 16);
            const int RS = S + a.NBUF;
            a.off_scale = off;
            off += (uint32_t)RS * 512u;
            a.off_bar = off;
            off += (uint32_t)(2 * S + 2 * a.NBUF + 2 * QS + RS + 1) * 8u;
            off = (uint32_t)align_up(off, 128);
            a.off_cand = off;
            int cap = 0;
            if (fused) {
                const long fixed = 64 + (long)sizeof(WgScratch);
                const long avail = (long)kMaxDynSmem - 1024 - (long)off - a.E * fixed;
                if (avail <= 0)
                    continue;
                cap = (int)std::min<long>(avail / ((long)a.E * a.rpw * 8), 4096) & ~127;
                if (cap < k + 256)
                    continue;
                off += (uint32_t)(a.E * ((long)a.rpw * cap * 8 + fixed));
            }
            uint32_t total = std::max<uint32_t>(off + 1024, kMinMainSmem);
            if (total > kMaxDynSmem)
                continue;
            a.S = S;
            a.QS = QS;
            a.RS = RS;
            a.cap = cap;
            a.smem_bytes = total;
            return true;
        }
    }
    return false;
}

int run_main(const pmqa_problem *p, bool fused, int k, int32_t *idx, float *vals, float *logits,
             void *ws, size_t ws_bytes, cudaStream_t stream)
{
    int rc = check_problem(p);
    if (rc != PMQA_OK)
        return rc;
    if (fused) {
        if (k < 1 || !idx)
            return PMQA_ERR_INVALID_ARG;
        if (!aligned(idx, 4) || (vals && !aligned(vals, 4)))
            return PMQA_ERR_INVALID_ARG;
    } else if (!logits) {
        return PMQA_ERR_INVALID_ARG;
    }
    if (logits && !aligned(logits, 4))
        return PMQA_ERR_INVALID_ARG;
    const long long rows = (long long)p->bs * p->next_n;
    WsLayout L;
    if (!ws_layout(rows, p->max_model_len, fused ? PMQA_OP_LOGITS_TOPK : PMQA_OP_LOGITS, &L))
        return PMQA_ERR_INVALID_ARG;
    if (!ws || !aligned(ws, kWsAlign))
        return PMQA_ERR_INVALID_ARG;
    if (ws_bytes < L.total)
        return PMQA_ERR_WORKSPACE;
    MainArgs a{};
    if (!main_layout(p->heads, p->next_n, fused, k, a))
        return PMQA_ERR_UNSUPPORTED;
    if (p->bs == 0)
        return PMQA_OK;
    a.q = static_cast<const uint8_t *>(p->q);
    a.kv = static_cast<const uint8_t *>(p->kv_cache);
    a.w = p->weights;
    a.ctx_lens = p->context_lens;
    a.bt = p->block_tables;
    a.num_blocks = p->num_blocks;
    a.bs = p->bs;
    a.nn = p->next_n;
    a.P = p->block_size;
    a.W = p->max_blocks_per_seq;
    a.mml = p->max_model_len;
    a.logits = logits;
    a.k = fused ? k : 0;
    a.out_idx = idx;
    a.out_vals = vals;
    a.ws = ws_view(ws, L, p->max_model_len);
    int sms = 0;
    if ((rc = sm_count(&sms)) != PMQA_OK)
        return rc;
    const int threads = 32 * (kFirstEpiWarp + 4 * a.E);
    cudaError_t e;
    switch (p->heads) {
    case 16: e = launch_main_h16(a, fused, sms, threads, stream); break;
    case 32: e = launch_main_h32(a, fused, sms, threads, stream); break;
    case 64: e = launch_main_h64(a, fused, sms, threads, stream); break;
    default: e = launch_main_h128(a, fused, sms, threads, stream); break;
    }
    return e == cudaSuccess ? PMQA_OK : PMQA_ERR_CUDA;
}

}  // namespace

extern "C" {

size_t pmqa_workspace_bytes(int32_t bs, int32_t next_n, int32_t max_model_len, int32_t k, int op)
{
    (void)k;
    if (bs < 0 || next_n < 1 || max_model_len < 1 || op < PMQA_OP_LOGITS ||
        op > PMQA_OP_LOGITS_TOPK)
        return 0;
    WsLayout L;
    if (!ws_layout((long long)bs * next_n, max_model_len, op, &L))
        return 0;
    return L.total;
}

int pmqa_workspace_init(void *ws, size_t ws_bytes, pmqa_stream_t stream)
{
    if (!ws || ws_bytes < kWsAlign || !aligned(ws, kWsAlign))
        return PMQA_ERR_INVALID_ARG;
    return cudaMemsetAsync(ws, 0, ws_bytes, stream) == cudaSuccess ? PMQA_OK : PMQA_ERR_CUDA;
}

int pmqa_logits(const pmqa_problem *p, float *logits, void *ws, size_t ws_bytes,
                pmqa_stream_t stream)
{
    return run_main(p, false, 0, nullptr, nullptr, logits, ws, ws_bytes, stream);
}

int pmqa_logits_topk(const pmqa_problem *p, int32_t k, int32_t *idx, float *vals, float *logits,
                     void *ws, size_t ws_bytes, pmqa_stream_t stream)
{
    return run_main(p, true, k, idx, vals, logits, ws, ws_bytes, stream);
}

int pmqa_topk(const float *logits, const int32_t *context_lens, int32_t bs, int32_t next_n,
              int32_t max_model_len, int32_t k, int32_t *idx, float *vals, void *ws,
              size_t ws_bytes, pmqa_stream_t stream)
{
    if (bs < 0 || next_n < 1 || max_model_len < 1 || k < 1)
        return PMQA_ERR_INVALID_ARG;
    const long long rows = (long long)bs * next_n;
    WsLayout L;
    if (!ws_layout(rows, max_model_len, PMQA_OP_TOPK, &L))
        return PMQA_ERR_INVALID_ARG;
    if (!ws || !aligned(ws, kWsAlign))
        return PMQA_ERR_INVALID_ARG;
    if (ws_bytes < L.total)
        return PMQA_ERR_WORKSPACE;
    if (bs == 0)
        return PMQA_OK;
    if (!logits || !context_lens || !idx || !aligned(logits, 4) || !aligned(context_lens, 4) ||
        !aligned(idx, 4) || (vals && !aligned(vals, 4)))
        return PMQA_ERR_INVALID_ARG;
    const long long cap = std::max<long long>(4096, (long long)align_up((size_t)k + 1024, 128));
    const size_t smem = sizeof(WgScratch) + 16 + (size_t)cap * 8;
    if (smem > kMaxDynSmem)
        return PMQA_ERR_UNSUPPORTED;
    TopkArgs a{};
    a.logits = logits;
    a.ctx_lens = context_lens;
    a.bs = bs;
    a.nn = next_n;
    a.mml = max_model_len;
    a.k = k;
    a.idx = idx;
    a.vals = vals;
    a.ws = ws_view(ws, L, max_model_len);
    a.cap = (int)cap;
    int sms = 0;
    int rc = sm_count(&sms);
    if (rc != PMQA_OK)
        return rc;
    if (cudaFuncSetAttribute(pmqa_topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem) != cudaSuccess)
        return PMQA_ERR_CUDA;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, pmqa_topk_kernel, 128, smem) !=
            cudaSuccess ||
        per_sm < 1)
        return PMQA_ERR_CUDA;
    pmqa_topk_kernel<<<sms * std::min(per_sm, 4), 128, smem, stream>>>(a);
    return cudaGetLastError() == cudaSuccess ? PMQA_OK : PMQA_ERR_CUDA;
}

int pmqa_read_device_status(void *ws, pmqa_stream_t stream)
{
    if (!ws || !aligned(ws, kWsAlign))
        return PMQA_ERR_INVALID_ARG;
    uint32_t host = 0;
    if (cudaMemcpyAsync(&host, ws, sizeof host, cudaMemcpyDeviceToHost, stream) != cudaSuccess ||
        cudaMemsetAsync(ws, 0, sizeof host, stream) != cudaSuccess ||
        cudaStreamSynchronize(stream) != cudaSuccess)
        return PMQA_ERR_CUDA;
    return (int)(host & 0x7FFFFFFFu);
}

const char *pmqa_status_string(int code)
{
    switch (code) {
    case PMQA_OK: return "ok";
    case PMQA_ERR_INVALID_ARG: return "invalid argument";
    case PMQA_ERR_UNSUPPORTED: return "unsupported shape";
    case PMQA_ERR_WORKSPACE: return "workspace too small";
    case PMQA_ERR_CUDA: return "CUDA runtime error";
    case PMQA_ERR_DEVICE: return "device-side check failed";
    default: return "unknown status";
    }
}

int pmqa_version(void) { return kVersion; }

}  // extern "C"
