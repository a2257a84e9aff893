// pmqa_api.cu -- the C ABI of include/pmqa.h: argument checks, workspace and
// shared-memory layout, TMA descriptor, kernel launches. No allocation, no
// synchronisation (except pmqa_read_device_status), no state kept between calls.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>

#include "../../include/pmqa.h"
#include "pmqa_main.cuh"
#include "pmqa_prefill.cuh"
#include "pmqa_select.cuh"

namespace pmqa {
cudaError_t launch_main_h16(const MainArgs &, int, int, cudaStream_t);
cudaError_t launch_main_h32(const MainArgs &, int, int, cudaStream_t);
cudaError_t launch_main_h64(const MainArgs &, int, int, cudaStream_t);
cudaError_t launch_main_h128(const MainArgs &, int, int, cudaStream_t);
cudaError_t launch_prefill_h16(const PfArgs &, int, int, cudaStream_t);
cudaError_t launch_prefill_h32(const PfArgs &, int, int, cudaStream_t);
cudaError_t launch_prefill_h64(const PfArgs &, int, int, cudaStream_t);
cudaError_t launch_prefill_h128(const PfArgs &, int, int, cudaStream_t);
cudaError_t launch_prefill_prep(const PfArgs &, int, cudaStream_t);
int fused_call_clearing_state(const pmqa_problem *p, int32_t k, int32_t *idx, float *vals,
                              float *logits, void *ws, size_t ws_bytes, cudaStream_t stream);
}  // namespace pmqa

using namespace pmqa;

namespace {

constexpr int kVersion = 300;  // 0.3.0
// 227 KB per CTA, shared between the static CtaCtl block and the dynamic layout
constexpr uint32_t kMaxDynSmem = 232448 - ((uint32_t)sizeof(CtaCtl) + 127u) / 128u * 128u;
constexpr uint32_t kMinMainSmem = 120 * 1024;  // > half an SM: one CTA per SM
constexpr size_t kWsAlign = 256;
constexpr int kSelChunk = kSelThreads * kSelPer;  // positions per selection CTA (8192)
// Tuning constants of the main kernel (compile time; -D overrides in tuning builds).
#ifndef PMQA_L2_POLICY
#define PMQA_L2_POLICY 0
#endif

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Workspace: status word | per-row counters | per-row histograms | tie lists
// of (position, order key) | compact logits (fused only). Everything before
// the tie lists must be zero when a call starts; every call leaves it zero
// again (status word aside).
struct WsLayout {
    size_t sel_cnt, tie_cnt, arrive, hist, ties, clogits, total;
};

bool ws_layout(long long rows, long long mml, int op, WsLayout *L)
{
    if (rows < 0 || mml < 1 || op < PMQA_OP_LOGITS || op > PMQA_OP_LOGITS_TOPK)
        return false;
    if (op == PMQA_OP_LOGITS) {
        L->sel_cnt = L->tie_cnt = L->arrive = L->hist = L->ties = L->clogits = L->total = kWsAlign;
        return true;
    }
    const size_t r4 = align_up((size_t)rows * 4, kWsAlign);
    L->sel_cnt = kWsAlign;
    L->tie_cnt = L->sel_cnt + r4;
    L->arrive = L->tie_cnt + r4;
    L->hist = L->arrive + r4;
    L->ties = L->hist + (size_t)rows * kHistBins * 4;
    L->clogits = L->ties + align_up((size_t)rows * (size_t)mml * 8, kWsAlign);
    L->total = op == PMQA_OP_LOGITS_TOPK ? L->clogits + (size_t)rows * (size_t)mml * 4 : L->clogits;
    return true;
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
    if (!aligned(p->q, 16) || !aligned(p->weights, 16) || !aligned(p->kv_cache, 16) ||
        !aligned(p->context_lens, 4) || !aligned(p->block_tables, 4))
        return PMQA_ERR_INVALID_ARG;
    return PMQA_OK;
}

// Shared-memory and TMEM layout of the main kernel: four warpgroup regions
// (staging slot + operand tile), then the query and weight slots (two when
// they fit) and the mbarriers. Each warpgroup owns cols TMEM columns.
bool main_layout(int heads, int nn, MainArgs &a)
{
    const int N = heads * nn;
    a.N = N;
    int cols = 32;
    while (cols < N && cols < kPassCols)
        cols <<= 1;
    a.cols = cols;
    a.tmem_cols = kGroups * cols;
    if (N > kPassCols && N <= 2 * kPassCols) {
        // two 256-column halves, each shared by two warpgroups in turn
        a.cols = 2 * kPassCols;
        a.tmem_cols = 4 * kPassCols;
    }
    for (int QS = 2; QS >= 1; --QS) {
        uint32_t off = 0;
        a.off_grp = off;
        off += (uint32_t)kGroups * kGroupBytes;
        a.off_q = off;  // 1024-byte aligned: 128B-swizzled TMA boxes
        off += (uint32_t)(QS * N * kHeadDim);
        a.off_w = off;
        off += (uint32_t)(QS * N * 4);
        off = (uint32_t)align_up(off, 16);
        a.off_bar = off;
        off += (uint32_t)(QS + kNumBars) * 8u;
        const uint32_t total = std::max<uint32_t>(off + 1024, kMinMainSmem);
        if (total > kMaxDynSmem)
            continue;
        a.QS = QS;
        a.smem_bytes = total;
        return true;
    }
    return false;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled()
{
    static EncodeTiledFn fn = nullptr;  // driver entry point, looked up once
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

// A [rows, 128 bytes] fp8 matrix as a 2-D tensor map; box [128 bytes, box_rows
// rows]; 128B swizzle (the K-major operand layout). Rows past the end read as zeros.
bool encode_rows_map(CUtensorMap *m, const void *q, long long rows, int box_rows)
{
    EncodeTiledFn fn = encode_tiled();
    if (!fn)
        return false;
    const cuuint64_t dims[2] = {(cuuint64_t)kHeadDim, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)kHeadDim};
    const cuuint32_t box[2] = {(cuuint32_t)kHeadDim, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(q), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

SelectArgs select_args(const float *logits, const int32_t *ctx, int bs, int nn, int mml,
                       long long ctx_lim, int k, int32_t *idx, float *vals, void *ws,
                       const WsLayout &L)
{
    uint8_t *b = static_cast<uint8_t *>(ws);
    SelectArgs s{};
    s.logits = logits;
    s.ctx_lens = ctx;
    s.bs = bs;
    s.nn = nn;
    s.mml = mml;
    s.ctx_lim = (int)std::min<long long>(ctx_lim, (long long)mml);
    s.k = k;
    s.idx = idx;
    s.vals = vals;
    s.status = reinterpret_cast<uint32_t *>(b);
    s.sel_cnt = reinterpret_cast<uint32_t *>(b + L.sel_cnt);
    s.tie_cnt = reinterpret_cast<uint32_t *>(b + L.tie_cnt);
    s.arrive = reinterpret_cast<uint32_t *>(b + L.arrive);
    s.hist = reinterpret_cast<uint32_t *>(b + L.hist);
    s.ties = reinterpret_cast<uint2 *>(b + L.ties);
    s.chunk = kSelChunk;
    s.splits = (mml + kSelChunk - 1) / kSelChunk;
    return s;
}

int launch_select(const SelectArgs &s, bool with_hist_pass, cudaStream_t stream)
{
    const long long rows = (long long)s.bs * s.nn;
    if (rows == 0)
        return PMQA_OK;
    if (rows > 65535)
        return PMQA_ERR_UNSUPPORTED;
    const dim3 grid((unsigned)s.splits, (unsigned)rows);
    if (with_hist_pass)
        pmqa_hist_kernel<<<grid, kSelThreads, 0, stream>>>(s);
    // a programmatic dependent of the preceding kernel (the KV pass on the
    // fused path): its launch overlaps that kernel's end
    cudaLaunchConfig_t cfg = {};
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (s.mml <= kRowMaxLen) {
        // rows short enough for one CTA each, the logits held in shared memory
        const int smem = s.mml * (int)sizeof(float);
        if (cudaFuncSetAttribute(pmqa_select_row_kernel<true>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kRowMaxLen * (int)sizeof(float)) != cudaSuccess)
            return PMQA_ERR_CUDA;
        cfg.gridDim = dim3((unsigned)rows);
        cfg.blockDim = dim3(kRowThreads);
        cfg.dynamicSmemBytes = (size_t)smem;
        if (cudaLaunchKernelEx(&cfg, pmqa_select_row_kernel<true>, s) != cudaSuccess)
            return PMQA_ERR_CUDA;
    } else if (s.mml <= kRowMaxLenStream) {
        // one CTA per row, the logits through shared memory in halves
        if (cudaFuncSetAttribute(pmqa_select_row_kernel<false>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kRowMaxLen * (int)sizeof(float)) != cudaSuccess)
            return PMQA_ERR_CUDA;
        cfg.gridDim = dim3((unsigned)rows);
        cfg.blockDim = dim3(kRowThreads);
        cfg.dynamicSmemBytes = (size_t)kRowMaxLen * sizeof(float);
        if (cudaLaunchKernelEx(&cfg, pmqa_select_row_kernel<false>, s) != cudaSuccess)
            return PMQA_ERR_CUDA;
    } else {
        cfg.gridDim = grid;
        cfg.blockDim = dim3(kSelThreads);
        cfg.dynamicSmemBytes = 0;
        if (cudaLaunchKernelEx(&cfg, pmqa_select_kernel, s) != cudaSuccess)
            return PMQA_ERR_CUDA;
    }
    return cudaGetLastError() == cudaSuccess ? PMQA_OK : PMQA_ERR_CUDA;
}

// clear_state: zero the workspace's counters and histograms on the stream
// first (after every argument check, so an error still enqueues nothing), for
// a workspace whose previous contents are unknown.
// tok_begin / tok_end: score and select only that slice of each request's
// tokens (the fused call without a logits output).
int run_main(const pmqa_problem *p, bool fused, int k, int32_t *idx, float *vals, float *logits,
             void *ws, size_t ws_bytes, cudaStream_t stream,
             int stages = PMQA_STAGE_SCORE | PMQA_STAGE_SELECT, bool clear_state = false,
             const int32_t *tok_begin = nullptr, const int32_t *tok_end = nullptr)
{
    if (stages < 1 || stages > (PMQA_STAGE_SCORE | PMQA_STAGE_SELECT))
        return PMQA_ERR_INVALID_ARG;
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
    if ((tok_begin != nullptr) != (tok_end != nullptr))
        return PMQA_ERR_INVALID_ARG;
    if (tok_begin && (!fused || logits || !aligned(tok_begin, 4) || !aligned(tok_end, 4)))
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
    if (!main_layout(p->heads, p->next_n, a))
        return PMQA_ERR_UNSUPPORTED;
    if (fused && rows > 65535)
        return PMQA_ERR_UNSUPPORTED;
    if (p->bs == 0)
        return PMQA_OK;
    const int nbox = (a.N + 255) / 256;
    a.q_box = a.N / nbox;
    if (a.q_box * nbox != a.N || a.q_box % 8 != 0)
        return PMQA_ERR_UNSUPPORTED;
    // q as [bs * N rows, 128 bytes]; q_box = N / ceil(N / 256) <= 256 rows, so
    // whole boxes cover one request exactly
    if (!encode_rows_map(&a.tmap_q, p->q, rows * p->heads, a.q_box))
        return PMQA_ERR_CUDA;
    uint8_t *wsb = static_cast<uint8_t *>(ws);
    a.q = static_cast<const uint8_t *>(p->q);
    a.kv = static_cast<const uint8_t *>(p->kv_cache);
    a.w = p->weights;
    a.ctx_lens = p->context_lens;
    a.bt = p->block_tables;
    a.num_blocks = p->num_blocks;
    a.pool_bytes = p->num_blocks * (long long)p->block_size * kKvRowBytes;
    a.bs = p->bs;
    a.nn = p->next_n;
    a.P = p->block_size;
    a.W = p->max_blocks_per_seq;
    a.mml = p->max_model_len;
    a.logits = logits;
    a.status = reinterpret_cast<uint32_t *>(wsb);
    a.l2_policy = PMQA_L2_POLICY;
    a.page_mode = (p->block_size % 4 == 0) ? 1 : 0;
    a.tok_begin = tok_begin;
    a.tok_end = tok_end;
    float *sel_src = logits;
    if (fused) {
        a.hist = reinterpret_cast<uint32_t *>(wsb + L.hist);
        if (!logits) {
            a.clogits = reinterpret_cast<float *>(wsb + L.clogits);
            sel_src = a.clogits;
        }
    }
    int sms = 0;
    if ((rc = sm_count(&sms)) != PMQA_OK)
        return rc;
    if (clear_state && fused && cudaMemsetAsync(ws, 0, L.ties, stream) != cudaSuccess)
        return PMQA_ERR_CUDA;
    if (stages & PMQA_STAGE_SCORE) {
        const int threads = kMaxThreads;
        cudaError_t e;
        switch (p->heads) {
        case 16: e = launch_main_h16(a, sms, threads, stream); break;
        case 32: e = launch_main_h32(a, sms, threads, stream); break;
        case 64: e = launch_main_h64(a, sms, threads, stream); break;
        default: e = launch_main_h128(a, sms, threads, stream); break;
        }
        if (e != cudaSuccess)
            return PMQA_ERR_CUDA;
    }
    if (!fused || !(stages & PMQA_STAGE_SELECT))
        return PMQA_OK;
    // the same context clamp as the KV pass, so both use one valid length
    SelectArgs s =
        select_args(sel_src, p->context_lens, p->bs, p->next_n, p->max_model_len,
                    (long long)p->max_blocks_per_seq * p->block_size, k, idx, vals, ws, L);
    s.tok_begin = tok_begin;
    s.tok_end = tok_end;
    return launch_select(s, false, stream);
}

// Shared-memory layout of the prefill kernel: a ring of S key stages, two query
// slots of 4 * G query rows (512 Q rows of 128 bytes) and their weights, the
// mbarriers.
bool pf_layout(int heads, PfArgs &a)
{
    a.SGR = kGroups * (kPassCols / heads);
    const uint32_t N = (uint32_t)(a.SGR * heads);
    const int QS = 2;  // the next super-group's MMAs start before the current one's slot is freed
    for (int S = kPfMaxStages; S >= 2; --S) {
        uint32_t off = 0;
        a.off_k = off;  // 1024-byte aligned stages
        off += (uint32_t)S * kStageBytes;
        a.off_q = off;
        off += (uint32_t)QS * N * kHeadDim;
        a.off_w = off;
        off += (uint32_t)QS * N * 4u;
        off = (uint32_t)align_up(off, 16);
        a.off_bar = off;
        off += (uint32_t)(S + QS + 4) * 8u;
        const uint32_t total = std::max<uint32_t>(off + 1024, kMinMainSmem);
        if (total > kMaxDynSmem)
            continue;
        a.S = S;
        a.QS = QS;
        a.smem_bytes = total;
        return true;
    }
    return false;
}

// Prefill workspace: the status word, then one (first tile, tile count) pair
// per super-group; super-groups hold at least 4 query rows.
size_t pf_ws_bytes(long long m) { return kWsAlign + align_up((size_t)((m + 3) / 4) * 8, kWsAlign); }

int run_prefill(const pmqa_mqa_problem *p, float *logits, void *ws, size_t ws_bytes,
                cudaStream_t stream)
{
    if (!p || p->m < 0 || p->n < 0 || p->heads < 1 || p->head_dim < 1)
        return PMQA_ERR_INVALID_ARG;
    if (p->head_dim != kHeadDim || !supported_heads(p->heads))
        return PMQA_ERR_UNSUPPORTED;
    // query rows address the q tensor map as int; key positions (tile * 128 + lane) as int
    if ((long long)p->m * p->heads >= (1ll << 31) || (long long)p->n > (1ll << 31) - 1 - kTileTokens)
        return PMQA_ERR_UNSUPPORTED;
    if (!ws || !aligned(ws, kWsAlign))
        return PMQA_ERR_INVALID_ARG;
    if (ws_bytes < pf_ws_bytes(p->m))
        return PMQA_ERR_WORKSPACE;
    if (p->m == 0 || p->n == 0)
        return PMQA_OK;
    if (!p->q || !p->k || !p->k_scale || !p->weights || !p->ks || !p->ke || !logits)
        return PMQA_ERR_INVALID_ARG;
    if (!aligned(p->q, 16) || !aligned(p->k, 16) || !aligned(p->weights, 16) ||
        !aligned(p->k_scale, 4) || !aligned(p->ks, 4) || !aligned(p->ke, 4) || !aligned(logits, 4))
        return PMQA_ERR_INVALID_ARG;
    PfArgs a{};
    if (!pf_layout(p->heads, a))
        return PMQA_ERR_UNSUPPORTED;
    const int N = a.SGR * p->heads;
    a.q_box = N / ((N + 255) / 256);
    if (!encode_rows_map(&a.tmap_q, p->q, (long long)p->m * p->heads, a.q_box) ||
        !encode_rows_map(&a.tmap_k, p->k, p->n, kTileTokens))
        return PMQA_ERR_CUDA;
    a.k_scale = p->k_scale;
    a.w = p->weights;
    a.ks = p->ks;
    a.ke = p->ke;
    a.logits = logits;
    a.status = static_cast<uint32_t *>(ws);
    a.ranges = reinterpret_cast<int2 *>(static_cast<uint8_t *>(ws) + kWsAlign);
    a.m = p->m;
    a.n = p->n;
    a.n_sg = (p->m + a.SGR - 1) / a.SGR;
    int sms = 0, rc;
    if ((rc = sm_count(&sms)) != PMQA_OK)
        return rc;
    if (launch_prefill_prep(a, std::min(a.n_sg, 8 * sms), stream) != cudaSuccess)
        return PMQA_ERR_CUDA;
    cudaError_t e;
    switch (p->heads) {
    case 16: e = launch_prefill_h16(a, sms, kPfThreads, stream); break;
    case 32: e = launch_prefill_h32(a, sms, kPfThreads, stream); break;
    case 64: e = launch_prefill_h64(a, sms, kPfThreads, stream); break;
    default: e = launch_prefill_h128(a, sms, kPfThreads, stream); break;
    }
    return e == cudaSuccess ? PMQA_OK : PMQA_ERR_CUDA;
}

}  // namespace

namespace pmqa {
// The fused call on a workspace whose previous contents are unknown: its
// counters and histograms are zeroed on the stream once every argument check
// has passed.
int fused_call_clearing_state(const pmqa_problem *p, int32_t k, int32_t *idx, float *vals,
                              float *logits, void *ws, size_t ws_bytes, cudaStream_t stream)
{
    return run_main(p, true, k, idx, vals, logits, ws, ws_bytes, stream,
                    PMQA_STAGE_SCORE | PMQA_STAGE_SELECT, true);
}
}  // namespace pmqa

extern "C" {

size_t pmqa_workspace_bytes(int32_t bs, int32_t next_n, int32_t max_model_len, int32_t k, int op)
{
    (void)k;
    if (op == PMQA_OP_MQA_LOGITS)
        return bs < 0 ? 0 : pf_ws_bytes(bs);
    if (bs < 0 || next_n < 1 || max_model_len < 1)
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

int pmqa_logits_topk_range(const pmqa_problem *p, const int32_t *token_begin,
                           const int32_t *token_end, int32_t k, int32_t *idx, float *vals,
                           void *ws, size_t ws_bytes, pmqa_stream_t stream)
{
    if (!token_begin || !token_end)
        return PMQA_ERR_INVALID_ARG;
    return run_main(p, true, k, idx, vals, nullptr, ws, ws_bytes, stream,
                    PMQA_STAGE_SCORE | PMQA_STAGE_SELECT, false, token_begin, token_end);
}

int pmqa_logits_topk_stages(const pmqa_problem *p, int32_t k, int32_t *idx, float *vals,
                            float *logits, void *ws, size_t ws_bytes, pmqa_stream_t stream,
                            int32_t stages)
{
    return run_main(p, true, k, idx, vals, logits, ws, ws_bytes, stream, stages);
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
    if (rows > 65535)
        return PMQA_ERR_UNSUPPORTED;
    if (bs == 0)
        return PMQA_OK;
    if (!logits || !context_lens || !idx || !aligned(logits, 4) || !aligned(context_lens, 4) ||
        !aligned(idx, 4) || (vals && !aligned(vals, 4)))
        return PMQA_ERR_INVALID_ARG;
    const SelectArgs s = select_args(logits, context_lens, bs, next_n, max_model_len,
                                     max_model_len, k, idx, vals, ws, L);
    return launch_select(s, true, stream);
}

int pmqa_topk_merge(const int32_t *idx, const float *vals, int32_t lists, int32_t rows,
                    int32_t k_in, int32_t k, int32_t *out_idx, float *out_vals,
                    pmqa_stream_t stream)
{
    if (lists < 1 || rows < 0 || k_in < 1 || k < 1)
        return PMQA_ERR_INVALID_ARG;
    if ((long long)lists * k_in >= (1ll << 31))
        return PMQA_ERR_UNSUPPORTED;
    if (rows == 0)
        return PMQA_OK;
    if (!idx || !vals || !out_idx || !aligned(idx, 4) || !aligned(vals, 4) || !aligned(out_idx, 4) ||
        (out_vals && !aligned(out_vals, 4)))
        return PMQA_ERR_INVALID_ARG;
    MergeArgs m{};
    m.idx = idx;
    m.vals = vals;
    m.lists = lists;
    m.rows = rows;
    m.k_in = k_in;
    m.k = k;
    m.out_idx = out_idx;
    m.out_vals = out_vals;
    pmqa_merge_kernel<<<(unsigned)rows, kSelThreads, 0, stream>>>(m);
    return cudaGetLastError() == cudaSuccess ? PMQA_OK : PMQA_ERR_CUDA;
}

int pmqa_mqa_logits(const pmqa_mqa_problem *p, float *logits, void *ws, size_t ws_bytes,
                    pmqa_stream_t stream)
{
    return run_prefill(p, logits, ws, ws_bytes, stream);
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
