// pmqa_noalloc.cu -- pmqa_logits_topk for callers that cannot allocate device
// memory: the workspace the fused kernel needs comes from a fixed array that
// the library itself places in device memory, instead of from the caller.
//
// Who needs this: code that is handed device pointers for its inputs and
// outputs but has no way to obtain more device memory -- for example a plugin
// running inside a host program that owns the whole device-memory pool and
// exposes no allocation hook, or a latency-critical loop that must not call
// cudaMalloc (which may synchronise the device).
//
// The array is 32 MiB; every GPU on which the library is loaded keeps it until
// the process exits. A problem whose workspace (pmqa_workspace_bytes for
// PMQA_OP_LOGITS_TOPK) exceeds it is rejected with PMQA_ERR_WORKSPACE before
// anything is enqueued.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "../../include/pmqa.h"

namespace pmqa {
int fused_call_clearing_state(const pmqa_problem *p, int32_t k, int32_t *idx, float *vals,
                              float *logits, void *ws, size_t ws_bytes, cudaStream_t stream);
}

namespace {

constexpr size_t kScratchBytes = size_t(32) << 20;
constexpr int kMaxDevices = 64;

// Device-resident scratch. In host code this name is only a handle for the
// runtime; its device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) uint8_t g_scratch[kScratchBytes];

std::mutex g_setup_mutex;
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of g_scratch on the current device, looked up once per device.
int scratch_for_current_device(void **out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return PMQA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || !p)
            return PMQA_ERR_CUDA;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return PMQA_OK;
}

}  // namespace

extern "C" int pmqa_logits_topk_noalloc(const pmqa_problem *p, int32_t k, int32_t *idx,
                                        float *vals, float *logits, pmqa_stream_t stream)
{
    if (!p)
        return PMQA_ERR_INVALID_ARG;
    const size_t need =
        pmqa_workspace_bytes(p->bs, p->next_n, p->max_model_len, k, PMQA_OP_LOGITS_TOPK);
    if (need == 0)
        return PMQA_ERR_INVALID_ARG;
    if (need > kScratchBytes)
        return PMQA_ERR_WORKSPACE;
    void *ws = nullptr;
    int rc = scratch_for_current_device(&ws);
    if (rc != PMQA_OK)
        return rc;
    // The array keeps whatever the previous call left. The fused call needs its
    // status word, per-row counters and per-row histograms at zero (the rest is
    // always written before it is read); it clears them on the stream once
    // every argument has been checked, so a rejected call enqueues nothing.
    return pmqa::fused_call_clearing_state(p, k, idx, vals, logits, ws, kScratchBytes, stream);
}
