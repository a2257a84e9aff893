// pmqa_prefill_inst.cu -- the prefill kernel for one head count per
// translation unit (-DPMQA_HEADS=16, 32, 64 or 128), compiled in parallel;
// the head-count-independent prep kernel lives in the 16-head unit.
#include <cuda_runtime.h>

#if PMQA_HEADS == 16
#define PMQA_PREFILL_PREP
#endif
#include "pmqa_prefill.cuh"

#ifndef PMQA_HEADS
#error "PMQA_HEADS must be defined"
#endif

#define PMQA_CAT2(a, b) a##b
#define PMQA_CAT(a, b) PMQA_CAT2(a, b)

namespace pmqa {

cudaError_t PMQA_CAT(launch_prefill_h, PMQA_HEADS)(const PfArgs &a, int grid, int threads,
                                                   cudaStream_t stream)
{
    cudaError_t e = cudaFuncSetAttribute(pmqa_prefill_kernel<PMQA_HEADS>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)a.smem_bytes);
    if (e != cudaSuccess)
        return e;
    // a programmatic dependent of the prep kernel: its launch and prologue
    // overlap the prep kernel's end
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3((unsigned)threads);
    cfg.dynamicSmemBytes = a.smem_bytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, pmqa_prefill_kernel<PMQA_HEADS>, a);
    if (e != cudaSuccess)
        return e;
    return cudaGetLastError();
}

#ifdef PMQA_PREFILL_PREP
cudaError_t launch_prefill_prep(const PfArgs &a, int grid, cudaStream_t stream)
{
    pmqa_prefill_prep_kernel<<<grid, 256, 0, stream>>>(a);
    return cudaGetLastError();
}
#endif

}  // namespace pmqa
