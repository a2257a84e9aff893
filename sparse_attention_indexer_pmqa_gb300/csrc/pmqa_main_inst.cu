// pmqa_main_inst.cu -- one translation unit per supported head count, so the
// four instantiations of the main kernel compile in parallel. Built with
// -DPMQA_HEADS=16, 32, 64 or 128.
#include <cuda_runtime.h>

#include "pmqa_main.cuh"

#ifndef PMQA_HEADS
#error "PMQA_HEADS must be defined"
#endif

#define PMQA_CAT2(a, b) a##b
#define PMQA_CAT(a, b) PMQA_CAT2(a, b)

namespace pmqa {

cudaError_t PMQA_CAT(launch_main_h, PMQA_HEADS)(const MainArgs &a, bool fused, int grid,
                                                int threads, cudaStream_t stream)
{
    const void *fn = fused ? reinterpret_cast<const void *>(&pmqa_main_kernel<PMQA_HEADS, true>)
                           : reinterpret_cast<const void *>(&pmqa_main_kernel<PMQA_HEADS, false>);
    cudaError_t e =
        cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)a.smem_bytes);
    if (e != cudaSuccess)
        return e;
    if (fused)
        pmqa_main_kernel<PMQA_HEADS, true><<<grid, threads, a.smem_bytes, stream>>>(a);
    else
        pmqa_main_kernel<PMQA_HEADS, false><<<grid, threads, a.smem_bytes, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace pmqa
