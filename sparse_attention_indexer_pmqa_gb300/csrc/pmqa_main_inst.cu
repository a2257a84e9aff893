// pmqa_main_inst.cu -- one translation unit per supported head count, so the
// main kernel's instantiations for the four head counts compile in parallel. Built with
// -DPMQA_HEADS=16, 32, 64 or 128.
#include <cuda_runtime.h>

#include "pmqa_kernel.cuh"

#ifndef PMQA_HEADS
#error "PMQA_HEADS must be defined"
#endif

#define PMQA_CAT2(a, b) a##b
#define PMQA_CAT(a, b) PMQA_CAT2(a, b)

namespace pmqa {

template <bool SLICED, bool PAGE>
static cudaError_t launch(const MainArgs &a, int grid, int threads, cudaStream_t stream)
{
    cudaError_t e = cudaFuncSetAttribute(pmqa_main_kernel<PMQA_HEADS, SLICED, PAGE>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)a.smem_bytes);
    if (e != cudaSuccess)
        return e;
    pmqa_main_kernel<PMQA_HEADS, SLICED, PAGE><<<grid, threads, a.smem_bytes, stream>>>(a);
    return cudaGetLastError();
}

cudaError_t PMQA_CAT(launch_main_h, PMQA_HEADS)(const MainArgs &a, int grid, int threads,
                                                cudaStream_t stream)
{
    // the gather's two row-copy modes and the slice variant compile apart
    if (a.page_mode)
        return a.tok_begin ? launch<true, true>(a, grid, threads, stream)
                           : launch<false, true>(a, grid, threads, stream);
    return a.tok_begin ? launch<true, false>(a, grid, threads, stream)
                       : launch<false, false>(a, grid, threads, stream);
}

}  // namespace pmqa
