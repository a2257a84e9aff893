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

template <int NN, bool SLICED, bool PAGE, bool POOL32>
static cudaError_t launch(const MainArgs &a, int grid, int threads, cudaStream_t stream)
{
    auto *kern = pmqa_main_kernel<PMQA_HEADS, NN, SLICED, PAGE, POOL32>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)a.smem_bytes);
    if (e != cudaSuccess)
        return e;
    kern<<<grid, threads, a.smem_bytes, stream>>>(a);
    return cudaGetLastError();
}

// The gather's row-copy mode (page runs; windows with 32- or 64-bit offsets)
// and the slice variant.
template <int NN>
static cudaError_t launch_nn(const MainArgs &a, int grid, int threads, cudaStream_t stream)
{
    const bool sliced = a.tok_begin != nullptr;
    if (a.page_mode)
        return sliced ? launch<NN, true, true, false>(a, grid, threads, stream)
                      : launch<NN, false, true, false>(a, grid, threads, stream);
    if (a.pool_bytes < (1ll << 31) - 1024)  // every byte offset fits in 31 bits
        return sliced ? launch<NN, true, false, true>(a, grid, threads, stream)
                      : launch<NN, false, false, true>(a, grid, threads, stream);
    return sliced ? launch<NN, true, false, false>(a, grid, threads, stream)
                  : launch<NN, false, false, false>(a, grid, threads, stream);
}

cudaError_t PMQA_CAT(launch_main_h, PMQA_HEADS)(const MainArgs &a, int grid, int threads,
                                                cudaStream_t stream)
{
    switch (a.nn) {
    case 1: return launch_nn<1>(a, grid, threads, stream);
    case 2: return launch_nn<2>(a, grid, threads, stream);
    case 3: return launch_nn<3>(a, grid, threads, stream);
    default: return launch_nn<4>(a, grid, threads, stream);
    }
}

}  // namespace pmqa
