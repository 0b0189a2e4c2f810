// Host launcher of gemv_kernel<FMT, B> for batch 1..8, shared by the per-format translation units
// (gemv_sparse.cu, gemv_sparse14.cu, gemv_dense.cu), each of which instantiates one format.
#pragma once

#include <atomic>

#include "gemv_kernel.cuh"

namespace sgemv {

template <int FMT, int B, bool kMulti>
cudaError_t launch_b(const LayerGroup& g, int grid, uint32_t smem, cudaStream_t s) {
    auto kern = gemv_kernel<FMT, B, kMulti>;
    static std::atomic<int> attr_smem[64];  // per device: dynamic shared memory already enabled
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (attr_smem[dev].load() < static_cast<int>(smem)) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        attr_smem[dev].store(static_cast<int>(smem));
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, g);
}

template <int FMT, bool kMulti>
cudaError_t launch_batch(int batch, const LayerGroup& g, int grid, uint32_t smem, cudaStream_t s) {
    switch (batch) {
        case 1: return launch_b<FMT, 1, kMulti>(g, grid, smem, s);
        case 2: return launch_b<FMT, 2, kMulti>(g, grid, smem, s);
        case 3: return launch_b<FMT, 3, kMulti>(g, grid, smem, s);
        case 4: return launch_b<FMT, 4, kMulti>(g, grid, smem, s);
        case 5: return launch_b<FMT, 5, kMulti>(g, grid, smem, s);
        case 6: return launch_b<FMT, 6, kMulti>(g, grid, smem, s);
        case 7: return launch_b<FMT, 7, kMulti>(g, grid, smem, s);
        case 8: return launch_b<FMT, 8, kMulti>(g, grid, smem, s);
        default: return cudaErrorInvalidValue;
    }
}

template <int FMT>
cudaError_t launch_gemv(int batch, const LayerGroup& g, int grid, uint32_t smem, cudaStream_t s) {
    return g.n_layers > 1 ? launch_batch<FMT, true>(batch, g, grid, smem, s)
                          : launch_batch<FMT, false>(batch, g, grid, smem, s);
}

}  // namespace sgemv
