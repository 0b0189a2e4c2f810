// Host launcher of gemv_kernel<FMT, B> for batch 1..8, shared by the per-format translation units
// (gemv_sparse.cu, gemv_sparse14.cu, gemv_dense.cu), each of which instantiates one format.
#pragma once

#include <atomic>

#include "gemv_kernel.cuh"

namespace sgemv {

template <int FMT, int B, bool kMulti, bool kSplit>
cudaError_t launch_b(const LayerGroup& g, int grid, uint32_t smem, cudaStream_t s) {
    auto kern = gemv_kernel<FMT, B, kMulti, kSplit>;
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
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (kSplit) {  // clusters of `split` CTAs share a row range (grid is a multiple of split)
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = static_cast<unsigned>(g.layer[0].split);
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        cfg.numAttrs = 2;
    }
    return cudaLaunchKernelEx(&cfg, kern, g);
}

template <int FMT, bool kMulti, bool kSplit>
cudaError_t launch_batch(int batch, const LayerGroup& g, int grid, uint32_t smem, cudaStream_t s) {
    switch (batch) {
        case 1: return launch_b<FMT, 1, kMulti, kSplit>(g, grid, smem, s);
        case 2: return launch_b<FMT, 2, kMulti, kSplit>(g, grid, smem, s);
        case 3: return launch_b<FMT, 3, kMulti, kSplit>(g, grid, smem, s);
        case 4: return launch_b<FMT, 4, kMulti, kSplit>(g, grid, smem, s);
        case 5: return launch_b<FMT, 5, kMulti, kSplit>(g, grid, smem, s);
        case 6: return launch_b<FMT, 6, kMulti, kSplit>(g, grid, smem, s);
        case 7: return launch_b<FMT, 7, kMulti, kSplit>(g, grid, smem, s);
        case 8: return launch_b<FMT, 8, kMulti, kSplit>(g, grid, smem, s);
        default: return cudaErrorInvalidValue;
    }
}

// A group of several layers (never split), one layer split over K by clusters, or one layer.
template <int FMT>
cudaError_t launch_gemv(int batch, const LayerGroup& g, int grid, uint32_t smem, cudaStream_t s) {
    if (g.n_layers > 1) return launch_batch<FMT, true, false>(batch, g, grid, smem, s);
    if (g.layer[0].split > 1) return launch_batch<FMT, false, true>(batch, g, grid, smem, s);
    return launch_batch<FMT, false, false>(batch, g, grid, smem, s);
}

}  // namespace sgemv
