// Instantiations of the 2:4 sparse INT4 GEMV kernel for batch 1..8 (see gemv_kernel.cuh).
#include "launch.cuh"

namespace sgemv {

cudaError_t launch_gemv_sparse(int batch, const LayerGroup& g, int grid, uint32_t smem, cudaStream_t s) {
    return launch_gemv<SGEMV_FMT_SPARSE24>(batch, g, grid, smem, s);
}

// Clusters of `split` CTAs of the split-K kernel that fit on the device at once. Every format and
// batch of that kernel has the same block (kThreads threads, one CTA per SM by its registers), so the
// 2:4 batch-1 instance with the largest x tile stands for all.
cudaError_t query_max_clusters(int split, int* out) {
    auto kern = gemv_kernel<SGEMV_FMT_SPARSE24, 1, false, true>;
    const int smem = static_cast<int>(kXTileBudget + 4u * kMaxPassRows);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(split));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(split);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaOccupancyMaxActiveClusters(out, kern, &cfg);
}

}  // namespace sgemv
