// Instantiations of the 2:4 sparse INT4 GEMV kernel on the sparse tensor cores for batch 1..8
// (see gemv_tc.cuh).
#include <atomic>

#include "gemv_tc.cuh"

namespace sgemv {

namespace {

template <int B, bool kMulti>
cudaError_t launch_tc_b(const LayerGroup& g, int grid, uint32_t smem, cudaStream_t s) {
    auto kern = gemv_tc_kernel<B, kMulti>;
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

template <bool kMulti>
cudaError_t launch_tc(int batch, const LayerGroup& g, int grid, uint32_t smem, cudaStream_t s) {
    switch (batch) {
        case 1: return launch_tc_b<1, kMulti>(g, grid, smem, s);
        case 2: return launch_tc_b<2, kMulti>(g, grid, smem, s);
        case 3: return launch_tc_b<3, kMulti>(g, grid, smem, s);
        case 4: return launch_tc_b<4, kMulti>(g, grid, smem, s);
        case 5: return launch_tc_b<5, kMulti>(g, grid, smem, s);
        case 6: return launch_tc_b<6, kMulti>(g, grid, smem, s);
        case 7: return launch_tc_b<7, kMulti>(g, grid, smem, s);
        case 8: return launch_tc_b<8, kMulti>(g, grid, smem, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_gemv_sparse_tc(int batch, const LayerGroup& g, int grid, uint32_t smem, cudaStream_t s) {
    return g.n_layers > 1 ? launch_tc<true>(batch, g, grid, smem, s) : launch_tc<false>(batch, g, grid, smem, s);
}

}  // namespace sgemv
