// Instantiations of the streaming 2:4 sparse INT4 GEMV kernel for batch 1..8 (see stream_kernel.cuh).
#include <atomic>

#include "stream_kernel.cuh"

namespace sgemv {

namespace {

template <int FMT, int B>
cudaError_t launch_stream_b(const StreamGroup& g, int grid, uint32_t smem, cudaStream_t s) {
    auto kern = stream_kernel<FMT, B>;
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

}  // namespace

cudaError_t launch_stream_sparse24(int batch, const StreamGroup& g, int grid, uint32_t smem, cudaStream_t s) {
    switch (batch) {
        case 1: return launch_stream_b<SGEMV_FMT_SPARSE24, 1>(g, grid, smem, s);
        case 2: return launch_stream_b<SGEMV_FMT_SPARSE24, 2>(g, grid, smem, s);
        case 3: return launch_stream_b<SGEMV_FMT_SPARSE24, 3>(g, grid, smem, s);
        case 4: return launch_stream_b<SGEMV_FMT_SPARSE24, 4>(g, grid, smem, s);
        case 5: return launch_stream_b<SGEMV_FMT_SPARSE24, 5>(g, grid, smem, s);
        case 6: return launch_stream_b<SGEMV_FMT_SPARSE24, 6>(g, grid, smem, s);
        case 7: return launch_stream_b<SGEMV_FMT_SPARSE24, 7>(g, grid, smem, s);
        case 8: return launch_stream_b<SGEMV_FMT_SPARSE24, 8>(g, grid, smem, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace sgemv
