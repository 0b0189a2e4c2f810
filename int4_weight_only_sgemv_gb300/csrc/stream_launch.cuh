// Host launcher of stream_kernel<FMT, B, LG, kCopyX> for batch 1..kStreamMaxBatch (3), shared by the
// per-format, per-group-size translation units (gemv_stream{24,14,d}_g{64,128,256}.cu), compiled in
// parallel.
#pragma once

#include <atomic>

#include "stream_kernel.cuh"

namespace sgemv {

template <int FMT, int B, int LG>
cudaError_t launch_stream_b(const StreamGroup& g, int grid, uint32_t smem, cudaStream_t s) {
    const bool copy_x = g.xraw_off != 0;
    auto kern = copy_x ? stream_kernel<FMT, B, LG, true> : stream_kernel<FMT, B, LG, false>;
    static std::atomic<int> attr_smem[2][64];  // per instance and device: dynamic shared memory enabled
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::atomic<int>& done = attr_smem[copy_x ? 1 : 0][dev];
    if (done.load() < static_cast<int>(smem)) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        done.store(static_cast<int>(smem));
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

template <int FMT, int LG>
cudaError_t launch_stream_lg(int batch, const StreamGroup& g, int grid, uint32_t smem, cudaStream_t s) {
    switch (batch) {
        case 1: return launch_stream_b<FMT, 1, LG>(g, grid, smem, s);
        case 2: return launch_stream_b<FMT, 2, LG>(g, grid, smem, s);
        case 3: return launch_stream_b<FMT, 3, LG>(g, grid, smem, s);
        default: return cudaErrorInvalidValue;  // batch > kStreamMaxBatch runs the tiled kernel
    }
}

}  // namespace sgemv
