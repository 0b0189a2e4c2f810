// Instantiations of the dense INT4 GEMV kernel for batch 1..8 (see gemv_kernel.cuh).
#include "launch.cuh"

namespace sgemv {

cudaError_t launch_gemv_dense(int batch, const LayerGroup& g, int grid, uint32_t smem, cudaStream_t s) {
    return launch_gemv<SGEMV_FMT_DENSE>(batch, g, grid, smem, s);
}

}  // namespace sgemv
