// Instantiations of the 2:4 sparse INT4 GEMV kernel for batch 1..8 (see gemv_kernel.cuh).
#include "launch.cuh"

namespace sgemv {

cudaError_t launch_gemv_sparse(int batch, const LayerGroup& g, int grid, uint32_t smem, cudaStream_t s) {
    return launch_gemv<SGEMV_FMT_SPARSE24>(batch, g, grid, smem, s);
}

}  // namespace sgemv
