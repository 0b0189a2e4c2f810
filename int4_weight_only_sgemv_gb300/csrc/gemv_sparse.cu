// Instantiations of the 2:4 sparse INT4 GEMV kernel on the CUDA cores (see gemv_kernel.cuh) for the
// batches below kTcMinBatch; larger batches run on the tensor-core kernel (gemv_tc.cuh).
#include "launch.cuh"

namespace sgemv {

static_assert(kTcMinBatch == 2, "the CUDA-core 2:4 kernel is instantiated for batch 1 only");

cudaError_t launch_gemv_sparse(int batch, const LayerGroup& g, int grid, uint32_t smem, cudaStream_t s) {
    if (batch != 1) return cudaErrorInvalidValue;
    return g.n_layers > 1 ? launch_b<SGEMV_FMT_SPARSE24, 1, true>(g, grid, smem, s)
                          : launch_b<SGEMV_FMT_SPARSE24, 1, false>(g, grid, smem, s);
}

}  // namespace sgemv
