// Instantiations of the streaming dense INT4 GEMV kernel, group size 128, batch 1..8
// (see stream_kernel.cuh).
#include "stream_launch.cuh"

namespace sgemv {

cudaError_t launch_streamd_g128(int batch, const StreamGroup& g, int grid, uint32_t smem, cudaStream_t s) {
    return launch_stream_lg<SGEMV_FMT_DENSE, 7>(batch, g, grid, smem, s);
}

}  // namespace sgemv
