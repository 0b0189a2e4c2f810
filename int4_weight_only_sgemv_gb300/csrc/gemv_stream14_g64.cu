// Instantiations of the streaming 1:4 sparse INT4 GEMV kernel, group size 64, batch 1..8
// (see stream_kernel.cuh).
#include "stream_launch.cuh"

namespace sgemv {

cudaError_t launch_stream14_g64(int batch, const StreamGroup& g, int grid, uint32_t smem, cudaStream_t s) {
    return launch_stream_lg<SGEMV_FMT_SPARSE14, 6>(batch, g, grid, smem, s);
}

}  // namespace sgemv
