// Instantiations of the streaming 2:4 sparse INT4 GEMV kernel, group size 256, batch 1..8
// (see stream_kernel.cuh).
#include "stream_launch.cuh"

namespace sgemv {

cudaError_t launch_stream24_g256(int batch, const StreamGroup& g, int grid, uint32_t smem, cudaStream_t s) {
    return launch_stream_lg<SGEMV_FMT_SPARSE24, 8>(batch, g, grid, smem, s);
}

}  // namespace sgemv
