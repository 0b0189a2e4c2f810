// Launchers that the host-only checks link instead of the kernels' translation units: the planner in
// abi.cu references them, the checks never call them.
#include "common.cuh"

namespace sgemv {
cudaError_t launch_gemv_sparse(int, const LayerGroup&, int, uint32_t, cudaStream_t) { return cudaErrorNotSupported; }
cudaError_t launch_gemv_sparse14(int, const LayerGroup&, int, uint32_t, cudaStream_t) { return cudaErrorNotSupported; }
cudaError_t launch_gemv_dense(int, const LayerGroup&, int, uint32_t, cudaStream_t) { return cudaErrorNotSupported; }
cudaError_t launch_pack(const PackParams&, int, cudaStream_t) { return cudaErrorNotSupported; }
cudaError_t query_max_clusters(int, int*) { return cudaErrorNotSupported; }
cudaError_t launch_stream24_g64(int, const StreamGroup&, int, uint32_t, cudaStream_t) { return cudaErrorNotSupported; }
cudaError_t launch_stream24_g128(int, const StreamGroup&, int, uint32_t, cudaStream_t) { return cudaErrorNotSupported; }
cudaError_t launch_stream24_g256(int, const StreamGroup&, int, uint32_t, cudaStream_t) { return cudaErrorNotSupported; }
cudaError_t launch_stream14_g64(int, const StreamGroup&, int, uint32_t, cudaStream_t) { return cudaErrorNotSupported; }
cudaError_t launch_stream14_g128(int, const StreamGroup&, int, uint32_t, cudaStream_t) { return cudaErrorNotSupported; }
cudaError_t launch_stream14_g256(int, const StreamGroup&, int, uint32_t, cudaStream_t) { return cudaErrorNotSupported; }
cudaError_t launch_streamd_g64(int, const StreamGroup&, int, uint32_t, cudaStream_t) { return cudaErrorNotSupported; }
cudaError_t launch_streamd_g128(int, const StreamGroup&, int, uint32_t, cudaStream_t) { return cudaErrorNotSupported; }
cudaError_t launch_streamd_g256(int, const StreamGroup&, int, uint32_t, cudaStream_t) { return cudaErrorNotSupported; }
}  // namespace sgemv
