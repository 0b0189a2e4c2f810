// Internal definitions shared by the CUDA sources of libsgemv (not part of the public ABI).
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "sgemv.h"

namespace sgemv {

// ------------------------------------------------------------------------------------------------
// Packed layout (FORMAT.md sections 3-4), computed on the host.

constexpr uint32_t kMagic = 0x564D4753u;  // "SGMV"
constexpr uint32_t kVersion = 1;

int compute_layout(int format, int n, int k, int group, sgemv_layout* out);
bool layout_equal(const sgemv_layout& a, const sgemv_layout& b);

// ------------------------------------------------------------------------------------------------
// Kernel parameters.

struct PackParams {
    const uint16_t* w;   // fp16 bits [n][k]
    uint8_t* packed;     // base of the packed buffer
    int32_t* status;     // nullable
    sgemv_layout L;
    int log2g;
};

// Shape of the GEMV work of one launch (both formats). All byte quantities are per row.
struct GemvParams {
    const uint8_t* vals;   // section bases
    const uint8_t* idx;
    const uint8_t* sz;
    uint32_t vals_pitch, idx_pitch, sz_pitch;
    const __half* x;       // [B][K]
    __half* y;             // [B][N]
    int32_t* status;       // nullable
    int n, k, log2g;
    // Row partition: CTA c owns rows [c*rows_base + min(c, rows_rem), ... + rows_base + (c < rows_rem)).
    int rows_base, rows_rem;
    int cs;                // columns per pipeline stage (multiple of 1024, the last stage may be shorter)
    int xt;                // columns per x tile (multiple of cs)
    int pass_rows;         // rows whose fp32 sums are held in shared memory at once (multiple of 4)
    int nstage;            // pipeline depth
    // shared-memory layout (byte offsets from the dynamic shared-memory base)
    uint32_t st_bytes;     // bytes of one stage slot
    uint32_t st_vals_pitch, st_idx_off, st_idx_pitch, st_sz_off, st_sz_pitch;
    uint32_t sm_x;         // x tile: [B][xt/64 chunks][144 bytes]
    uint32_t x_b_stride;   // bytes per batch row of the x tile
    uint32_t sm_acc;       // fp32 [B][pass_rows]
    uint32_t sm_bar;       // 2*nstage mbarriers (full, empty) + abort flag
};

constexpr int kConsumerWarps = 16;
constexpr int kThreads = (kConsumerWarps + 1) * 32;  // + one producer warp
constexpr int kSlabCols = 512;                       // columns of one consumer task (8 lanes x 64)
constexpr int kRowsPerStage = 4;                     // rows of one stage = rows of one task
constexpr uint32_t kXChunkBytes = 144;               // 64 fp16 columns + 16 bytes of padding

// ------------------------------------------------------------------------------------------------
// Device helpers (inline PTX): mbarriers, bulk async copies, timers, dependent launch.

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bulk copy global -> shared of `bytes` (multiple of 16, both addresses 16-byte aligned); completion
// is signalled on the mbarrier as transaction bytes.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Programmatic dependent launch: block until the preceding kernel in the stream has completed and
// its memory is visible / allow the next kernel in the stream to be scheduled.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Named barrier 1 among the consumer warps only (the producer warp never takes part).
__device__ __forceinline__ void consumer_bar() {
    asm volatile("bar.sync 1, %0;" ::"r"(kConsumerWarps * 32) : "memory");
}

// Every wait on an mbarrier gives up after this long; the kernel then records SGEMV_ERR_TIMEOUT,
// stops issuing work and drains its own copies before exiting.
constexpr uint64_t kWaitTimeoutNs = 200ull * 1000 * 1000;
constexpr uint32_t kWaitMaxIters = 1u << 28;

// Wait for phase `parity` of `bar`. Returns false if the CTA abort flag is (or becomes) set or if the
// wait exceeds its time/iteration limit (in which case this call sets the abort flag).
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                                  int32_t* status) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 1; it < kWaitMaxIters; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 15u) == 0) {
            if (*abort_flag) return false;
            if (globaltimer_ns() - t0 > kWaitTimeoutNs) break;
        }
    }
    *abort_flag = 1;
    if (status) atomicCAS(reinterpret_cast<int*>(status), 0, SGEMV_ERR_TIMEOUT);
    return false;
}

// Device-side information cached per device by the host code.
struct DeviceInfo {
    int sm_count = 0;
    int max_smem_optin = 0;
};
int device_info(DeviceInfo* out);  // host: for the current device

// Launch geometry and shared-memory plan of one GEMV (abi.cu); exposed for host-side checks.
int plan_gemv(const sgemv_layout& L, const void* packed, const void* x, int batch, void* y, int32_t* status,
              const DeviceInfo& di, GemvParams* pp, int* grid, uint32_t* smem);

// Host launchers implemented in gemv_sparse.cu / gemv_dense.cu / pack.cu.
cudaError_t launch_gemv_sparse(int batch, const GemvParams& p, int grid, uint32_t smem, cudaStream_t s);
cudaError_t launch_gemv_dense(int batch, const GemvParams& p, int grid, uint32_t smem, cudaStream_t s);
cudaError_t launch_pack(const PackParams& p, int grid, cudaStream_t s);

}  // namespace sgemv
