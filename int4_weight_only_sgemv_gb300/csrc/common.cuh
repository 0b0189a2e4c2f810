// Internal definitions shared by the CUDA sources of libsgemv (not part of the public ABI).
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "sgemv.h"

namespace sgemv {

// ------------------------------------------------------------------------------------------------
// Packed layout (packed format v1, sections 3-4), computed on the host.

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
    // Row partition over the first nctas row units of the grid: unit u < nctas owns rows
    // [u*rows_base + min(u, rows_rem), ... + rows_base + (u < rows_rem)); units u >= nctas own none. A row
    // unit is one CTA, or with split-K (split > 1) one cluster of `split` CTAs that share the unit's rows
    // and take consecutive, balanced ranges of 1024-column blocks of K.
    int nctas, rows_base, rows_rem;
    int xt;                // columns per x tile (multiple of kTaskCols, or K)
    int pass_rows;         // rows whose fp32 sums are held in shared memory at once (multiple of 4)
    // shared-memory layout (byte offsets from the dynamic shared-memory base)
    uint32_t sm_x;         // x tile: [B][roundup(xt, 1024)/64 chunks][144 bytes], zero beyond the tile
    uint32_t x_b_stride;   // bytes per batch row of the x tile
    uint32_t sm_acc;       // fp32 [B][pass_rows]
    int split;             // CTAs per row unit: 1, or the cluster size with split-K
};

// Layers one launch can run (a group of independent layers of the same format and batch).
constexpr int kMaxGroup = 8;
struct LayerGroup {
    int n_layers;
    GemvParams layer[kMaxGroup];
};

constexpr int kWarps = 16;
constexpr int kThreads = kWarps * 32;
constexpr int kChunkCols = 64;                       // columns of one chunk (32 kept when sparse)
constexpr int kLaneCols = 2 * kChunkCols;            // columns of one lane in a task: two adjacent chunks
constexpr int kTaskCols = 8 * kLaneCols;             // 1024: columns of one task (8 column-lanes)
constexpr int kRowsPerTask = 4;                      // rows of one task (4 lane groups of 8)
// Tasks whose weights a warp keeps in flight: deeper at small batch, where the compute per byte is short.
template <int B>
__host__ __device__ constexpr int prefetch_depth() { return B <= 2 ? 3 : (B <= 4 ? 2 : 1); }
constexpr uint32_t kXLaneBytes = 272;                // x of one lane's 128 columns (256 bytes) + 16 bytes of padding
constexpr int kXWarps = 8;                           // warps that stage x into shared memory
constexpr int kXThreads = kXWarps * 32;
constexpr uint32_t kPrefetchPiece = 32768;             // bytes per L2 prefetch request
constexpr int kXStageRegs = 8;                       // 16-byte x units a staging thread has in flight

// Streaming kernel (stream_kernel.cuh). The rows of every layer of a launch are taken four at a time
// (a quad) and cut into units; a (quad, unit) pair is 4 units of the same columns. The pairs
// of all layers form one flat list per CTA; a warp takes 8 consecutive pairs per round (lane (r, j):
// row r of pair j), so the 4 row-lanes of a pair read the same x.
// Columns of one unit: 64 bytes of nibbles (256 columns for 2:4 and 1:4, 128 for dense INT4).
__host__ __device__ constexpr int stream_unit_cols(int fmt) { return fmt == SGEMV_FMT_DENSE ? 128 : 256; }
// x of one unit in shared memory: 2 bytes per column plus 16 bytes of padding.
__host__ __device__ constexpr uint32_t stream_x_unit_bytes(int fmt) {
    return 2u * static_cast<uint32_t>(stream_unit_cols(fmt)) + 16u;
}
constexpr int kStreamMaxLayers = 8;
constexpr int kStreamMaxBatch = 3;  // larger batches run the tiled kernel
// x of a streaming launch by the copy engine: at least this many layers, no copy (one layer's x row)
// above kCopyXMaxCopy bytes, at most kCopyXMaxBytes bytes in all
constexpr int kCopyXMinLayers = 3;
constexpr uint64_t kCopyXMaxCopy = 24 * 1024;
constexpr uint64_t kCopyXMaxBytes = 96 * 1024;
constexpr int kPairsPerRound = kThreads / 4;  // 128 pairs per CTA round
constexpr uint32_t kCtaLayerBytes = 64;     // one entry of the per-CTA layer table in shared memory

// One layer of a streaming launch (host-planned).
struct StreamLayer {
    const uint8_t* vals;   // section bases
    const uint8_t* idx;
    const uint8_t* sz;
    uint32_t vals_pitch, idx_pitch, sz_pitch;
    const __half* x;       // [B][K]
    __half* y;             // [B][N]
    int n, k;
    // Row partition in quads of 4 rows (the last quad of the layer may be short): CTA c < nctas owns
    // q_base quads, plus one more when (c - q_rot) mod nctas < q_rem; its quads follow those of CTA c - 1.
    // q_rot rotates the CTAs that take the extra quads, so that the layers of a launch give their extras
    // to different CTAs and the CTAs' pair counts stay even.
    int nctas, q_base, q_rem, q_rot;
    int cpr;               // units per row (the last one a half unit when a 256-column unit meets K % 256 == 128)
    int full;              // complete units per row
    int dq, dc;            // kPairsPerRound / cpr and kPairsPerRound % cpr: a lane's step in (quad, unit)
    uint32_t xoff;         // shared-memory offset of this layer's x (batch row b at b * xbs + xoff)
};

struct StreamGroup {
    int n_layers;
    int log2g;             // every layer of a launch has this group size
    uint32_t xbs;          // bytes of x per batch row in shared memory: the x of every layer, side by side
    uint32_t part_off;     // shared-memory offset of the unit sums: fp32 [B][4][pstride]
    uint32_t pstride;      // pairs per row slot (>= the pairs of any CTA)
    uint32_t tab_off;      // shared-memory offset of the per-layer table (kStreamMaxLayers + 1 entries)
    // x by the copy engine (launches of several layers, when it fits): the raw x of every layer and batch
    // row, side by side (2 * K bytes each), at xraw_off, and its mbarrier at xbar_off; xraw_off = 0: x is
    // staged with plain loads
    uint32_t xraw_off, xraw_bytes, xbar_off;
    int32_t* status;       // nullable: receives SGEMV_ERR_TIMEOUT if the x copy never completes
    StreamLayer layer[kStreamMaxLayers];
};

// ------------------------------------------------------------------------------------------------
// Device helpers (inline PTX): streaming loads, dependent launch.

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Weights are read exactly once: load them without allocating in L1.
struct U8 {
    uint4 lo, hi;
};
__device__ __forceinline__ U8 ldg_stream_v8(const void* p) {  // p: 32-byte aligned
    U8 v;
    asm volatile("ld.global.nc.L1::no_allocate.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=r"(v.lo.x), "=r"(v.lo.y), "=r"(v.lo.z), "=r"(v.lo.w), "=r"(v.hi.x), "=r"(v.hi.y), "=r"(v.hi.z),
                   "=r"(v.hi.w)
                 : "l"(p));
    return v;
}
__device__ __forceinline__ uint4 ldg_stream_v4(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}
__device__ __forceinline__ uint2 ldg_stream_v2(const void* p) {
    uint2 v;
    asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
    return v;
}
__device__ __forceinline__ uint32_t ldg_stream_u32(const void* p) {
    uint32_t v;
    asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}

// Ask L2 to fetch [p, p + bytes) from HBM (p and bytes multiples of 16). A hint without architectural
// effect: L2 is the point of coherence of global memory, so it can never make a load see stale data.
__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// Programmatic dependent launch: block until the preceding kernel in the stream has completed and
// its memory is visible / allow the next kernel in the stream to be scheduled.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// mbarrier and bulk-copy (TMA) helpers. mbar_wait is bounded: it gives up after kMbarWaitNs of the
// global timer and returns false, so that no kernel can hang on a copy that never lands.
constexpr uint64_t kMbarWaitNs = 200ull * 1000 * 1000;
__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}
// makes initialised barriers visible to the copy engine (async proxy)
__device__ __forceinline__ void mbar_fence_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t done;
    asm volatile("{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(done) : "r"(smem_addr(bar)), "r"(parity) : "memory");
    return done != 0;
}
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 63u) == 0 && global_ns() - t0 > kMbarWaitNs) return false;
    }
}
// bytes (a multiple of 16) from global src to shared dst (both 16-byte aligned), counted on bar's
// transaction count
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(smem_addr(dst)), "l"(src), "r"(bytes), "r"(smem_addr(bar)) : "memory");
}

// Named CTA barriers (id 0 is __syncthreads). n = threads taking part (a multiple of 32).
__device__ __forceinline__ void named_bar_sync(int id, int n) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}
__device__ __forceinline__ void named_bar_arrive(int id, int n) {
    asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// Beam-score step (beam.cu): most input / output beams, and capacity of the candidate key array.
constexpr int kMaxBeam = 64;
constexpr int kMaxCandidates = 16384;

// Device-side information cached per device by the host code.
struct DeviceInfo {
    int sm_count = 0;
    int max_smem_optin = 0;
    // clusters of 2, 4 and 8 CTAs of the split-K kernel that can be resident at once (index log2(size) - 1);
    // without a query (host-only checks) no limit
    int max_clusters[3] = {1 << 30, 1 << 30, 1 << 30};
};
int device_info(DeviceInfo* out);  // host: for the current device

// Split-K for layers with few rows and a long K: clusters of 2, 4 or 8 CTAs share a row range when K
// has at least kSplitMinK columns, the rows alone would leave SMs idle (n * split <= SMs), K has at
// least `split` 1024-column blocks, and all n clusters can be resident at once. Below kSplitMinK a
// layer's few rows stream faster on their own: the cluster barriers and the DSMEM reduction cost more
// than the shorter rows save.
constexpr int kMaxSplit = 8;
constexpr int kSplitMinK = 32768;
constexpr int kMaxPassRows = 256;             // rows of one accumulator pass of the GEMV kernel
constexpr uint32_t kXTileBudget = 96 * 1024;  // bytes of shared memory for its x tile
int split_factor(int n, int k, const DeviceInfo& di);
// host (gemv_sparse.cu): how many clusters of `split` CTAs of the split-K kernel can be resident at once
cudaError_t query_max_clusters(int split, int* out);

// Launch geometry and shared-memory plan of one GEMV (abi.cu); exposed for host-side checks.
int plan_gemv(const sgemv_layout& L, const void* packed, const void* x, int batch, void* y, int32_t* status,
              const DeviceInfo& di, GemvParams* pp, int* grid, uint32_t* smem);

// Plan of one streaming launch over table[0 .. n) (abi.cu); exposed for host-side checks.
int plan_stream(const sgemv_layer* table, int n, int batch, const DeviceInfo& di, StreamGroup* g, int* grid,
                uint32_t* smem);

// Host launchers implemented in gemv_sparse.cu / gemv_sparse14.cu / gemv_dense.cu / pack.cu.
cudaError_t launch_gemv_sparse(int batch, const LayerGroup& g, int grid, uint32_t smem, cudaStream_t s);
cudaError_t launch_gemv_sparse14(int batch, const LayerGroup& g, int grid, uint32_t smem, cudaStream_t s);
cudaError_t launch_gemv_dense(int batch, const LayerGroup& g, int grid, uint32_t smem, cudaStream_t s);
cudaError_t launch_pack(const PackParams& p, int grid, cudaStream_t s);
cudaError_t launch_stream(int format, int batch, const StreamGroup& g, int grid, uint32_t smem, cudaStream_t s);
// one translation unit per (format, group size): gemv_stream{24,14,d}_g{64,128,256}.cu
#define SGEMV_STREAM_LAUNCHER(NAME) \
    cudaError_t NAME(int batch, const StreamGroup& g, int grid, uint32_t smem, cudaStream_t s);
SGEMV_STREAM_LAUNCHER(launch_stream24_g64)
SGEMV_STREAM_LAUNCHER(launch_stream24_g128)
SGEMV_STREAM_LAUNCHER(launch_stream24_g256)
SGEMV_STREAM_LAUNCHER(launch_stream14_g64)
SGEMV_STREAM_LAUNCHER(launch_stream14_g128)
SGEMV_STREAM_LAUNCHER(launch_stream14_g256)
SGEMV_STREAM_LAUNCHER(launch_streamd_g64)
SGEMV_STREAM_LAUNCHER(launch_streamd_g128)
SGEMV_STREAM_LAUNCHER(launch_streamd_g256)
#undef SGEMV_STREAM_LAUNCHER

}  // namespace sgemv
