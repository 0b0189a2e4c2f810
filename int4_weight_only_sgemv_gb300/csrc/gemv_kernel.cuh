// INT4 weight-only GEMV kernels for GB300 (sm_103a): the SparseGemv of the paper "Efficient LLM-based
// Advertising via Model Compression and Parallel Verification" (§3.3 "Revised Kernel") over the 2:4
// "2bit-CSR" format, and the dense INT4 variant ("previous generation Gemv", same section).
//
// Work split (one persistent CTA per SM):
//   * CTA c owns a contiguous, balanced range of output rows (±1 row between CTAs). Its share of the
//     packed layer is three contiguous byte ranges (vals, idx, sz), streamed once from HBM.
//   * One producer warp moves the share into a ring of shared-memory stages with bulk asynchronous
//     copies (cp.async.bulk, completion counted on an mbarrier per stage). A stage holds 4 rows x up to
//     `cs` columns of every section, each row at a padded, bank-conflict-free pitch.
//   * 16 consumer warps take tasks (4 rows x 512 columns) from the stages in a global round robin.
//     Lane (r, j) = (lane / 8, lane % 8) handles 64 columns of row r: 16 bytes of nibbles, 8 bytes of
//     2-bit positions and one {scale, zero} pair.
//   * x is staged once per CTA (per x tile when B*K is too large) into shared memory by the consumer
//     warps, 64 columns per 144-byte chunk, so the 8 column-lanes of a task read 8 different bank
//     groups and the 4 row-lanes of a column broadcast (the paper's conflict-free activation layout and
//     block-level cooperative load, §3.3 "Accelerate Memory Access").
//   * Row partial sums of the 8 column-lanes are combined with warp shuffles, then added into an fp32
//     accumulator per (row, batch) in shared memory; the CTA writes y once at the end.
//
// Per 8 kept elements (one 32-bit word of nibbles, one 16-bit word of positions) and batch row:
//   * dequantisation (§3.3 "Reduce Computational Burden", lop3): one AND-OR per nibble pair gives
//     half2 {1024+q0, 1024+q1} (or 1024+16q for the odd nibbles), one HSUB2 removes 1024+z exactly;
//   * the 2-bit positions of a block become a byte-permute selector with one mask and one integer
//     multiply-add, and one PRMT gathers the two activations of the block from the two 32-bit words
//     that hold its four fp16 activations;
//   * products (q - z) * x are exact in fp32 (mixed-precision FMA, fp16 sources, fp32 accumulate); the
//     group scale is applied once per 64 columns.
// No tensor cores: at batch <= 8 the product is bound by HBM (batch 1-2) or by the integer/FP32 issue
// rate (batch 4-8), not by a dense contraction.
//
// Every mbarrier wait is bounded in time; on expiry the CTA records SGEMV_ERR_TIMEOUT, stops issuing
// copies, lets its copies in flight land and exits.
#pragma once

#include "common.cuh"

namespace sgemv {

// acc + a.lo*b.lo + a.hi*b.hi with fp16 sources and fp32 accumulation (products exact in fp32).
__device__ __forceinline__ float fma_h2_f32(uint32_t a, uint32_t b, float c) {
    float d;
    asm("{\n\t.reg .f16 a0, a1, b0, b1;\n\t.reg .f32 t;\n\t"
        "mov.b32 {a0, a1}, %1;\n\t"
        "mov.b32 {b0, b1}, %2;\n\t"
        "fma.rn.f32.f16 t, a0, b0, %3;\n\t"
        "fma.rn.f32.f16 %0, a1, b1, t;\n\t}"
        : "=f"(d)
        : "r"(a), "r"(b), "f"(c));
    return d;
}

__device__ __forceinline__ uint32_t hsub2_bits(uint32_t a, uint32_t b) {
    __half2 r = __hsub2(*reinterpret_cast<const __half2*>(&a), *reinterpret_cast<const __half2*>(&b));
    return *reinterpret_cast<const uint32_t*>(&r);
}

__device__ __forceinline__ uint32_t half2_splat_bits(float v) {
    __half2 h = __float2half2_rn(v);
    return *reinterpret_cast<const uint32_t*>(&h);
}

// Nibble pairs of one word as half2 codes minus the zero point:
//   d[0] = {q(slot0), q(slot4)} - z,   d[1] = 16*({q(slot1), q(slot5)} - z),
//   d[2] = {q(slot2), q(slot6)} - z,   d[3] = 16*({q(slot3), q(slot7)} - z).
// (1024 + q and 1024 + 16q are exact fp16 values: the mantissa of 1024 has unit spacing.)
__device__ __forceinline__ void dequant_word(uint32_t w, uint32_t zA, uint32_t zB, uint32_t (&d)[4]) {
    const uint32_t magic = 0x64006400u;
    const uint32_t hi = w >> 8;
    d[0] = hsub2_bits((w & 0x000F000Fu) | magic, zA);
    d[1] = hsub2_bits((w & 0x00F000F0u) | magic, zB);
    d[2] = hsub2_bits((hi & 0x000F000Fu) | magic, zA);
    d[3] = hsub2_bits((hi & 0x00F000F0u) | magic, zB);
}

// One lane of a sparse task: 64 dense columns (32 kept) of one row, for every batch row.
//   v   : 4 words of nibbles (blocks 16 of the chunk), ix: 4 u16 words of positions,
//   szw : {s, z}, xp: the chunk's activations in shared memory (batch row 0), xbs: batch stride.
template <int B>
__device__ __forceinline__ void sparse_lane(const uint4 v, const uint2 ix, const uint32_t szw,
                                            const uint8_t* xp, const uint32_t xbs, float (&part)[B]) {
    const float s = __half2float(__ushort_as_half(static_cast<unsigned short>(szw & 0xFFFFu)));
    const float zf = __half2float(__ushort_as_half(static_cast<unsigned short>(szw >> 16)));
    const uint32_t zA = half2_splat_bits(1024.0f + zf);
    const uint32_t zB = half2_splat_bits(1024.0f + 16.0f * zf);
    float accA[B], accB[B];
#pragma unroll
    for (int b = 0; b < B; ++b) accA[b] = accB[b] = 0.0f;
    const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
    const uint32_t i2[2] = {ix.x, ix.y};
#pragma unroll
    for (int u = 0; u < 2; ++u) {
        // i2[u] holds the positions of vals words 2u (low 16 bits) and 2u+1 (high 16 bits).
        // For block t: byte 0/1 of m = p0/p1 of word 2u, byte 2/3 = p0/p1 of word 2u+1.
        // Selector for positions (p0, p1): nibbles (2p0, 2p0+1, 2p1, 2p1+1) = Q*0x22 + 0x1010 with
        // Q = p0 + 256*p1; the high-half selector is taken from the upper 32 bits of a 64-bit product.
        uint32_t S[2][4];
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            const uint32_t m = (i2[u] >> (2 * t)) & 0x03030303u;
            S[0][t] = m * 0x22u + 0x1010u;
            S[1][t] = __umulhi(m, 0x220000u) + 0x1010u;
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            uint32_t d[4];
            dequant_word(w4[2 * u + h], zA, zB, d);
#pragma unroll
            for (int b = 0; b < B; ++b) {
                const uint8_t* xw = xp + b * xbs + 32 * (2 * u + h);
                const uint4 xa = *reinterpret_cast<const uint4*>(xw);
                const uint4 xb = *reinterpret_cast<const uint4*>(xw + 16);
                const uint32_t xs0 = __byte_perm(xa.x, xa.y, S[h][0]);
                const uint32_t xs1 = __byte_perm(xa.z, xa.w, S[h][1]);
                const uint32_t xs2 = __byte_perm(xb.x, xb.y, S[h][2]);
                const uint32_t xs3 = __byte_perm(xb.z, xb.w, S[h][3]);
                accA[b] = fma_h2_f32(d[0], xs0, accA[b]);
                accB[b] = fma_h2_f32(d[1], xs1, accB[b]);
                accA[b] = fma_h2_f32(d[2], xs2, accA[b]);
                accB[b] = fma_h2_f32(d[3], xs3, accB[b]);
            }
        }
    }
#pragma unroll
    for (int b = 0; b < B; ++b) part[b] = s * fmaf(accB[b], 0.0625f, accA[b]);
}

// One lane of a dense task: 64 columns of one row. va = columns 0..31, vb = columns 32..63.
template <int B>
__device__ __forceinline__ void dense_lane(const uint4 va, const uint4 vb, const uint32_t szw,
                                           const uint8_t* xp, const uint32_t xbs, float (&part)[B]) {
    const float s = __half2float(__ushort_as_half(static_cast<unsigned short>(szw & 0xFFFFu)));
    const float zf = __half2float(__ushort_as_half(static_cast<unsigned short>(szw >> 16)));
    const uint32_t zA = half2_splat_bits(1024.0f + zf);
    const uint32_t zB = half2_splat_bits(1024.0f + 16.0f * zf);
    float accA[B], accB[B];
#pragma unroll
    for (int b = 0; b < B; ++b) accA[b] = accB[b] = 0.0f;
    const uint32_t w8[8] = {va.x, va.y, va.z, va.w, vb.x, vb.y, vb.z, vb.w};
#pragma unroll
    for (int w = 0; w < 8; ++w) {
        // word w: columns 8w..8w+7; d[0] = cols {0,1}, d[1] = 16*{2,3}, d[2] = {4,5}, d[3] = 16*{6,7}
        uint32_t d[4];
        dequant_word(w8[w], zA, zB, d);
#pragma unroll
        for (int b = 0; b < B; ++b) {
            const uint4 xa = *reinterpret_cast<const uint4*>(xp + b * xbs + 16 * w);
            accA[b] = fma_h2_f32(d[0], xa.x, accA[b]);
            accB[b] = fma_h2_f32(d[1], xa.y, accB[b]);
            accA[b] = fma_h2_f32(d[2], xa.z, accA[b]);
            accB[b] = fma_h2_f32(d[3], xa.w, accB[b]);
        }
    }
#pragma unroll
    for (int b = 0; b < B; ++b) part[b] = s * fmaf(accB[b], 0.0625f, accA[b]);
}

// Geometry of one pipeline stage.
struct Stage {
    int row0;   // first row, relative to the CTA's first row
    int nrows;  // 1..4
    int col0;   // first column (absolute)
    int ncols;  // columns in this stage (multiple of 128)
};

// Walks the stage sequence of one CTA in the order the producer fills the ring:
// for each pass of rows, for each x tile, for each 4-row quad, for each column stage.
struct StageWalker {
    int nrows_cta, k, cs, xt, pass_rows;
    int pass, tile, quad, cstage;
    int npass, ntile;

    __host__ __device__ void init(int nrows, const GemvParams& p) {
        nrows_cta = nrows;
        k = p.k;
        cs = p.cs;
        xt = p.xt;
        pass_rows = p.pass_rows;
        npass = (nrows + pass_rows - 1) / pass_rows;
        ntile = (k + xt - 1) / xt;
        pass = tile = quad = cstage = 0;
    }
    __host__ __device__ int pass_row0() const { return pass * pass_rows; }
    __host__ __device__ int pass_nrows() const { return min(pass_rows, nrows_cta - pass_row0()); }
    __host__ __device__ int nquads() const { return (pass_nrows() + 3) / 4; }
    __host__ __device__ int tile_col0() const { return tile * xt; }
    __host__ __device__ int tile_ncols() const { return min(xt, k - tile_col0()); }
    __host__ __device__ int ncstages() const { return (tile_ncols() + cs - 1) / cs; }
    __host__ __device__ Stage stage() const {
        Stage s;
        s.row0 = pass_row0() + 4 * quad;
        s.nrows = min(4, pass_nrows() - 4 * quad);
        s.col0 = tile_col0() + cstage * cs;
        s.ncols = min(cs, tile_ncols() - cstage * cs);
        return s;
    }
};

template <int FMT>
__host__ __device__ __forceinline__ uint32_t stage_tx_bytes(const Stage& s, int log2g) {
    const uint32_t szb = ((static_cast<uint32_t>(s.ncols) * 4u >> log2g) + 15u) & ~15u;
    if (FMT == SGEMV_FMT_SPARSE24)
        return static_cast<uint32_t>(s.nrows) * (s.ncols / 4 + s.ncols / 8 + szb);
    return static_cast<uint32_t>(s.nrows) * (s.ncols / 2 + szb);
}

template <int FMT, int B>
__global__ void __launch_bounds__(kThreads, 1) gemv_kernel(const GemvParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    constexpr bool kSparse = (FMT == SGEMV_FMT_SPARSE24);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int cta = blockIdx.x;
    const int row_begin = cta * p.rows_base + min(cta, p.rows_rem);
    const int nrows_cta = p.rows_base + (cta < p.rows_rem ? 1 : 0);
    const int nst = p.nstage;
    const uint32_t bar0 = smem_addr(smem + p.sm_bar);  // full[i] = bar0 + 8i, empty[i] = bar0 + 8(nst+i)
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + p.sm_bar + 16 * nst);

    if (threadIdx.x == 0) {
        for (int i = 0; i < nst; ++i) {
            mbar_init(bar0 + 8 * i, 1);
            mbar_init(bar0 + 8 * (nst + i), kConsumerWarps);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    // The next kernel in the stream may be scheduled now; it reads its own inputs only after this
    // grid has completed (its own griddepcontrol.wait).
    pdl_launch_dependents();
    if (nrows_cta <= 0) return;

    StageWalker sw;
    sw.init(nrows_cta, p);

    if (warp == kConsumerWarps) {
        // ------------------------------------------------------------------ producer warp
        // The packed weights do not depend on the previous kernel: start streaming immediately.
        int sigma = 0;
        bool ok = true;
        for (sw.pass = 0; ok && sw.pass < sw.npass; ++sw.pass)
            for (sw.tile = 0; ok && sw.tile < sw.ntile; ++sw.tile)
                for (sw.quad = 0; ok && sw.quad < sw.nquads(); ++sw.quad)
                    for (sw.cstage = 0; ok && sw.cstage < sw.ncstages(); ++sw.cstage, ++sigma) {
                        const int slot = sigma % nst;
                        const int use = sigma / nst;
                        if (use > 0 && !mbar_wait_bounded(bar0 + 8 * (nst + slot), (use - 1) & 1, abort_flag,
                                                          p.status)) {
                            ok = false;
                            break;
                        }
                        const Stage st = sw.stage();
                        const uint32_t full = bar0 + 8 * slot;
                        if (lane == 0) mbar_arrive_expect_tx(full, stage_tx_bytes<FMT>(st, p.log2g));
                        __syncwarp();
                        const uint32_t sbase = smem_addr(smem) + slot * p.st_bytes;
                        constexpr int kSec = kSparse ? 3 : 2;
                        if (lane < st.nrows * kSec) {
                            const int i = lane / kSec;
                            const int sec = lane % kSec;
                            const size_t grow = static_cast<size_t>(row_begin + st.row0 + i);
                            if (sec == 0) {
                                const uint32_t vb = kSparse ? st.ncols / 4 : st.ncols / 2;
                                const uint32_t vo = kSparse ? st.col0 / 4 : st.col0 / 2;
                                bulk_g2s(sbase + i * p.st_vals_pitch, p.vals + grow * p.vals_pitch + vo, vb, full);
                            } else if (kSparse && sec == 1) {
                                bulk_g2s(sbase + p.st_idx_off + i * p.st_idx_pitch,
                                         p.idx + grow * p.idx_pitch + st.col0 / 8, st.ncols / 8, full);
                            } else {
                                const uint32_t szb = ((static_cast<uint32_t>(st.ncols) * 4u >> p.log2g) + 15u) & ~15u;
                                const uint32_t szo = (static_cast<uint32_t>(st.col0) * 4u) >> p.log2g;
                                bulk_g2s(sbase + p.st_sz_off + i * p.st_sz_pitch, p.sz + grow * p.sz_pitch + szo,
                                         szb, full);
                            }
                        }
                    }
        // Let every copy this warp issued land before the CTA can exit (matters only after an abort).
        __syncwarp();
        if (lane == 0) {
            volatile int never = 0;
            for (int s = max(0, sigma - nst); s < sigma; ++s)
                mbar_wait_bounded(bar0 + 8 * (s % nst), (s / nst) & 1, &never, nullptr);
        }
        return;
    }

    // ---------------------------------------------------------------------- consumer warps
    const int ctid = threadIdx.x;  // 0 .. 16*32-1
    float* acc = reinterpret_cast<float*>(smem + p.sm_acc);
    uint8_t* xs = smem + p.sm_x;
    const int r = lane >> 3;  // row of the task handled by this lane
    const int j = lane & 7;   // 64-column chunk of the task handled by this lane
    int sigma = 0;
    int task_base = 0;
    bool aborted = false;
    bool waited_pdl = false;

    for (sw.pass = 0; sw.pass < sw.npass; ++sw.pass) {
        const int prow0 = sw.pass_row0();
        const int prows = sw.pass_nrows();
        for (int i = ctid; i < B * p.pass_rows; i += kConsumerWarps * 32) acc[i] = 0.0f;
        for (sw.tile = 0; sw.tile < sw.ntile; ++sw.tile) {
            const int tc0 = sw.tile_col0();
            const int tcols = sw.tile_ncols();
            consumer_bar();  // previous tile's x no longer read; accumulators zeroed
            if (!waited_pdl) {
                pdl_wait();  // x may be the output of the previous kernel in the stream
                waited_pdl = true;
            }
            {
                const int units = tcols / 8;  // 16-byte units per batch row
                for (int u = ctid; u < B * units; u += kConsumerWarps * 32) {
                    const int b = u / units;
                    const int v = u - b * units;
                    const uint4 val = __ldg(reinterpret_cast<const uint4*>(p.x + static_cast<size_t>(b) * p.k + tc0) + v);
                    *reinterpret_cast<uint4*>(xs + b * p.x_b_stride + (v >> 3) * kXChunkBytes + (v & 7) * 16) = val;
                }
            }
            consumer_bar();  // x tile visible to every consumer warp
            for (sw.quad = 0; sw.quad < sw.nquads(); ++sw.quad)
                for (sw.cstage = 0; sw.cstage < sw.ncstages(); ++sw.cstage, ++sigma) {
                    const Stage st = sw.stage();
                    const int slot = sigma % nst;
                    const int ntasks = (st.ncols + kSlabCols - 1) / kSlabCols;
                    if (!aborted && !mbar_wait_bounded(bar0 + 8 * slot, (sigma / nst) & 1, abort_flag, p.status))
                        aborted = true;
                    const uint8_t* sb = smem + slot * p.st_bytes;
                    // tasks t of this stage with (task_base + t) % 16 == warp
                    int t = warp - (task_base % kConsumerWarps);
                    if (t < 0) t += kConsumerWarps;
                    for (; !aborted && t < ntasks; t += kConsumerWarps) {
                        const int ccol = t * kSlabCols + 64 * j;  // column within the stage
                        const bool valid = (r < st.nrows) && (ccol < st.ncols);
                        float part[B];
#pragma unroll
                        for (int b = 0; b < B; ++b) part[b] = 0.0f;
                        if (valid) {
                            const uint8_t* xp = xs + ((st.col0 - tc0 + ccol) >> 6) * kXChunkBytes;
                            const uint32_t szw = *reinterpret_cast<const uint32_t*>(
                                sb + p.st_sz_off + r * p.st_sz_pitch + ((static_cast<uint32_t>(ccol) >> p.log2g) << 2));
                            if (kSparse) {
                                const uint4 v = *reinterpret_cast<const uint4*>(sb + r * p.st_vals_pitch + ccol / 4);
                                const uint2 ix = *reinterpret_cast<const uint2*>(sb + p.st_idx_off + r * p.st_idx_pitch + ccol / 8);
                                sparse_lane<B>(v, ix, szw, xp, p.x_b_stride, part);
                            } else {
                                // the two 16-byte halves are read in a lane-dependent order so that the
                                // 8 column-lanes of a row hit 8 disjoint bank groups
                                const uint8_t* vp = sb + r * p.st_vals_pitch + ccol / 2;
                                const int hsw = (j >> 2) & 1;
                                const uint4 first = *reinterpret_cast<const uint4*>(vp + 16 * hsw);
                                const uint4 second = *reinterpret_cast<const uint4*>(vp + 16 * (1 - hsw));
                                uint4 va, vb;
                                va.x = hsw ? second.x : first.x;
                                va.y = hsw ? second.y : first.y;
                                va.z = hsw ? second.z : first.z;
                                va.w = hsw ? second.w : first.w;
                                vb.x = hsw ? first.x : second.x;
                                vb.y = hsw ? first.y : second.y;
                                vb.z = hsw ? first.z : second.z;
                                vb.w = hsw ? first.w : second.w;
                                dense_lane<B>(va, vb, szw, xp, p.x_b_stride, part);
                            }
                        }
#pragma unroll
                        for (int b = 0; b < B; ++b) {
                            float v = part[b];
                            v += __shfl_xor_sync(0xFFFFFFFFu, v, 1);
                            v += __shfl_xor_sync(0xFFFFFFFFu, v, 2);
                            v += __shfl_xor_sync(0xFFFFFFFFu, v, 4);
                            part[b] = v;
                        }
                        if (j == 0 && r < st.nrows) {
#pragma unroll
                            for (int b = 0; b < B; ++b) atomicAdd(acc + b * p.pass_rows + st.row0 - prow0 + r, part[b]);
                        }
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar0 + 8 * (nst + slot));
                    task_base += ntasks;
                }
        }
        consumer_bar();  // all partial sums of this pass are in `acc`
        if (!aborted && !*abort_flag) {
            for (int i = ctid; i < B * prows; i += kConsumerWarps * 32) {
                const int b = i / prows;
                const int rr = i - b * prows;
                p.y[static_cast<size_t>(b) * p.n + row_begin + prow0 + rr] = __float2half_rn(acc[b * p.pass_rows + rr]);
            }
        }
        consumer_bar();  // y written before the accumulators are cleared for the next pass
    }
}

}  // namespace sgemv
