// INT4 weight-only GEMV kernels for GB300 (sm_103a): the SparseGemv of the paper "Efficient LLM-based
// Advertising via Model Compression and Parallel Verification" (§3.3 "Revised Kernel") over the 2:4
// "2bit-CSR" format, and the dense INT4 variant ("previous generation Gemv", same section).
//
// Work split (one persistent CTA of 16 warps per SM):
//   * CTA c owns a contiguous, balanced range of output rows (±1 row between CTAs); its share of the
//     packed layer is read exactly once from HBM.
//   * The CTA's rows are cut into tasks of 4 rows x 1024 columns; warp w takes a contiguous run of
//     tasks (runs differ by at most one task). Lane (r, j) = (lane / 8, lane % 8) handles chunks j and
//     j + 8 (64 columns each) of row r, so the 8 column-lanes of a row read 128 contiguous bytes of
//     nibbles per chunk and every load instruction of a warp covers 4 whole 128-byte lines.
//   * The weights go straight from HBM into registers with 128-bit streaming loads; each warp keeps
//     the next 1-3 tasks (fewer at larger batch) in flight while it computes, and issues its first loads before the
//     dependent-launch wait, since the weights never depend on the previous kernel.
//   * x is staged once per CTA (per x tile when B*K is too large) into shared memory by all warps,
//     64 columns per 144-byte chunk: the 8 column-lanes of a task read 8 different bank groups and
//     the 4 row-lanes of a column broadcast (the paper's conflict-free activation layout and
//     block-level cooperative load, §3.3 "Accelerate Memory Access").
//   * A lane accumulates its row's partial sum in registers over consecutive tasks of the same 4 rows;
//     when the rows change, the 8 column-lanes combine with warp shuffles and add into an fp32
//     accumulator per (row, batch) in shared memory. The CTA writes y once at the end.
//
// Per 8 kept elements (one 32-bit word of nibbles, one 16-bit word of positions) and batch row:
//   * dequantisation (§3.3 "Reduce Computational Burden", lop3): one AND-OR per nibble pair gives
//     half2 {1024+q0, 1024+q1} (or 1024+16q for the odd nibbles), one HSUB2 removes 1024+z exactly;
//   * the 2-bit positions of a block become a byte-permute selector: one mask, and one 32x32->64-bit
//     multiply-add yields the selectors of the same block in two consecutive words; one PRMT gathers
//     the two activations of the block from the two 32-bit words holding its four fp16 activations;
//   * products (q - z) * x are exact in fp32 (mixed-precision FMA, fp16 sources, fp32 accumulate); the
//     group scale is applied once per 64 columns.
// The integer operations are written as PTX (prmt, lop3, mad.wide) so that each is one instruction.
// No tensor cores: at batch <= 8 the product is bound by HBM (batch 1-2) or by the integer/FP32 issue
// rate (batch 4-8), not by a dense contraction. There are no waits on other threads other than
// __syncthreads, so the kernel cannot hang.
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

// Byte permute with a selector whose nibbles never set their sign-replicate bit (plain PRMT).
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

// (a & mask) | c in one LOP3.
__device__ __forceinline__ uint32_t and_or(uint32_t a, uint32_t mask, uint32_t c) {
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(mask), "r"(c));
    return d;
}

// Gather selectors for two blocks: m holds Q0 = p0 + 256*p1 of one block in its low 16 bits and Q1 of
// another block in its high 16 bits. Selector for (p0, p1) = nibbles (2p0, 2p0+1, 2p1, 2p1+1) =
// Q*0x22 + 0x1010. One 64-bit multiply-add by 0x220022 gives Q0*0x22 in bits 0..15 and Q1*0x22 in bits
// 32..47 (the cross term (Q0+Q1)*0x22 stays inside bits 16..31: no carry, since it is < 2^16).
__device__ __forceinline__ void selector_pair(uint32_t m, uint32_t& s0, uint32_t& s1) {
    asm("{\n\t.reg .b64 r;\n\t"
        "mad.wide.u32 r, %2, 0x220022, 0x0000101000001010;\n\t"
        "mov.b64 {%0, %1}, r;\n\t}"
        : "=r"(s0), "=r"(s1)
        : "r"(m));
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
    d[0] = hsub2_bits(and_or(w, 0x000F000Fu, magic), zA);
    d[1] = hsub2_bits(and_or(w, 0x00F000F0u, magic), zB);
    d[2] = hsub2_bits(and_or(hi, 0x000F000Fu, magic), zA);
    d[3] = hsub2_bits(and_or(hi, 0x00F000F0u, magic), zB);
}

struct GroupParams {
    float s;
    uint32_t zA, zB;
};

__device__ __forceinline__ GroupParams group_params(uint32_t szw) {
    GroupParams g;
    g.s = __half2float(__ushort_as_half(static_cast<unsigned short>(szw & 0xFFFFu)));
    const float zf = __half2float(__ushort_as_half(static_cast<unsigned short>(szw >> 16)));
    g.zA = half2_splat_bits(1024.0f + zf);
    g.zB = half2_splat_bits(1024.0f + 16.0f * zf);
    return g;
}

// One 64-column chunk (32 kept) of one row for every batch row, added into part[b].
//   v: 4 words of nibbles, ix: 4 u16 words of positions, xp: the chunk's activations (batch row 0).
template <int B>
__device__ __forceinline__ void sparse_chunk(const uint4 v, const uint2 ix, const uint32_t szw,
                                             const uint8_t* xp, const uint32_t xbs, float (&part)[B]) {
    const GroupParams gp = group_params(szw);
    float accA[B], accB[B];
#pragma unroll
    for (int b = 0; b < B; ++b) accA[b] = accB[b] = 0.0f;
    const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
    const uint32_t i2[2] = {ix.x, ix.y};
#pragma unroll
    for (int u = 0; u < 2; ++u) {
        // i2[u] holds the positions of vals words 2u (low 16 bits) and 2u+1 (high 16 bits); for block
        // t, bytes 0/1 of m are p0/p1 of word 2u and bytes 2/3 are p0/p1 of word 2u+1.
        uint32_t S[2][4];
#pragma unroll
        for (int t = 0; t < 4; ++t) selector_pair((i2[u] >> (2 * t)) & 0x03030303u, S[0][t], S[1][t]);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            uint32_t d[4];
            dequant_word(w4[2 * u + h], gp.zA, gp.zB, d);
#pragma unroll
            for (int b = 0; b < B; ++b) {
                const uint8_t* xw = xp + b * xbs + 32 * (2 * u + h);
                const uint4 xa = *reinterpret_cast<const uint4*>(xw);
                const uint4 xb = *reinterpret_cast<const uint4*>(xw + 16);
                accA[b] = fma_h2_f32(d[0], prmt(xa.x, xa.y, S[h][0]), accA[b]);
                accB[b] = fma_h2_f32(d[1], prmt(xa.z, xa.w, S[h][1]), accB[b]);
                accA[b] = fma_h2_f32(d[2], prmt(xb.x, xb.y, S[h][2]), accA[b]);
                accB[b] = fma_h2_f32(d[3], prmt(xb.z, xb.w, S[h][3]), accB[b]);
            }
        }
    }
#pragma unroll
    for (int b = 0; b < B; ++b) part[b] = fmaf(gp.s, fmaf(accB[b], 0.0625f, accA[b]), part[b]);
}

// One 64-column chunk of a dense row. va = columns 0..31, vb = columns 32..63.
template <int B>
__device__ __forceinline__ void dense_chunk(const uint4 va, const uint4 vb, const uint32_t szw,
                                            const uint8_t* xp, const uint32_t xbs, float (&part)[B]) {
    const GroupParams gp = group_params(szw);
    float accA[B], accB[B];
#pragma unroll
    for (int b = 0; b < B; ++b) accA[b] = accB[b] = 0.0f;
    const uint32_t w8[8] = {va.x, va.y, va.z, va.w, vb.x, vb.y, vb.z, vb.w};
#pragma unroll
    for (int w = 0; w < 8; ++w) {
        // word w: columns 8w..8w+7; d[0] = cols {0,1}, d[1] = 16*{2,3}, d[2] = {4,5}, d[3] = 16*{6,7}
        uint32_t d[4];
        dequant_word(w8[w], gp.zA, gp.zB, d);
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
    for (int b = 0; b < B; ++b) part[b] = fmaf(gp.s, fmaf(accB[b], 0.0625f, accA[b]), part[b]);
}

// Registers holding the weights of one task for one lane: two chunks of 64 columns.
template <int FMT>
struct TaskRegs;

template <>
struct TaskRegs<SGEMV_FMT_SPARSE24> {
    uint4 v[2];      // nibbles (16 bytes per chunk)
    uint2 ix[2];     // positions (8 bytes per chunk)
    uint32_t sz[2];  // {s, z} of each chunk's group
};

template <>
struct TaskRegs<SGEMV_FMT_DENSE> {
    uint4 v[2][2];   // nibbles (32 bytes per chunk)
    uint32_t sz[2];
};

// Geometry of the tasks of one (pass, x tile): task t -> (quad t / nblk, column block t % nblk).
struct TaskSpace {
    int prow0, prows;  // pass rows, relative to the CTA's first row
    int tc0, tcols;    // x tile columns
    int nblk;          // 1024-column blocks in the tile
    int ntasks;
    __host__ __device__ void set(int prow0_, int prows_, int tc0_, int tcols_) {
        prow0 = prow0_;
        prows = prows_;
        tc0 = tc0_;
        tcols = tcols_;
        nblk = (tcols + kTaskCols - 1) / kTaskCols;
        ntasks = ((prows + kRowsPerTask - 1) / kRowsPerTask) * nblk;
    }
};

// Walks tasks in order without divisions: (quad, blk) advance like an odometer.
struct TaskCursor {
    int quad, blk;
    __host__ __device__ void start(const TaskSpace& ts, int t) {
        quad = t / ts.nblk;
        blk = t - quad * ts.nblk;
    }
    __host__ __device__ void next(const TaskSpace& ts) {
        if (++blk == ts.nblk) {
            blk = 0;
            ++quad;
        }
    }
    // row within the pass handled by row-lane r (-1 if beyond the pass)
    __host__ __device__ int row(int r, const TaskSpace& ts) const {
        const int rr = quad * kRowsPerTask + r;
        return rr < ts.prows ? rr : -1;
    }
    // column within the tile of chunk c (0 or 1) of column-lane j (-1 if beyond the tile)
    __host__ __device__ int col(int j, int c, const TaskSpace& ts) const {
        const int cc = blk * kTaskCols + c * (8 * kChunkCols) + j * kChunkCols;
        return cc < ts.tcols ? cc : -1;
    }
};

// Warp w's contiguous run of tasks [begin, end).
__host__ __device__ __forceinline__ void warp_run(int ntasks, int w, int& begin, int& end) {
    begin = static_cast<int>((static_cast<long long>(ntasks) * w) / kWarps);
    end = static_cast<int>((static_cast<long long>(ntasks) * (w + 1)) / kWarps);
}

// The load side of a warp: the next task to load and the lane's pointers into its row's sections,
// positioned at column tc0 + 64j (chunk 0 of block 0), so a task only adds its block offset.
struct LoadState {
    TaskCursor cur;
    int rows_quad;  // quad the pointers below belong to
    bool row_ok;
    const uint8_t* vp;  // vals of (row, tc0 + 64j)
    const uint8_t* ip;  // idx
    const uint8_t* sp;  // sz row start
};

// A task is full when all 4 of its rows exist and it covers 1024 columns of the tile (warp-uniform).
__host__ __device__ __forceinline__ bool task_full(const TaskCursor& c, const TaskSpace& ts) {
    return (c.quad + 1) * kRowsPerTask <= ts.prows && (c.blk + 1) * kTaskCols <= ts.tcols;
}

template <int FMT>
__device__ __forceinline__ void load_next(const GemvParams& p, const TaskSpace& ts, int row_begin, int r, int j,
                                          LoadState& ls, TaskRegs<FMT>& tr) {
    constexpr bool kSparse = (FMT == SGEMV_FMT_SPARSE24);
    if (ls.cur.quad != ls.rows_quad) {  // warp-uniform: new rows, new row pointers
        ls.rows_quad = ls.cur.quad;
        const int rr = ls.cur.row(r, ts);
        ls.row_ok = rr >= 0;
        const size_t grow = static_cast<size_t>(row_begin + ts.prow0 + (ls.row_ok ? rr : 0));
        const uint32_t c0 = static_cast<uint32_t>(ts.tc0 + j * kChunkCols);
        ls.vp = p.vals + grow * p.vals_pitch + (kSparse ? c0 / 4 : c0 / 2);
        ls.ip = p.idx + grow * p.idx_pitch + c0 / 8;
        ls.sp = p.sz + grow * p.sz_pitch;
    }
    const uint32_t bcol = static_cast<uint32_t>(ls.cur.blk * kTaskCols);  // block offset within the tile
    const uint32_t gcol0 = static_cast<uint32_t>(ts.tc0 + j * kChunkCols) + bcol;
    if (task_full(ls.cur, ts)) {
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            const uint32_t coff = bcol + c * (8 * kChunkCols);
            tr.sz[c] = ldg_stream_u32(ls.sp + (((gcol0 + c * (8 * kChunkCols)) >> p.log2g) << 2));
            if constexpr (kSparse) {
                tr.v[c] = ldg_stream_v4(ls.vp + coff / 4);
                tr.ix[c] = ldg_stream_v2(ls.ip + coff / 8);
            } else {
                tr.v[c][0] = ldg_stream_v4(ls.vp + coff / 2);
                tr.v[c][1] = ldg_stream_v4(ls.vp + coff / 2 + 16);
            }
        }
    } else {
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            const int cc = ls.cur.col(j, c, ts);
            tr.sz[c] = 0;
            if constexpr (kSparse) {
                tr.v[c] = make_uint4(0, 0, 0, 0);
                tr.ix[c] = make_uint2(0, 0);
            } else {
                tr.v[c][0] = tr.v[c][1] = make_uint4(0, 0, 0, 0);
            }
            if (!ls.row_ok || cc < 0) continue;
            const uint32_t coff = bcol + c * (8 * kChunkCols);
            tr.sz[c] = ldg_stream_u32(ls.sp + (((gcol0 + c * (8 * kChunkCols)) >> p.log2g) << 2));
            if constexpr (kSparse) {
                tr.v[c] = ldg_stream_v4(ls.vp + coff / 4);
                tr.ix[c] = ldg_stream_v2(ls.ip + coff / 8);
            } else {
                tr.v[c][0] = ldg_stream_v4(ls.vp + coff / 2);
                tr.v[c][1] = ldg_stream_v4(ls.vp + coff / 2 + 16);
            }
        }
    }
    ls.cur.next(ts);
}

template <int FMT, int B>
__device__ __forceinline__ void compute_task(const GemvParams& p, const TaskSpace& ts, const uint8_t* xtile,
                                             const TaskCursor& tc, int r, int j, const TaskRegs<FMT>& tr,
                                             float (&part)[B]) {
    const uint8_t* xp0 = xtile + (tc.blk * (kTaskCols / kChunkCols) + j) * kXChunkBytes;
    if (task_full(tc, ts)) {
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            const uint8_t* xp = xp0 + c * 8 * kXChunkBytes;
            if constexpr (FMT == SGEMV_FMT_SPARSE24)
                sparse_chunk<B>(tr.v[c], tr.ix[c], tr.sz[c], xp, p.x_b_stride, part);
            else
                dense_chunk<B>(tr.v[c][0], tr.v[c][1], tr.sz[c], xp, p.x_b_stride, part);
        }
        return;
    }
    if (tc.row(r, ts) < 0) return;
#pragma unroll
    for (int c = 0; c < 2; ++c) {
        if (tc.col(j, c, ts) < 0) continue;
        const uint8_t* xp = xp0 + c * 8 * kXChunkBytes;
        if constexpr (FMT == SGEMV_FMT_SPARSE24)
            sparse_chunk<B>(tr.v[c], tr.ix[c], tr.sz[c], xp, p.x_b_stride, part);
        else
            dense_chunk<B>(tr.v[c][0], tr.v[c][1], tr.sz[c], xp, p.x_b_stride, part);
    }
}

// Combine the 8 column-lanes of each row and add the row sums into the shared accumulators.
template <int B>
__device__ __forceinline__ void flush_rows(float* acc, int pass_rows, int row, int j, float (&part)[B]) {
#pragma unroll
    for (int b = 0; b < B; ++b) {
        float v = part[b];
        v += __shfl_xor_sync(0xFFFFFFFFu, v, 1);
        v += __shfl_xor_sync(0xFFFFFFFFu, v, 2);
        v += __shfl_xor_sync(0xFFFFFFFFu, v, 4);
        if (j == 0 && row >= 0) atomicAdd(acc + b * pass_rows + row, v);
        part[b] = 0.0f;
    }
}

template <int FMT, int B>
__global__ void __launch_bounds__(kThreads, 1) gemv_kernel(const GemvParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    constexpr int kPrefetch = prefetch_depth<B>();
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int r = lane >> 3;  // row of a task handled by this lane
    const int j = lane & 7;   // chunk column of a task handled by this lane
    const int cta = blockIdx.x;
    const int row_begin = cta * p.rows_base + min(cta, p.rows_rem);
    const int nrows_cta = p.rows_base + (cta < p.rows_rem ? 1 : 0);
    // The next kernel in the stream may be scheduled now; it reads its own inputs only after this
    // grid has completed (its own griddepcontrol.wait).
    pdl_launch_dependents();
    if (nrows_cta <= 0) return;

    float* acc = reinterpret_cast<float*>(smem + p.sm_acc);
    uint8_t* xs = smem + p.sm_x;
    const int ntile = (p.k + p.xt - 1) / p.xt;
    const int npass = (nrows_cta + p.pass_rows - 1) / p.pass_rows;
    bool waited_pdl = false;

    for (int pass = 0; pass < npass; ++pass) {
        const int prow0 = pass * p.pass_rows;
        const int prows = min(p.pass_rows, nrows_cta - prow0);
        for (int tile = 0; tile < ntile; ++tile) {
            TaskSpace ts;
            ts.set(prow0, prows, tile * p.xt, min(p.xt, p.k - tile * p.xt));
            int t_begin, t_end;
            warp_run(ts.ntasks, warp, t_begin, t_end);
            if (!waited_pdl) {
                pdl_wait();  // x may be the output of the previous kernel in the stream
                waited_pdl = true;
            }
            // x first (every warp needs it before any product), then the weights: the x round trip to
            // L2 overlaps the weight loads instead of queueing behind them.
            const int units = ts.tcols / 8;  // 16-byte units of x per batch row
            const uint4* xg = reinterpret_cast<const uint4*>(p.x + ts.tc0);
            uint4 xr[kXStageRegs];
#pragma unroll
            for (int q = 0; q < kXStageRegs; ++q) {
                const int u = threadIdx.x + q * kThreads;  // unit u: batch row u / units (B*units <= bound)
                xr[q] = make_uint4(0, 0, 0, 0);
                if (u < B * units) {
                    const int b = (B == 1) ? 0 : u / units;
                    xr[q] = __ldg(xg + static_cast<size_t>(b) * (p.k / 8) + (u - b * units));
                }
            }
            LoadState ls;
            ls.cur.start(ts, t_begin);
            ls.rows_quad = -1;
            TaskRegs<FMT> buf[kPrefetch];
#pragma unroll
            for (int q = 0; q < kPrefetch; ++q)
                if (t_begin + q < t_end) load_next<FMT>(p, ts, row_begin, r, j, ls, buf[q]);
            __syncthreads();  // the previous tile's x and the previous pass's accumulators are no longer read
            if (tile == 0)
                for (int i = threadIdx.x; i < B * p.pass_rows; i += kThreads) acc[i] = 0.0f;
#pragma unroll
            for (int q = 0; q < kXStageRegs; ++q) {
                const int u = threadIdx.x + q * kThreads;
                if (u < B * units) {
                    const int b = (B == 1) ? 0 : u / units;
                    const int v = u - b * units;
                    *reinterpret_cast<uint4*>(xs + b * p.x_b_stride + (v >> 3) * kXChunkBytes + (v & 7) * 16) = xr[q];
                }
            }
            for (int u = threadIdx.x + kXStageRegs * kThreads; u < B * units; u += kThreads) {  // rest, if any
                const int b = u / units;
                const int v = u - b * units;
                *reinterpret_cast<uint4*>(xs + b * p.x_b_stride + (v >> 3) * kXChunkBytes + (v & 7) * 16) =
                    __ldg(xg + static_cast<size_t>(b) * (p.k / 8) + v);
            }
            __syncthreads();  // x tile and zeroed accumulators visible to every warp

            float part[B];
#pragma unroll
            for (int b = 0; b < B; ++b) part[b] = 0.0f;
            TaskCursor cc;
            cc.start(ts, t_begin);
            int flush_quad = cc.quad;
            for (int t0 = t_begin; t0 < t_end; t0 += kPrefetch) {
#pragma unroll
                for (int q = 0; q < kPrefetch; ++q) {
                    if (t0 + q >= t_end) break;
                    if (cc.quad != flush_quad) {  // warp-uniform
                        TaskCursor fq = cc;
                        fq.quad = flush_quad;
                        flush_rows<B>(acc, p.pass_rows, fq.row(r, ts), j, part);
                        flush_quad = cc.quad;
                    }
                    compute_task<FMT, B>(p, ts, xs, cc, r, j, buf[q], part);
                    cc.next(ts);
                    // refill the registers just consumed with the task kPrefetch ahead
                    if (t0 + q + kPrefetch < t_end) load_next<FMT>(p, ts, row_begin, r, j, ls, buf[q]);
                }
            }
            if (t_begin < t_end) {
                TaskCursor fq = cc;
                fq.quad = flush_quad;
                flush_rows<B>(acc, p.pass_rows, fq.row(r, ts), j, part);
            }
        }
        __syncthreads();  // all partial sums of this pass are in `acc`
        for (int i = threadIdx.x; i < B * prows; i += kThreads) {
            const int b = i / prows;
            const int rr = i - b * prows;
            p.y[static_cast<size_t>(b) * p.n + row_begin + prow0 + rr] = __float2half_rn(acc[b * p.pass_rows + rr]);
        }
    }
}

}  // namespace sgemv
