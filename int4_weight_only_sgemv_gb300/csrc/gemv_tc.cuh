// 2:4 sparse INT4 GEMV on the sparse tensor cores of GB300 (sm_103a): the SparseGemv of the paper
// "Efficient LLM-based Advertising via Model Compression and Parallel Verification" (§3.3 "Revised
// Kernel"), reading the same "2bit-CSR" packed layout as the CUDA-core kernel (gemv_kernel.cuh).
//
// The 2:4 pattern with a 2-bit in-block position per kept element is exactly the operand format of the
// sparse matrix-multiply-accumulate (mma.sp, m16n8k32, fp16 sources, fp32 accumulation): A is 16 rows
// x 32 dense columns given as its 16 kept values per row plus a 4-bit (p0, p1) field per 4-column
// block; the instruction itself gathers the activations at the kept positions. One instruction thus
// retires the gather and the multiply-adds of 256 kept weights, for up to 8 batch rows (n = 8), and the
// CUDA cores are left with the dequantisation only. The DRAM traffic is that of the CUDA-core kernel:
// every packed byte is read once, x is read from shared memory.
//
// Work split (one persistent CTA of 16 warps per SM, as in the CUDA-core kernel):
//   * CTA c owns a contiguous, balanced range of output rows; tasks are 16 rows x 256 columns, each
//     warp takes a contiguous run of tasks (along the columns of a 16-row tile first).
//   * Each warp streams its tasks' packed bytes into a private ring of tc_stages(B) shared-memory stages
//     (16 rows x 256 columns: vals, idx and {s, z} words) with 16-byte asynchronous copies (3-4 per
//     lane per stage, no register cost while in flight), tc_stages(B) - 1 stages ahead of its compute.
//     Rows beyond the pass and columns beyond the x tile copy valid bytes of the task's own rows (the
//     first row / the tile's first columns), against zero activations, so the compute needs no checks
//     and every position field the instruction sees is a valid ordered pair.
//   * x is staged once per CTA (per x tile) in the order of the B fragments of the instruction, so
//     that a lane reads its 4 activation pairs of a 32-column window with one 16-byte load.
//
// Lane (g, t) = (lane / 4, lane % 4) of a warp holds rows g and g + 8 of the task's 16 rows. For the
// 32 columns = 2 vals words (u, u+1) = 8 blocks of a window, the instruction's block j (0..7) is block
// kPerm[j % 4] of word u + j / 4, with kPerm = {0, 2, 1, 3}:
//   * A: lane t holds block kPerm[t] of words u and u+1 for both rows: the two nibbles of a block sit in
//     slots s and s+4 of the word (bits 4s and 16+4s), so one shift (by 0 or 8), one AND-OR with the
//     fp16 exponent of 1024 (mask at bits 0-3 or 4-7) and one HFMA2 (scale 1 or 1/16, minus 1024+z or
//     64+z) give the exact half2 {q0 - z, q1 - z};
//   * metadata: lanes t = 0 / 1 give blocks 0-3 / 4-7 of rows g (bits 0-15) and g+8 (bits 16-31). The
//     16-bit position word of one vals word holds p0 of its 4 blocks in its low byte and p1 in its high
//     byte; with kPerm the instruction's nibbles are (low byte & 0x33 | (high byte & 0x33) << 2) and
//     ((low byte >> 2) & 0x33 | high byte & 0xCC), i.e. one byte permute, two shifts and two LOP3 for
//     both rows.
//   * the group scale multiplies the fp32 accumulator of each group (g columns) once.
// The only waits are cp.async.wait_group (on the lane's own copies), __syncwarp and CTA barriers that
// every thread reaches, so the kernel cannot hang.
#pragma once

#include "gemv_kernel.cuh"

namespace sgemv {

// ------------------------------------------------------------------------------------------------
// PTX helpers.

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async8(uint32_t dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ uint4 lds128(uint32_t a) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
    return v;
}
__device__ __forceinline__ uint2 lds64(uint32_t a) {
    uint2 v;
    asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a));
    return v;
}
__device__ __forceinline__ uint32_t lds32(uint32_t a) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
    return v;
}

// (a & m) | (b & ~m) in one LOP3.
__device__ __forceinline__ uint32_t bitsel(uint32_t a, uint32_t b, uint32_t m) {
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0xE4;" : "=r"(d) : "r"(a), "r"(b), "r"(m));
    return d;
}

// d += A(16x32, 2:4 sparse, fp16) * B(32x8, fp16), fp32 accumulation; metadata from lanes t = 0, 1.
__device__ __forceinline__ void mma_sp(float (&d)[4], const uint32_t (&a)[4], const uint4& b, uint32_t e) {
    asm volatile(
        "mma.sp::ordered_metadata.sync.aligned.m16n8k32.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
        "{%8, %9, %10, %11}, {%0, %1, %2, %3}, %12, 0x0;"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b.x), "r"(b.y), "r"(b.z), "r"(b.w), "r"(e));
}

// Position words of word u of rows g (bytes 0-1 of x) and g+8 (bytes 2-3) -> the instruction's
// metadata nibbles (p0 | p1 << 2) of blocks kPerm = {0, 2, 1, 3}:
//   byte 0 = (b0 & 0x33) | ((b1 & 0x33) << 2),   byte 1 = ((b0 >> 2) & 0x33) | (b1 & 0xCC)
// for (b0, b1) = bytes 0-1, and the same for bytes 2-3.
__device__ __forceinline__ uint32_t tc_metadata(uint32_t x) {
    const uint32_t t = bitsel(x, x >> 6, 0xCC33CC33u);
    return bitsel(x << 6, t, 0x33003300u);
}

// Lane constants of the dequantisation (t = lane % 4 takes block kPerm[t] of each word).
struct TcLane {
    uint32_t shift;   // 0 or 8
    uint32_t mask;    // nibble pair at bits 0-3 / 16-19 or 4-7 / 20-23
    uint32_t c1;      // half2 scale: 1 or 1/16
    uint32_t nbase;   // half2 -(1024) or -(64)
    uint32_t msel;    // byte permute picking the position words of word u (t = 0) or u+1 (t = 1)
};
__device__ __forceinline__ TcLane tc_lane(int t) {
    TcLane L;
    L.shift = (t & 1) ? 8u : 0u;
    L.mask = (t & 2) ? 0x00F000F0u : 0x000F000Fu;
    L.c1 = (t & 2) ? 0x2C002C00u : 0x3C003C00u;      // 1/16 : 1
    L.nbase = (t & 2) ? 0xD400D400u : 0xE400E400u;   // -64 : -1024
    L.msel = (t & 1) ? 0x7632u : 0x5410u;
    return L;
}

// {q - z} for the lane's block of vals word w; c2 = -(base + z) as half2.
__device__ __forceinline__ uint32_t tc_dequant(uint32_t w, const TcLane& L, uint32_t c2) {
    return hfma2_bits(and_or(w >> L.shift, L.mask, 0x64006400u), L.c1, c2);
}

// c2 = -(base + z) (exact: base + z is an integer below 2048) and s of one {s, z} word.
__device__ __forceinline__ uint32_t tc_c2(uint32_t szw, const TcLane& L) {
    return hsub2_bits(L.nbase, prmt(szw, szw, 0x3232u));
}
__device__ __forceinline__ float tc_s(uint32_t szw) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(szw & 0xFFFFu)));
}

// Tasks of one (pass, x tile): task t -> (16-row tile t / nblk, 256-column block t % nblk).
__host__ __device__ __forceinline__ void tc_task_space(TaskSpace& ts, int prow0, int prows, int tc0, int tcols) {
    ts.prow0 = prow0;
    ts.prows = prows;
    ts.tc0 = tc0;
    ts.tcols = tcols;
    ts.nblk = (tcols + kTcStageCols - 1) / kTcStageCols;
    ts.nfull = tcols / kTcStageCols;
    ts.ntasks = ((prows + kTcRows - 1) / kTcRows) * ts.nblk;
}

// ------------------------------------------------------------------------------------------------
// Copy side: lane L copies, per stage, vals chunk L % 4 (64 columns) of rows L / 4 and L / 4 + 8, idx
// chunk L % 2 (128 columns) of row L / 2 and, for L < 16, the {s, z} words of row L.

struct TcCopier {
    int quad, blk;             // next task to copy: 16-row tile `quad`, 256-column block `blk`
    const uint8_t* v0;         // the task's sources: vals of the lane's two rows (lane's 64 columns)
    const uint8_t* v1;
    const uint8_t* ip;         // idx of the lane's idx row (lane's 128 columns)
    const uint8_t* sp;         // {s, z} words of the lane's sz row (the task's groups)

    __host__ __device__ void set_quad(const GemvParams& p, const TaskSpace& ts, int row_begin, int lane, int q) {
        quad = q;
        blk = 0;
        const int last = ts.prows - 1;  // rows beyond the pass copy the pass's last row (results dropped)
        const size_t r0 = static_cast<size_t>(row_begin + ts.prow0);
        const int rv = q * kTcRows + (lane >> 2);
        const int ri = q * kTcRows + (lane >> 1);
        const int rs = q * kTcRows + (lane & 15);
        const uint32_t ov = static_cast<uint32_t>(ts.tc0) / 4 + 16 * (lane & 3);
        v0 = p.vals + (r0 + (rv < last ? rv : last)) * p.vals_pitch + ov;
        v1 = p.vals + (r0 + (rv + 8 < last ? rv + 8 : last)) * p.vals_pitch + ov;
        ip = p.idx + (r0 + (ri < last ? ri : last)) * p.idx_pitch + static_cast<uint32_t>(ts.tc0) / 8 + 16 * (lane & 1);
        sp = p.sz + (r0 + (rs < last ? rs : last)) * p.sz_pitch + ((static_cast<uint32_t>(ts.tc0) >> p.log2g) << 2);
    }
    __host__ __device__ void step(const GemvParams& p, int nb) {  // move the sources nb blocks right
        v0 += 64 * nb;
        v1 += 64 * nb;
        ip += 32 * nb;
        sp += (1024 >> p.log2g) * nb;
    }
    __host__ __device__ void start(const GemvParams& p, const TaskSpace& ts, int row_begin, int lane, int t) {
        const int q = t / ts.nblk;
        set_quad(p, ts, row_begin, lane, q);
        blk = t - q * ts.nblk;
        step(p, blk);
    }
    // Sources of the next task's copies (16 bytes each): vals of the two rows, idx, and the 16-byte unit
    // of {s, z} words that holds the task's groups (sz rows are 16-byte aligned and padded to 16 bytes;
    // lanes L and L + 16 copy the same unit). In the last block of a tile whose width is not a multiple
    // of 256, chunks beyond the tile copy the tile's first columns of the same rows instead.
    __host__ __device__ void sources(const GemvParams& p, const TaskSpace& ts, int lane, const uint8_t* (&src)[4]) const {
        src[0] = v0;
        src[1] = v1;
        src[2] = ip;
        src[3] = sp;
        if (blk >= ts.nfull) {
            const int col = blk * kTcStageCols;
            const int cv = col + 64 * (lane & 3), ci = col + 128 * (lane & 1);
            if (cv >= ts.tcols) src[0] = v0 - cv / 4, src[1] = v1 - cv / 4;
            if (ci >= ts.tcols) src[2] = ip - ci / 8;
            if (col >= ts.tcols) src[3] = sp - ((col >> p.log2g) << 2);
        }
        src[3] = reinterpret_cast<const uint8_t*>(reinterpret_cast<uintptr_t>(src[3]) & ~static_cast<uintptr_t>(15));
    }
    __host__ __device__ void advance(const GemvParams& p, const TaskSpace& ts, int row_begin, int lane) {
        if (++blk == ts.nblk)
            set_quad(p, ts, row_begin, lane, quad + 1);
        else
            step(p, 1);
    }
};

// Destinations of lane L's copies within a stage.
__host__ __device__ __forceinline__ uint32_t tc_dst_vals(int lane) { return (lane >> 2) * kTcValsPitch + 16 * (lane & 3); }
__host__ __device__ __forceinline__ uint32_t tc_dst_idx(int lane) { return kTcIdxOff + (lane >> 1) * kTcIdxPitch + 16 * (lane & 1); }
__host__ __device__ __forceinline__ uint32_t tc_dst_sz(int lane) { return kTcSzOff + lane * kTcSzPitch; }

// Issue the copies of the copier's next stage into the stage at shared address `slot`, then advance.
__device__ __forceinline__ void tc_issue(TcCopier& cp, const GemvParams& p, const TaskSpace& ts, int row_begin,
                                         int lane, uint32_t slot) {
    const uint8_t* src[4];
    cp.sources(p, ts, lane, src);
    const uint32_t dv = slot + tc_dst_vals(lane);
    cp_async16(dv, src[0]);
    cp_async16(dv + 8 * kTcValsPitch, src[1]);
    cp_async16(slot + tc_dst_idx(lane), src[2]);
    cp_async16(slot + tc_dst_sz(lane & 15), src[3]);  // lanes L and L + 16 write the same bytes
    cp.advance(p, ts, row_begin, lane);
}

// ------------------------------------------------------------------------------------------------
// Compute side.

// One task (256 columns, 8 instructions) of the lane's rows, for groups of 2^LOG2G columns; xw = x tile
// at the task's first window (lane's batch column and 16-byte slot), szoff = byte offset of the task's
// first {s, z} word in the copied 16-byte unit.
template <int LOG2G>
__device__ __forceinline__ void tc_stage(uint32_t slot, int g8, const TcLane& L, uint32_t xw, uint32_t szoff,
                                         float (&acc)[4]) {
    constexpr int kGroups = kTcStageCols >> LOG2G;  // groups per task: 4, 2 or 1
    constexpr int kWinPerGroup = (1 << LOG2G) / 32;
    const uint32_t rv = slot + g8 * kTcValsPitch;   // row g's vals; row g + 8 at + 8 pitches
    const uint32_t ri = slot + kTcIdxOff + g8 * kTcIdxPitch;
    const uint32_t rs = slot + kTcSzOff + g8 * kTcSzPitch + szoff;
    uint32_t sa[kGroups], sb[kGroups];  // {s, z} words of rows g / g+8
    if constexpr (kGroups == 4) {
        const uint4 a = lds128(rs), b = lds128(rs + 8 * kTcSzPitch);
        sa[0] = a.x, sa[1] = a.y, sa[2] = a.z, sa[3] = a.w;
        sb[0] = b.x, sb[1] = b.y, sb[2] = b.z, sb[3] = b.w;
    } else if constexpr (kGroups == 2) {
        const uint2 a = lds64(rs), b = lds64(rs + 8 * kTcSzPitch);
        sa[0] = a.x, sa[1] = a.y;
        sb[0] = b.x, sb[1] = b.y;
    } else {
        sa[0] = lds32(rs);
        sb[0] = lds32(rs + 8 * kTcSzPitch);
    }
    float d[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
    for (int h = 0; h < 2; ++h) {  // 128 columns: 8 vals words, 8 position words per row
        const uint4 va0 = lds128(rv + 32 * h), va1 = lds128(rv + 32 * h + 16);
        const uint4 vb0 = lds128(rv + 8 * kTcValsPitch + 32 * h), vb1 = lds128(rv + 8 * kTcValsPitch + 32 * h + 16);
        const uint4 ia = lds128(ri + 16 * h), ib = lds128(ri + 8 * kTcIdxPitch + 16 * h);
        const uint32_t wa[8] = {va0.x, va0.y, va0.z, va0.w, va1.x, va1.y, va1.z, va1.w};
        const uint32_t wb[8] = {vb0.x, vb0.y, vb0.z, vb0.w, vb1.x, vb1.y, vb1.z, vb1.w};
        const uint32_t xa[4] = {ia.x, ia.y, ia.z, ia.w};
        const uint32_t xb[4] = {ib.x, ib.y, ib.z, ib.w};
        uint32_t ca = 0, cb = 0;
#pragma unroll
        for (int m = 0; m < 4; ++m) {  // one 32-column window: vals words 2m, 2m+1
            const int w = 4 * h + m;   // window within the task
            const int q = w / kWinPerGroup;
            if (w % kWinPerGroup == 0 || m == 0) {
                ca = tc_c2(sa[q], L);
                cb = tc_c2(sb[q], L);
            }
            const uint32_t a[4] = {tc_dequant(wa[2 * m], L, ca), tc_dequant(wb[2 * m], L, cb),
                                   tc_dequant(wa[2 * m + 1], L, ca), tc_dequant(wb[2 * m + 1], L, cb)};
            const uint32_t e = tc_metadata(prmt(xa[m], xb[m], L.msel));
            mma_sp(d, a, lds128(xw + w * kTcWindowBytes), e);
            if ((w + 1) % kWinPerGroup == 0) {  // the group's last window: scale its sums
                const float s0 = tc_s(sa[q]), s1 = tc_s(sb[q]);
                acc[0] = fmaf(s0, d[0], acc[0]);
                acc[1] = fmaf(s0, d[1], acc[1]);
                acc[2] = fmaf(s1, d[2], acc[2]);
                acc[3] = fmaf(s1, d[3], acc[3]);
                d[0] = d[1] = d[2] = d[3] = 0.0f;
            }
        }
    }
}

// Add the lane's sums (rows g, g+8 of the task; batch columns 2t, 2t+1) into the shared accumulators.
template <int B>
__device__ __forceinline__ void tc_flush(float* acc_sm, int pass_rows, int row0, int prows, int g8, int t,
                                         float (&acc)[4]) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int n = 2 * t + (k & 1);
        const int row = row0 + g8 + 8 * (k >> 1);
        if (n < B && row < prows) atomicAdd(acc_sm + n * pass_rows + row, acc[k]);
        acc[k] = 0.0f;
    }
}

// Stage x (all batch rows of one x tile) in B-fragment order: for the 32-column window w of batch row
// b, the 16 bytes of lane t at xs + b*x_b_stride + 64w + 16t hold the activation pairs (32-bit words of
// the window) {0, 2, 8, 10} + {0, 1, 4, 5}[t], the pairs that the instruction's fragment of lane t
// multiplies under kPerm. Columns beyond the tile, up to whole 1024-column blocks, are zero.
template <int B>
__device__ __forceinline__ void tc_stage_x(const GemvParams& p, const TaskSpace& ts, uint8_t* xs) {
    const int units = ts.tcols / 8;                // 16-byte units of x per batch row
    const int punits = ts.nblk * (kTcStageCols / 8);  // staged units per batch row
    const int nunits = B * punits;
    const uint4* xg = reinterpret_cast<const uint4*>(p.x + ts.tc0);
    for (int u0 = threadIdx.x; u0 < nunits; u0 += kXStageRegs * kXThreads) {
        uint4 xr[kXStageRegs];
#pragma unroll
        for (int q = 0; q < kXStageRegs; ++q) {
            const int u = u0 + q * kXThreads;
            const int b = (B == 1) ? 0 : u / punits;
            const int v = u - b * punits;
            xr[q] = make_uint4(0, 0, 0, 0);
            if (u < nunits && v < units) xr[q] = __ldg(xg + static_cast<size_t>(b) * (p.k / 8) + v);
        }
#pragma unroll
        for (int q = 0; q < kXStageRegs; ++q) {
            const int u = u0 + q * kXThreads;
            if (u < nunits) {
                const int b = (B == 1) ? 0 : u / punits;
                const int v = u - b * punits;
                const int e = v & 3;  // words 4e .. 4e+3 of window v / 4
                uint8_t* base = xs + b * p.x_b_stride + (v >> 2) * kTcWindowBytes + 32 * (e & 1) + 8 * (e >> 1);
                const uint32_t w[4] = {xr[q].x, xr[q].y, xr[q].z, xr[q].w};
#pragma unroll
                for (int k = 0; k < 4; ++k)  // word 4e + k -> lane 2(e & 1) + (k & 1), register (k >> 1) + 2(e >> 1)
                    *reinterpret_cast<uint32_t*>(base + 16 * (k & 1) + 4 * (k >> 1)) = w[k];
            }
        }
    }
}

// One layer of a launch on the tensor-core path: this CTA's rows (all passes and x tiles).
template <int B>
__device__ __forceinline__ void run_layer_tc(const GemvParams& p, int cta, int warp, int lane, uint8_t* smem,
                                             const TcLane& L, bool& waited_pdl, bool& smem_in_use) {
    constexpr int S = tc_stages(B);
    const int g8 = lane >> 2;  // rows g8 and g8 + 8 of a task; batch column g8 of the B fragment
    const int t = lane & 3;
    int row_begin, nrows_cta;
    cta_rows(p, cta, row_begin, nrows_cta);
    if (nrows_cta <= 0) return;

    float* acc_sm = reinterpret_cast<float*>(smem + p.sm_acc);
    uint8_t* xs = smem + p.sm_x;
    const uint32_t ring = smem_addr(smem + p.sm_ring) + static_cast<uint32_t>(warp) * S * kTcStageBytes;
    // lanes of batch columns >= B read batch row 0 (same addresses as its lanes: a broadcast); their
    // columns of the result are never used
    const uint32_t xw_lane = smem_addr(xs) + (g8 < B ? g8 : 0) * p.x_b_stride + 16 * t;
    const int ntile = (p.k + p.xt - 1) / p.xt;
    const int npass = (nrows_cta + p.pass_rows - 1) / p.pass_rows;

    for (int pass = 0; pass < npass; ++pass) {
        const int prow0 = pass * p.pass_rows;
        const int prows = min(p.pass_rows, nrows_cta - prow0);
        for (int tile = 0; tile < ntile; ++tile) {
            TaskSpace ts;
            tc_task_space(ts, prow0, prows, tile * p.xt, min(p.xt, p.k - tile * p.xt));
            int t_begin, t_end;
            warp_run(ts.ntasks, warp, t_begin, t_end);
            if (!waited_pdl) {
                // x and the packed weights may be written by the previous kernel in the stream
                pdl_wait();
                waited_pdl = true;
            }
            if (smem_in_use) __syncthreads();  // the previous x tile / accumulators are no longer read
            smem_in_use = true;
            const int ns = t_end - t_begin;  // tasks (= ring stages) of this warp
            TcCopier cp;
            if (ns > 0) cp.start(p, ts, row_begin, lane, t_begin);
            uint32_t islot = ring;  // next stage to fill / to compute
            uint32_t cslot = ring;
            const uint32_t ring_end = ring + S * kTcStageBytes;
#pragma unroll
            for (int q = 0; q < S - 1; ++q) {
                if (q < ns) tc_issue(cp, p, ts, row_begin, lane, islot);
                islot += kTcStageBytes;
                cp_async_commit();
            }
            if (warp >= kXWarps) {
                named_bar_sync(1, kThreads);  // x tile and zeroed accumulators visible
            } else {
                if (tile == 0)
                    for (int i = threadIdx.x; i < B * p.pass_rows; i += kXThreads) acc_sm[i] = 0.0f;
                tc_stage_x<B>(p, ts, xs);
                named_bar_sync(2, kXThreads);   // every staging thread's stores are done
                named_bar_arrive(1, kThreads);  // release the other warps
            }

            float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
            int cquad = t_begin / ts.nblk;  // task being computed: (cquad, cblk)
            int cblk = t_begin - cquad * ts.nblk;
            // the task at (cquad, cblk): stage at cslot, x windows from xw, {s, z} offset of its groups
            auto compute = [&]() {
                const uint32_t xw = xw_lane + cblk * (kTcStageCols / 32) * kTcWindowBytes;
                const uint32_t szoff = (static_cast<uint32_t>(cblk) << (10 - p.log2g)) & 15u;
                if (p.log2g == 7)
                    tc_stage<7>(cslot, g8, L, xw, szoff, acc);
                else if (p.log2g == 6)
                    tc_stage<6>(cslot, g8, L, xw, szoff, acc);
                else
                    tc_stage<8>(cslot, g8, L, xw, szoff, acc);
                cslot = cslot + kTcStageBytes == ring_end ? ring : cslot + kTcStageBytes;
                if (++cblk == ts.nblk) {  // warp-uniform: the 16 rows are done
                    tc_flush<B>(acc_sm, p.pass_rows, cquad * kTcRows, prows, g8, t, acc);
                    ++cquad;
                    cblk = 0;
                }
            };
            int i = 0;
            for (; i + S - 1 < ns; ++i) {  // steady state: refill the stage computed last
                cp_async_wait<S - 2>();    // this lane's copies of stage i have landed
                __syncwarp();              // ... and every lane's; stage i - 1 is no longer read
                tc_issue(cp, p, ts, row_begin, lane, islot);
                islot = islot + kTcStageBytes == ring_end ? ring : islot + kTcStageBytes;
                cp_async_commit();
                compute();
            }
            for (; i < ns; ++i) {  // drain
                cp_async_wait<S - 2>();
                __syncwarp();
                cp_async_commit();
                compute();
            }
            if (ns > 0 && cblk != 0) tc_flush<B>(acc_sm, p.pass_rows, cquad * kTcRows, prows, g8, t, acc);
            __syncwarp();
        }
        __syncthreads();  // all partial sums of this pass are in `acc_sm`
        for (int i = threadIdx.x; i < B * prows; i += kThreads) {
            const int b = i / prows;
            const int rr = i - b * prows;
            p.y[static_cast<size_t>(b) * p.n + row_begin + prow0 + rr] = __float2half_rn(acc_sm[b * p.pass_rows + rr]);
        }
    }
}

// The tensor-core kernel: one layer, or a group of independent layers run one after the other (as in
// gemv_kernel).
template <int B, bool kMulti>
__global__ void __launch_bounds__(kThreads, 1) gemv_tc_kernel(const __grid_constant__ LayerGroup g) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int cta = blockIdx.x;
    pdl_launch_dependents();
    if (warp == kWarps - 1) {
        // while the previous kernel in the stream finishes, have L2 fetch this CTA's first weights
        int rb, nr;
        cta_rows(g.layer[0], cta, rb, nr);
        if (nr > 0) prefetch_layer<true>(g.layer[0], rb, min(nr, g.layer[0].pass_rows), lane);
    }
    const TcLane L = tc_lane(lane & 3);
    bool waited_pdl = false;
    bool smem_in_use = false;
    if constexpr (!kMulti) {
        run_layer_tc<B>(g.layer[0], cta, warp, lane, smem, L, waited_pdl, smem_in_use);
    } else {
        for (int layer = 0; layer < g.n_layers; ++layer)
            run_layer_tc<B>(g.layer[layer], cta, warp, lane, smem, L, waited_pdl, smem_in_use);
    }
}

}  // namespace sgemv
