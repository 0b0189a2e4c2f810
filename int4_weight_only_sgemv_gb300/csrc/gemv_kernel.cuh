// INT4 weight-only GEMV kernels for GB300 (sm_103a): the SparseGemv of the paper "Efficient LLM-based
// Advertising via Model Compression and Parallel Verification" (§3.3 "Revised Kernel") over the 2:4
// "2bit-CSR" format, and the dense INT4 variant ("previous generation Gemv", same section).
//
// Work split (one persistent CTA of 16 warps per SM):
//   * CTA c owns a contiguous, balanced range of output rows (±1 row between CTAs); its share of the
//     packed layer is read exactly once from HBM.
//   * The CTA's rows are cut into tasks of 4 rows x 1024 columns; warp w takes a contiguous run of
//     tasks (runs differ by at most one task). Lane (r, j) = (lane / 8, lane % 8) handles columns
//     128j .. 128j + 127 (two chunks of 64) of row r, so one 256-bit load brings a lane's nibbles and
//     the 8 column-lanes of a row read 256 contiguous bytes.
//   * The weights go straight from HBM into registers with streaming loads; each warp keeps the next
//     1-3 tasks (fewer at larger batch) in flight while it computes. Nothing is read before the
//     dependent-launch wait (a packer, like the previous GEMV, may precede the kernel in the stream),
//     but one warp first asks L2 to prefetch the CTA's weights, so they stream from HBM while the
//     previous kernel finishes.
//   * x is staged once per CTA (per x tile when B*K is too large) into shared memory by 8 warps while
//     the others issue their first weight loads: 272 bytes per lane's 128 columns (as byte planes of
//     4-column blocks for the sparse kernel, zero beyond the tile up to whole 1024-column blocks), so
//     that the 8 column-lanes of a task read 8 different bank groups and the 4 row-lanes of a column
//     broadcast (the paper's conflict-free activation layout and block-level cooperative load, §3.3
//     "Accelerate Memory Access").
//   * A lane accumulates its row's partial sum in registers over consecutive tasks of the same 4 rows;
//     when the rows change, the 8 column-lanes combine with warp shuffles and add into an fp32
//     accumulator per (row, batch) in shared memory. The CTA writes y once at the end.
//
// Per 8 kept elements (one 32-bit word of nibbles, one 16-bit word of positions) and batch row:
//   * dequantisation (§3.3 "Reduce Computational Burden", lop3): one AND-OR per nibble pair gives
//     half2 {1024+q0, 1024+q1} (or 1024+16q for the odd nibbles), one HSUB2 removes 1024+z exactly;
//   * the 2-bit positions of a block become a byte-permute selector: one mask (which also adds a fill
//     constant) and one multiply per selector; one PRMT gathers the two activations of the block from
//     the two 32-bit words holding its four fp16 activations as byte planes;
//   * products (q - z) * x are exact in fp32 (mixed-precision FMA, fp16 sources, fp32 accumulate); the
//     group scale is applied once per 64 columns.
// The byte permutes and AND-ORs are written as PTX (prmt, lop3) so that each is one instruction.
// No tensor cores: a batch <= 8 GEMV is no dense contraction; what bounds this kernel on GB300 is the
// issue rate of the integer and FP32 work per kept weight (and HBM on large layers). The only waits on other threads are CTA barriers
// (__syncthreads and two named barriers) that every thread of the CTA reaches, so the kernel cannot hang.
#pragma once

#include <cooperative_groups.h>

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

// acc + a.lo*b.lo + a.hi*c.lo: the two halves of a against the low halves of b and c (fp16 sources,
// fp32 accumulation, products exact in fp32).
__device__ __forceinline__ float fma_h2_lo_f32(uint32_t a, uint32_t b, uint32_t c, float acc) {
    float d;
    asm("{\n\t.reg .f16 a0, a1, b0, b1, c0, c1;\n\t.reg .f32 t;\n\t"
        "mov.b32 {a0, a1}, %1;\n\t"
        "mov.b32 {b0, b1}, %2;\n\t"
        "mov.b32 {c0, c1}, %3;\n\t"
        "fma.rn.f32.f16 t, a0, b0, %4;\n\t"
        "fma.rn.f32.f16 %0, a1, c0, t;\n\t}"
        : "=f"(d)
        : "r"(a), "r"(b), "r"(c), "f"(acc));
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

// Gather selectors. In the x tile of the sparse kernel the four fp16 activations of a block sit in two
// 32-bit words as byte planes: word 0 = low bytes of x0..x3, word 1 = high bytes. The selector that
// gathers {x_p0, x_p1} is then the nibbles (p0, p0+4, p1, p1+4) = Q*0x11 + 0x4040, Q = p0 + 256*p1.
// m carries Q0 (block of one vals word) in bytes 0-1 and Q1 (same block of the next word) in bytes
// 2-3, plus the constant 0xF4B87C40 in the bits the 2-bit fields leave free (so that the mask that
// extracts the fields adds it for free):
//   * m * 0x11 (low 32 bits): 0x7C40 * 0x11 = 0x84040, so bits 0-15 are Q0*0x11 + 0x4040;
//   * hi32(m * 0x110000) = floor(m * 0x11 / 2^16) = (Q1 + 0xF4B8) * 0x11 + 8, since (Q0 + 0x7C40) * 0x11
//     lies in [0x84040, 0x87373], and 0xF4B8 * 0x11 + 8 = 0x104040: bits 0-15 are Q1*0x11 + 0x4040.
// prmt reads only bits 0-15 of its selector.
constexpr uint32_t kSelFill = 0xF4B87C40u;
__device__ __forceinline__ uint32_t sel_lo(uint32_t m) { return m * 0x11u; }
__device__ __forceinline__ uint32_t sel_hi(uint32_t m) { return __umulhi(m, 0x110000u); }

// 16 bytes of x (x0..x7, fp16) -> the byte-plane form of its two blocks.
__device__ __forceinline__ uint4 byte_planes(uint4 u) {
    return make_uint4(prmt(u.x, u.y, 0x6420u), prmt(u.x, u.y, 0x7531u), prmt(u.z, u.w, 0x6420u),
                      prmt(u.z, u.w, 0x7531u));
}

__device__ __forceinline__ uint32_t hsub2_bits(uint32_t a, uint32_t b) {
    __half2 r = __hsub2(*reinterpret_cast<const __half2*>(&a), *reinterpret_cast<const __half2*>(&b));
    return *reinterpret_cast<const uint32_t*>(&r);
}

__device__ __forceinline__ uint32_t hfma2_bits(uint32_t a, uint32_t b, uint32_t c) {
    __half2 r = __hfma2(*reinterpret_cast<const __half2*>(&a), *reinterpret_cast<const __half2*>(&b),
                        *reinterpret_cast<const __half2*>(&c));
    return *reinterpret_cast<const uint32_t*>(&r);
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

// {s, z} word of a group -> s in fp32 and the half2 constants 1024 + z and 1024 + 16z (exact for the
// integer zero points 0..15 the packer writes).
__device__ __forceinline__ GroupParams group_params(uint32_t szw) {
    GroupParams g;
    g.s = __half2float(__ushort_as_half(static_cast<unsigned short>(szw & 0xFFFFu)));
    const uint32_t zz = prmt(szw, szw, 0x3232u);  // {z, z}
    g.zA = hsub2_bits(zz, 0xE400E400u);             // z - (-1024)
    g.zB = hfma2_bits(zz, 0x4C004C00u, 0x64006400u);  // z * 16 + 1024
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
        for (int t = 0; t < 4; ++t) {
            const uint32_t m = and_or(i2[u] >> (2 * t), 0x03030303u, kSelFill);
            S[0][t] = sel_lo(m);
            S[1][t] = sel_hi(m);
        }
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

// One 64-column chunk (16 blocks, 16 kept) of a 1:4 row for every batch row, added into part[b].
//   v: 2 words of nibbles (word h: blocks 8h..8h+7, one per slot), ix: 2 u16 words of positions,
//   xp: the chunk's activations as byte planes (16-byte unit u: blocks 2u and 2u+1).
// Selectors: m_t = fields of blocks t, 4+t, 8+t, 12+t (bytes 0..3) plus the fill constant; byte k of
// m_t * 0x11 is the selector (nibbles p, p+4) for block 4k+t, brought down to bits 0-7 by the low or a
// high product (prmt reads only the low nibbles here: one activation per block).
template <int B>
__device__ __forceinline__ void sparse14_chunk(const uint2 v, const uint32_t ix, const uint32_t szw,
                                               const uint8_t* xp, const uint32_t xbs, float (&part)[B]) {
    const GroupParams gp = group_params(szw);
    float accA[B], accB[B];
#pragma unroll
    for (int b = 0; b < B; ++b) accA[b] = accB[b] = 0.0f;
    uint32_t S[4][4];  // [t][k]: selector of block 4k+t
#pragma unroll
    for (int t = 0; t < 4; ++t) {
        const uint32_t m = and_or(ix >> (2 * t), 0x03030303u, kSelFill);
        S[t][0] = sel_lo(m);
        S[t][1] = __umulhi(m, 0x11000000u);
        S[t][2] = __umulhi(m, 0x00110000u);
        S[t][3] = __umulhi(m, 0x00001100u);
    }
    const uint32_t w2[2] = {v.x, v.y};
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        uint32_t d[4];  // d[i] = {q of block 8h+i, q of block 8h+i+4} - z (x16 for odd i)
        dequant_word(w2[h], gp.zA, gp.zB, d);
#pragma unroll
        for (int b = 0; b < B; ++b) {
            const uint8_t* xw = xp + b * xbs + 64 * h;  // units 4h..4h+3: blocks 8h..8h+7
            const uint4 u0 = *reinterpret_cast<const uint4*>(xw);
            const uint4 u1 = *reinterpret_cast<const uint4*>(xw + 16);
            const uint4 u2 = *reinterpret_cast<const uint4*>(xw + 32);
            const uint4 u3 = *reinterpret_cast<const uint4*>(xw + 48);
            // block 8h+i (i = 0..3) sits in u0/u1, block 8h+i+4 in u2/u3; even blocks in .x/.y
            accA[b] = fma_h2_lo_f32(d[0], prmt(u0.x, u0.y, S[0][2 * h]), prmt(u2.x, u2.y, S[0][2 * h + 1]), accA[b]);
            accB[b] = fma_h2_lo_f32(d[1], prmt(u0.z, u0.w, S[1][2 * h]), prmt(u2.z, u2.w, S[1][2 * h + 1]), accB[b]);
            accA[b] = fma_h2_lo_f32(d[2], prmt(u1.x, u1.y, S[2][2 * h]), prmt(u3.x, u3.y, S[2][2 * h + 1]), accA[b]);
            accB[b] = fma_h2_lo_f32(d[3], prmt(u1.z, u1.w, S[3][2 * h]), prmt(u3.z, u3.w, S[3][2 * h + 1]), accB[b]);
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

// Registers holding the weights of one task for one lane: two adjacent chunks of 64 columns.
template <int FMT>
struct TaskRegs;

template <>
struct TaskRegs<SGEMV_FMT_SPARSE24> {
    uint4 v[2];      // nibbles (16 bytes per chunk)
    uint4 ix;        // positions: chunk 0 in .x/.y, chunk 1 in .z/.w
    uint32_t sz[2];  // {s, z} of each chunk's group
};

template <>
struct TaskRegs<SGEMV_FMT_SPARSE14> {
    uint4 v;         // nibbles: chunk 0 in .x/.y, chunk 1 in .z/.w (8 bytes per chunk)
    uint2 ix;        // positions: chunk 0 in .x, chunk 1 in .y
    uint32_t sz[2];
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
    int nblk;          // 1024-column blocks in the tile (the last one may be partial)
    int nfull;         // complete 1024-column blocks
    int ntasks;
    __host__ __device__ void set(int prow0_, int prows_, int tc0_, int tcols_) {
        prow0 = prow0_;
        prows = prows_;
        tc0 = tc0_;
        tcols = tcols_;
        nblk = (tcols + kTaskCols - 1) / kTaskCols;
        nfull = tcols / kTaskCols;
        ntasks = ((prows + kRowsPerTask - 1) / kRowsPerTask) * nblk;
    }
};

// Warp w's contiguous run of tasks [begin, end).
__host__ __device__ __forceinline__ void warp_run(int ntasks, int w, int& begin, int& end) {
    begin = static_cast<int>((static_cast<long long>(ntasks) * w) / kWarps);
    end = static_cast<int>((static_cast<long long>(ntasks) * (w + 1)) / kWarps);
}

// The load side of a warp: the next task to load and lane (r, j)'s addresses for it. Within a quad the
// addresses advance by constant steps from one 1024-column block to the next; they are recomputed only
// when the quad changes.
template <int FMT>
struct Loader {
    // dense columns per byte of the vals and idx sections
    static constexpr uint32_t kValsCols = FMT == SGEMV_FMT_SPARSE24 ? 4 : (FMT == SGEMV_FMT_SPARSE14 ? 8 : 2);
    static constexpr uint32_t kIdxCols = FMT == SGEMV_FMT_SPARSE14 ? 16 : 8;
    static constexpr uint32_t kValsStep = kTaskCols / kValsCols;  // bytes per 1024-column block
    static constexpr uint32_t kIdxStep = kTaskCols / kIdxCols;
    int quad, blk;       // next task
    bool quad_full;      // all 4 rows of the quad are in the pass
    bool row_ok;         // this lane's row of the quad is in the pass
    const uint8_t* vp;   // vals at (row, tile column 1024 blk + 128 j)
    const uint8_t* ip;   // idx at the same column
    const uint8_t* sp0;  // {s, z} word of chunk 0's group
    const uint8_t* sp1;  // {s, z} word of chunk 1's group
    uint32_t gstep;      // bytes of {s, z} words per 1024 columns

    __host__ __device__ void set_quad(const GemvParams& p, const TaskSpace& ts, int row_begin, int r, int j, int q) {
        quad = q;
        blk = 0;
        const int rr = q * kRowsPerTask + r;
        quad_full = (q + 1) * kRowsPerTask <= ts.prows;
        row_ok = rr < ts.prows;
        const size_t grow = static_cast<size_t>(row_begin + ts.prow0 + (row_ok ? rr : 0));
        const uint32_t c0 = static_cast<uint32_t>(ts.tc0 + j * kLaneCols);
        vp = p.vals + grow * p.vals_pitch + c0 / kValsCols;
        ip = p.idx + grow * p.idx_pitch + c0 / kIdxCols;
        const uint8_t* srow = p.sz + grow * p.sz_pitch;
        sp0 = srow + ((c0 >> p.log2g) << 2);
        sp1 = srow + (((c0 + kChunkCols) >> p.log2g) << 2);
        gstep = static_cast<uint32_t>(kTaskCols >> p.log2g) << 2;
    }
    __host__ __device__ void start(const GemvParams& p, const TaskSpace& ts, int row_begin, int r, int j, int t) {
        const int q = t / ts.nblk;
        set_quad(p, ts, row_begin, r, j, q);
        const int b = t - q * ts.nblk;
        blk = b;
        vp += static_cast<uint32_t>(b) * kValsStep;
        ip += static_cast<uint32_t>(b) * kIdxStep;
        sp0 += static_cast<uint32_t>(b) * gstep;
        sp1 += static_cast<uint32_t>(b) * gstep;
    }
    __host__ __device__ void advance(const GemvParams& p, const TaskSpace& ts, int row_begin, int r, int j) {
        if (++blk == ts.nblk) {
            set_quad(p, ts, row_begin, r, j, quad + 1);
        } else {
            vp += kValsStep;
            ip += kIdxStep;
            sp0 += gstep;
            sp1 += gstep;
        }
    }
    // Fast path: every lane's row and both chunks exist (warp-uniform).
    __host__ __device__ bool full(const TaskSpace& ts) const { return quad_full && blk < ts.nfull; }
    // This lane's two chunks exist (row in the pass, columns inside the tile; the tile width is a
    // multiple of 128, so the two chunks exist together).
    __host__ __device__ bool lane_on(const TaskSpace& ts, int j) const {
        return row_ok && blk * kTaskCols + j * kLaneCols < ts.tcols;
    }
};

template <int FMT>
__device__ __forceinline__ void load_lane(const Loader<FMT>& ld, TaskRegs<FMT>& tr) {
    tr.sz[0] = ldg_stream_u32(ld.sp0);
    tr.sz[1] = ldg_stream_u32(ld.sp1);
    if constexpr (FMT == SGEMV_FMT_SPARSE24) {
        const U8 v = ldg_stream_v8(ld.vp);
        tr.v[0] = v.lo;
        tr.v[1] = v.hi;
        tr.ix = ldg_stream_v4(ld.ip);
    } else if constexpr (FMT == SGEMV_FMT_SPARSE14) {
        tr.v = ldg_stream_v4(ld.vp);
        tr.ix = ldg_stream_v2(ld.ip);
    } else {
        const U8 v0 = ldg_stream_v8(ld.vp);
        const U8 v1 = ldg_stream_v8(ld.vp + 32);
        tr.v[0][0] = v0.lo;
        tr.v[0][1] = v0.hi;
        tr.v[1][0] = v1.lo;
        tr.v[1][1] = v1.hi;
    }
}

// Load the loader's next task into tr and advance. Chunks that do not exist are zero: zero codes with a
// zero {s, z} word contribute exactly 0 against the zero padding of the x tile, so the compute side
// needs no bounds checks (lanes of rows outside the pass are dropped when the rows are flushed).
template <int FMT>
__device__ __forceinline__ void load_task(const GemvParams& p, const TaskSpace& ts, int row_begin, int r, int j,
                                          Loader<FMT>& ld, TaskRegs<FMT>& tr) {
    if (ld.full(ts) || ld.lane_on(ts, j)) {
        load_lane<FMT>(ld, tr);
    } else {
        tr.sz[0] = tr.sz[1] = 0;
        if constexpr (FMT == SGEMV_FMT_SPARSE24) {
            tr.v[0] = tr.v[1] = tr.ix = make_uint4(0, 0, 0, 0);
        } else if constexpr (FMT == SGEMV_FMT_SPARSE14) {
            tr.v = make_uint4(0, 0, 0, 0);
            tr.ix = make_uint2(0, 0);
        } else {
            tr.v[0][0] = tr.v[0][1] = tr.v[1][0] = tr.v[1][1] = make_uint4(0, 0, 0, 0);
        }
    }
    ld.advance(p, ts, row_begin, r, j);
}

// Both chunks of a task; xq = the x tile at the lane's 128 columns (batch row 0).
template <int FMT, int B>
__device__ __forceinline__ void compute_task(const TaskRegs<FMT>& tr, const uint8_t* xq, uint32_t xbs,
                                             float (&part)[B]) {
#pragma unroll
    for (int c = 0; c < 2; ++c) {
        const uint8_t* xp = xq + c * 128;
        if constexpr (FMT == SGEMV_FMT_SPARSE24)
            sparse_chunk<B>(tr.v[c], c ? make_uint2(tr.ix.z, tr.ix.w) : make_uint2(tr.ix.x, tr.ix.y), tr.sz[c], xp,
                            xbs, part);
        else if constexpr (FMT == SGEMV_FMT_SPARSE14)
            sparse14_chunk<B>(c ? make_uint2(tr.v.z, tr.v.w) : make_uint2(tr.v.x, tr.v.y), c ? tr.ix.y : tr.ix.x,
                              tr.sz[c], xp, xbs, part);
        else
            dense_chunk<B>(tr.v[c][0], tr.v[c][1], tr.sz[c], xp, xbs, part);
    }
}

// Combine the 8 column-lanes of each row and add the row sums into the shared accumulators
// (row = row within the pass; rows outside the pass, row >= prows, are dropped).
template <int B>
__device__ __forceinline__ void flush_rows(float* acc, int pass_rows, int row, int prows, int j, float (&part)[B]) {
#pragma unroll
    for (int b = 0; b < B; ++b) {
        float v = part[b];
        v += __shfl_xor_sync(0xFFFFFFFFu, v, 1);
        v += __shfl_xor_sync(0xFFFFFFFFu, v, 2);
        v += __shfl_xor_sync(0xFFFFFFFFu, v, 4);
        if (j == 0 && row < prows) atomicAdd(acc + b * pass_rows + row, v);
        part[b] = 0.0f;
    }
}

// Ask L2 to fetch the packed rows [row_begin, row_begin + rows) of every section of one layer: one
// warp, 32 KB requests spread over its lanes (a hint only: see prefetch_l2).
template <bool kSparse>
__device__ __forceinline__ void prefetch_layer(const GemvParams& p, int row_begin, int rows_, int lane) {
    const uint32_t rows = static_cast<uint32_t>(rows_);
    const uint8_t* base[3] = {p.vals + static_cast<size_t>(row_begin) * p.vals_pitch,
                              p.idx + static_cast<size_t>(row_begin) * p.idx_pitch,
                              p.sz + static_cast<size_t>(row_begin) * p.sz_pitch};
    const uint32_t bytes[3] = {rows * p.vals_pitch, kSparse ? rows * p.idx_pitch : 0u, rows * p.sz_pitch};
#pragma unroll
    for (int s = 0; s < 3; ++s) {
        if (bytes[s] == 0) continue;
        // widened to 16-byte boundaries (1:4 idx rows are only 8-byte aligned); sections start on
        // 256-byte boundaries and are zero-padded to 256 bytes, so the range stays in its section
        const uintptr_t a0 = reinterpret_cast<uintptr_t>(base[s]) & ~static_cast<uintptr_t>(15);
        const uintptr_t a1 = (reinterpret_cast<uintptr_t>(base[s]) + bytes[s] + 15) & ~static_cast<uintptr_t>(15);
        const uint32_t span = static_cast<uint32_t>(a1 - a0);
        for (uint32_t off = static_cast<uint32_t>(lane) * kPrefetchPiece; off < span; off += 32 * kPrefetchPiece)
            prefetch_l2(reinterpret_cast<const void*>(a0 + off), min(kPrefetchPiece, span - off));
    }
}

// The row range of row unit u of one layer: unit u < nctas owns rows [u*rows_base + min(u, rows_rem), ...
// + count); the units beyond the layer's own grid own none.
__host__ __device__ __forceinline__ void cta_rows(const GemvParams& p, int u, int& row_begin, int& nrows) {
    row_begin = u * p.rows_base + min(u, p.rows_rem);
    nrows = u < p.nctas ? p.rows_base + (u < p.rows_rem ? 1 : 0) : 0;
}

// The rows and columns CTA `cta` works on: the rows of its row unit (the CTA itself, or its cluster
// with split-K) and, with split-K, the cluster rank's balanced share of the 1024-column blocks of K
// (never empty: the planner splits only K with at least `split` blocks).
__host__ __device__ __forceinline__ void cta_work(const GemvParams& p, int cta, int& row_begin, int& nrows, int& kbeg,
                                                  int& kend) {
    const int unit = cta / p.split, rank = cta - unit * p.split;
    cta_rows(p, unit, row_begin, nrows);
    const int nb = (p.k + kTaskCols - 1) / kTaskCols;
    kbeg = (rank * nb / p.split) * kTaskCols;
    kend = min(p.k, ((rank + 1) * nb / p.split) * kTaskCols);
}

// One layer of a launch: this CTA's rows (all passes and x tiles). `waited_pdl` and `smem_in_use` carry
// over from layer to layer. With kSplit the CTAs of a cluster share their rows and split K (cta_work):
// each sums its columns into its own shared accumulators, and at the end of every pass cluster rank 0
// adds the ranks' sums in rank order through distributed shared memory and writes y, between two
// cluster barriers (deterministic, no scratch memory, no waits but barriers every CTA reaches).
template <int FMT, int B, bool kSplit>
__device__ __forceinline__ void run_layer(const GemvParams& p, int cta, int warp, int lane, uint8_t* smem,
                                          bool& waited_pdl, bool& smem_in_use) {
    constexpr int kPrefetch = prefetch_depth<B>();
    constexpr bool kSparse = (FMT != SGEMV_FMT_DENSE);  // x staged as byte planes
    const int r = lane >> 3;  // row of a task handled by this lane
    const int j = lane & 7;   // chunk column of a task handled by this lane
    int row_begin, nrows_cta, kbeg = 0, kend = p.k;
    if constexpr (kSplit)
        cta_work(p, cta, row_begin, nrows_cta, kbeg, kend);
    else
        cta_rows(p, cta, row_begin, nrows_cta);
    if (nrows_cta <= 0) return;  // the whole CTA (with split-K, its whole cluster) skips the layer

    float* acc = reinterpret_cast<float*>(smem + p.sm_acc);
    uint8_t* xs = smem + p.sm_x;
    const int ntile = (kend - kbeg + p.xt - 1) / p.xt;
    const int npass = (nrows_cta + p.pass_rows - 1) / p.pass_rows;

    for (int pass = 0; pass < npass; ++pass) {
        const int prow0 = pass * p.pass_rows;
        const int prows = min(p.pass_rows, nrows_cta - prow0);
        for (int tile = 0; tile < ntile; ++tile) {
            TaskSpace ts;
            ts.set(prow0, prows, kbeg + tile * p.xt, min(p.xt, kend - kbeg - tile * p.xt));
            int t_begin, t_end;
            warp_run(ts.ntasks, warp, t_begin, t_end);
            if (!waited_pdl) {
                // Everything this kernel reads (x, and the packed weights too: a packer may precede it)
                // may be written by the previous kernel in the stream.
                pdl_wait();
                waited_pdl = true;
            }
            // Warps 0..kXWarps-1 stage x (staged over nblk * 1024 columns, zero beyond the tile's tcols)
            // and zero the accumulators, then signal barrier 1; the other warps issue their weight loads
            // first and wait on barrier 1 only then. The weight loads can be held back by the memory
            // system's request limits, which must not delay x.
            if (smem_in_use) __syncthreads();  // the previous x tile / accumulators are no longer read
            smem_in_use = true;
            Loader<FMT> ld;
            TaskRegs<FMT> buf[kPrefetch];
            if (t_begin < t_end) ld.start(p, ts, row_begin, r, j, t_begin);
            if (warp >= kXWarps) {
#pragma unroll
                for (int q = 0; q < kPrefetch; ++q)
                    if (t_begin + q < t_end) load_task<FMT>(p, ts, row_begin, r, j, ld, buf[q]);
                named_bar_sync(1, kThreads);  // x tile and zeroed accumulators visible
            } else {
                if (tile == 0)
                    for (int i = threadIdx.x; i < B * p.pass_rows; i += kXThreads) acc[i] = 0.0f;
                const int units = ts.tcols / 8;                // 16-byte units of x per batch row
                const int punits = ts.nblk * (kTaskCols / 8);  // staged units per batch row
                const int nunits = B * punits;
                const uint4* xg = reinterpret_cast<const uint4*>(p.x + ts.tc0);
                for (int u0 = threadIdx.x; u0 < nunits; u0 += kXStageRegs * kXThreads) {
                    uint4 xr[kXStageRegs];
#pragma unroll
                    for (int q = 0; q < kXStageRegs; ++q) {
                        const int u = u0 + q * kXThreads;  // unit u: batch row u / punits
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
                            *reinterpret_cast<uint4*>(xs + b * p.x_b_stride + (v >> 4) * kXLaneBytes + (v & 15) * 16) =
                                kSparse ? byte_planes(xr[q]) : xr[q];
                        }
                    }
                }
                named_bar_sync(2, kXThreads);    // every staging thread's stores are done
                named_bar_arrive(1, kThreads);  // release the other warps
#pragma unroll
                for (int q = 0; q < kPrefetch; ++q)
                    if (t_begin + q < t_end) load_task<FMT>(p, ts, row_begin, r, j, ld, buf[q]);
            }

            float part[B];
#pragma unroll
            for (int b = 0; b < B; ++b) part[b] = 0.0f;
            int cquad = t_begin / ts.nblk;  // task being computed: (cquad, cblk)
            int cblk = t_begin - cquad * ts.nblk;
            const uint8_t* xq = xs + (cblk * (kTaskCols / kLaneCols) + j) * kXLaneBytes;
            for (int t0 = t_begin; t0 < t_end; t0 += kPrefetch) {
#pragma unroll
                for (int q = 0; q < kPrefetch; ++q) {
                    if (t0 + q < t_end) {
                        compute_task<FMT, B>(buf[q], xq, p.x_b_stride, part);
                        // refill the registers just consumed with the task kPrefetch ahead
                        if (t0 + q + kPrefetch < t_end) load_task<FMT>(p, ts, row_begin, r, j, ld, buf[q]);
                        xq += (kTaskCols / kLaneCols) * kXLaneBytes;
                        if (++cblk == ts.nblk) {  // warp-uniform: the quad's rows are done
                            flush_rows<B>(acc, p.pass_rows, cquad * kRowsPerTask + r, prows, j, part);
                            ++cquad;
                            cblk = 0;
                            xq = xs + j * kXLaneBytes;
                        }
                    }
                }
            }
            if (t_begin < t_end && cblk != 0) flush_rows<B>(acc, p.pass_rows, cquad * kRowsPerTask + r, prows, j, part);
        }
        __syncthreads();  // all partial sums of this pass are in `acc`
        if constexpr (kSplit) {
            cooperative_groups::cluster_group cl = cooperative_groups::this_cluster();
            cl.sync();  // every rank's sums of this pass are complete
            if (cl.block_rank() == 0) {
                for (int i = threadIdx.x; i < B * prows; i += kThreads) {
                    const int b = i / prows;
                    const int rr = i - b * prows;
                    float v = 0.0f;
                    for (int q = 0; q < p.split; ++q) v += cl.map_shared_rank(acc, q)[b * p.pass_rows + rr];
                    p.y[static_cast<size_t>(b) * p.n + row_begin + prow0 + rr] = __float2half_rn(v);
                }
            }
            cl.sync();  // rank 0 has read every rank's sums: they may be cleared or released
        } else {
            for (int i = threadIdx.x; i < B * prows; i += kThreads) {
                const int b = i / prows;
                const int rr = i - b * prows;
                p.y[static_cast<size_t>(b) * p.n + row_begin + prow0 + rr] = __float2half_rn(acc[b * p.pass_rows + rr]);
            }
        }
    }
}

// One launch runs a group of independent layers (same format and batch) one after the other: a CTA
// moves on to the next layer as soon as it has written its rows of the current one, so there is no
// launch gap and no tail between the layers of a group. Single-layer launches use the kMulti = false
// instance, whose parameters stay compile-time offsets into the kernel parameters (each instance holds
// one copy of the layer code).
template <int FMT, int B, bool kMulti, bool kSplit = false>
__global__ void __launch_bounds__(kThreads, 1) gemv_kernel(const __grid_constant__ LayerGroup g) {
    extern __shared__ __align__(128) uint8_t smem[];
    constexpr bool kSparse = (FMT != SGEMV_FMT_DENSE);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int cta = blockIdx.x;
    // The next kernel in the stream may be scheduled now; it reads its own inputs only after this
    // grid has completed (its own griddepcontrol.wait).
    pdl_launch_dependents();
    if (!kSplit && warp == kWarps - 1) {
        // While the previous kernel in the stream finishes, have L2 fetch the weights of this CTA's
        // first pass of the first layer (not with split-K, whose CTAs each read a slice of K).
        int rb, nr;
        cta_rows(g.layer[0], cta, rb, nr);
        if (nr > 0) prefetch_layer<kSparse>(g.layer[0], rb, min(nr, g.layer[0].pass_rows), lane);
    }
    bool waited_pdl = false;
    bool smem_in_use = false;  // shared memory holds a previous tile's x / a previous pass's sums
    if constexpr (!kMulti) {
        run_layer<FMT, B, kSplit>(g.layer[0], cta, warp, lane, smem, waited_pdl, smem_in_use);
    } else {
        // (prefetching the next layer's weights into L2 while a layer runs measured slower: its
        // requests compete with the current layer's loads)
        for (int layer = 0; layer < g.n_layers; ++layer)
            run_layer<FMT, B, false>(g.layer[layer], cta, warp, lane, smem, waited_pdl, smem_in_use);
    }
}

}  // namespace sgemv
