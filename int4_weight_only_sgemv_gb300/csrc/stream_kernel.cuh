// Streaming INT4 GEMV kernel for GB300 (sm_103a): the SparseGemv of the paper "Efficient LLM-based
// Advertising via Model Compression and Parallel Verification" (§3.3 "Revised Kernel") over the 2:4
// "2bit-CSR" format, and with the same skeleton over the 1:4 and dense INT4 formats.
//
// Work split (one persistent CTA of 16 warps per SM):
//   * CTA c owns a contiguous range of whole quads (4 rows) of every layer of the launch, q_base or
//     q_base + 1 of them; the CTAs that take the extra quad rotate from layer to layer, which evens out
//     the CTAs' work over the launch.
//   * The CTA's rows are taken four at a time (a quad) and cut into units of 64 bytes of nibbles: 256
//     columns for 2:4 and 1:4 (a 128-column half unit ends a row whose K is an odd multiple of 128), 128
//     for dense. A pair (quad, unit column) is the 4 units
//     of those columns in the quad's rows. The pairs of all layers of the launch form ONE flat list,
//     quad after quad, layer after layer; warp w takes pairs 8w .. 8w+7 of every round of 128 pairs, and
//     lane (r, j) = (lane / 8, lane % 8) the unit of row r of pair j. So the 4 row-lanes of a pair read
//     the same x (one shared-memory wavefront serves 4 lanes), every lane has the same number of units
//     (±1), and a lane's next unit follows from its current one by a few additions.
//   * Each unit's weights go straight from HBM into registers (256-bit streaming loads); the next unit
//     is in flight while the current one is computed. Nothing is read before the dependent-launch wait
//     (a packer or the previous layer may precede the kernel), but one warp first asks L2 to prefetch
//     the CTA's rows of the first layer, so they stream from HBM while the previous kernel finishes.
//   * x of every layer of the launch is staged once into shared memory (as byte planes, 16 bytes of
//     padding after every unit, so that the 8 unit columns a warp reads hit 8 different bank groups):
//     the paper's block-level cooperative activation load with a conflict-free layout (§3.3 "Accelerate
//     Memory Access"). Plain loads by every thread fetch it layer by layer; a launch of three or more
//     layers with short x rows (the kCopyX instance) has the copy engine fetch every layer's x at once
//     (one bulk copy per layer and batch row, one mbarrier) while the lanes issue their first weight
//     loads.
//   * A unit's fp32 sum goes to its own slot in shared memory. When every unit is done, each row's
//     slots are added in a fixed order (lane-strided sums, then a shuffle tree) and y is written once:
//     y does not depend on scheduling, run to run.
//
// Per 8 kept elements (one 32-bit word of nibbles, one 16-bit word of positions) and batch row:
//   * dequantisation (§3.3 "Reduce Computational Burden", lop3): one AND-OR per nibble pair gives
//     half2 {1024+q0, 1024+q1} (or 1024+16q for the odd nibbles), one HSUB2 removes 1024+z exactly;
//   * x sits in shared memory as byte planes (per 4-column block, the low bytes of x0..x3 in one 32-bit
//     word, the high bytes in the next), so the two 2-bit positions p0, p1 of a block become the
//     byte-permute selector (p0, p0+4, p1, p1+4) = (p0 + 256 p1) * 0x11 + 0x4040: one mask (which also
//     adds a fill constant) for two blocks, then one low or high product per block; one PRMT gathers the
//     block's two activations {x[p0], x[p1]};
//   * products (q - z) * x are exact in fp32 (mixed-precision FMA, fp16 sources, fp32 accumulate); the
//     group scale is applied once per group. The group size is a template parameter of the kernel: a
//     unit's {s, z} words are one 16-, 8- or 4-byte load.
// No tensor cores: a batch <= 8 GEMV is no dense contraction. The only waits are CTA barriers that every
// thread reaches and, in the kCopyX instance, the wait for the x copies, bounded by the global timer (a
// wait that gives up reports SGEMV_ERR_TIMEOUT), so the kernel cannot hang.
#pragma once

#include "gemv_kernel.cuh"

namespace sgemv {

// {s, z} word of a group -> s in fp32 and the half2 constants 1024 + z and 1024 + 16z.
__device__ __forceinline__ GroupParams group_params_nat(uint32_t szw) {
    GroupParams g;
    asm("{\n\t.reg .f16 s, z;\n\t.reg .b32 zz;\n\t"
        "mov.b32 {s, z}, %3;\n\t"
        "cvt.f32.f16 %0, s;\n\t"
        "mov.b32 zz, {z, z};\n\t"
        "add.rn.f16x2 %1, zz, %4;\n\t"
        "fma.rn.f16x2 %2, zz, %5, %4;\n\t}"
        : "=f"(g.s), "=r"(g.zA), "=r"(g.zB)
        : "r"(szw), "r"(0x64006400u), "r"(0x4C004C00u));
    return g;
}

// Per-layer numbers of this CTA, kept in shared memory (64 bytes).
struct CtaLayer {
    const uint8_t* vals;   // the CTA's first row of each section
    const uint8_t* idx;
    const uint8_t* sz;
    uint32_t vpitch, ipitch, spitch;
    uint32_t xoff;         // shared-memory offset of the layer's x (batch row 0)
    int full;              // complete units per row
    int nrows;             // the CTA's rows of the layer
    uint32_t pbase;        // first pair of the layer in the CTA's flat list
    int cpr, dq, dc;       // units per row; a lane's step in (quad, unit) per round
};
static_assert(sizeof(CtaLayer) == kCtaLayerBytes, "CtaLayer is read as four 16-byte words");

// Quads of the layer before CTA cta's (cta < nctas): q_base per CTA plus the extra quads of the CTAs
// before it in the rotated window [q_rot, q_rot + q_rem) mod nctas.
__host__ __device__ __forceinline__ int cta_quad_begin(const StreamLayer& L, int cta) {
    const int s = L.q_rot, n = L.nctas;
    const int first = min(max(cta - s, 0), min(L.q_rem, n - s));  // extras in [s, n) before cta
    const int wrap = min(cta, max(0, s + L.q_rem - n));             // extras in [0, s + q_rem - n)
    return cta * L.q_base + first + wrap;
}
__host__ __device__ __forceinline__ int cta_row_begin(const StreamLayer& L, int cta) {
    return 4 * cta_quad_begin(L, cta);
}
// Rows of the layer that CTA cta owns (0 for cta >= nctas; the CTA holding the last quad may own fewer
// than 4 per quad).
__host__ __device__ __forceinline__ int cta_nrows(const StreamLayer& L, int cta) {
    if (cta >= L.nctas) return 0;
    int d = cta - L.q_rot;
    if (d < 0) d += L.nctas;
    const int quads = L.q_base + (d < L.q_rem ? 1 : 0);
    return min(4 * quads, L.n - cta_row_begin(L, cta));
}

// The CTA's rows and first pair of every layer; tab has n_layers + 1 entries (the last holds only pbase,
// the CTA's total number of pairs).
__host__ __device__ __forceinline__ void build_table(const StreamGroup& g, int cta, CtaLayer* tab) {
    uint32_t pb = 0;
    for (int l = 0; l < g.n_layers; ++l) {
        const StreamLayer& L = g.layer[l];
        CtaLayer e;
        e.nrows = cta_nrows(L, cta);
        const size_t rb = static_cast<size_t>(e.nrows > 0 ? cta_row_begin(L, cta) : 0);
        e.vals = L.vals + rb * L.vals_pitch;
        e.idx = L.idx + rb * L.idx_pitch;
        e.sz = L.sz + rb * L.sz_pitch;
        e.vpitch = L.vals_pitch;
        e.ipitch = L.idx_pitch;
        e.spitch = L.sz_pitch;
        e.xoff = L.xoff;
        e.full = L.full;
        e.pbase = pb;
        e.cpr = L.cpr;
        e.dq = L.dq;
        e.dc = L.dc;
        pb += static_cast<uint32_t>(((e.nrows + 3) / 4) * L.cpr);
        tab[l] = e;
    }
    CtaLayer end = {};
    end.pbase = pb;
    tab[g.n_layers] = end;
}

// A lane's position in the flat pair list, with the current layer's stepping constants.
struct PairCursor {
    uint32_t p;            // flat pair index
    uint32_t pend;         // end of the current layer's pairs
    int l;                 // layer
    int q, c;              // quad within the CTA's rows of layer l, unit column
    int cpr, dq, dc;
};

__host__ __device__ __forceinline__ void cursor_set(int n_layers, const CtaLayer* tab, uint32_t p, PairCursor& cu) {
    cu.p = p;
    int l = 0;
    while (l + 1 < n_layers && p >= tab[l + 1].pbase) ++l;
    const CtaLayer& e = tab[l];
    cu.l = l;
    cu.pend = tab[l + 1].pbase;
    cu.cpr = e.cpr;
    cu.dq = e.dq;
    cu.dc = e.dc;
    const uint32_t o = p - e.pbase;
    const uint32_t cpr = static_cast<uint32_t>(e.cpr);
    cu.q = static_cast<int>(o / cpr);
    cu.c = static_cast<int>(o - static_cast<uint32_t>(cu.q) * cpr);
}

// The lane's next pair, kPairsPerRound further in the flat list. Called only when that pair exists, so
// the layer switch always finds a layer.
__host__ __device__ __forceinline__ void cursor_advance(int n_layers, const CtaLayer* tab, PairCursor& cu) {
    cu.p += kPairsPerRound;
    cu.c += cu.dc;
    cu.q += cu.dq;
    if (cu.c >= cu.cpr) {
        cu.c -= cu.cpr;
        ++cu.q;
    }
    if (cu.p >= cu.pend) cursor_set(n_layers, tab, cu.p, cu);  // next layer (rare)
}

// Where lane row r's unit of the pair at the cursor lives: its nibbles, positions and first {s, z} word
// in global memory, its x in shared memory (batch row 0), its sum slot. h2 is the byte offset of the
// second half of the unit's nibbles (half of it for the positions): half the unit, or 0 for the half unit
// that ends a row with K % 256 == 128 (sparse formats), whose second half then re-reads the first,
// harmlessly: x is zero there. A row beyond the CTA's rows (the last quad may be short) loads the CTA's
// last row and has no slot.
struct UnitAddr {
    const uint8_t* vp;
    const uint8_t* ip;
    const uint8_t* sp;
    uint32_t xo;
    uint32_t slot;         // r * pstride + pair, or kNoSlot
    uint32_t h2;
};
constexpr uint32_t kNoSlot = 0xFFFFFFFFu;

// Per-format geometry of a unit: every unit holds 64 bytes of nibbles.
template <int FMT>
struct StreamFmt {
    static constexpr int kCols = stream_unit_cols(FMT);        // 256 (2:4, 1:4) or 128 (dense)
    static constexpr uint32_t kVB = FMT == SGEMV_FMT_SPARSE14 ? 32u : 64u;  // nibble bytes per unit
    static constexpr uint32_t kIB = FMT == SGEMV_FMT_SPARSE24 ? 32u : (FMT == SGEMV_FMT_SPARSE14 ? 16u : 0u);
    static constexpr int kChunks = kCols / 64;                 // 64-column chunks per unit
    static constexpr uint32_t kXU = stream_x_unit_bytes(FMT);  // x bytes of a unit in shared memory
    static constexpr bool kPlanes = FMT != SGEMV_FMT_DENSE;    // x staged as byte planes
};

// {s, z} words of a unit: 4, 2 or 1 for g = 64, 128, 256 with 256-column units; 2, 1, 1 with 128-column
// units (two consecutive units then share a g = 256 word).
template <int FMT, int LG>
__host__ __device__ constexpr int unit_groups() {
    return (StreamFmt<FMT>::kCols >> LG) > 0 ? (StreamFmt<FMT>::kCols >> LG) : 1;
}

template <int FMT, int LG>
__host__ __device__ __forceinline__ UnitAddr unit_addr(const CtaLayer& e, const PairCursor& cu, int r,
                                                       uint32_t pstride) {
    using F = StreamFmt<FMT>;
    const int row = 4 * cu.q + r;
    const bool ok = row < e.nrows;
    const uint32_t rr = static_cast<uint32_t>(ok ? row : e.nrows - 1);
    const uint32_t c = static_cast<uint32_t>(cu.c);
    UnitAddr a;
    a.vp = e.vals + static_cast<size_t>(rr) * e.vpitch + c * F::kVB;
    a.ip = e.idx + static_cast<size_t>(rr) * e.ipitch + c * F::kIB;
    a.sp = e.sz + static_cast<size_t>(rr) * e.spitch + (((c * F::kCols) >> LG) << 2);
    a.xo = e.xoff + c * F::kXU;
    a.slot = ok ? static_cast<uint32_t>(r) * pstride + cu.p : kNoSlot;
    a.h2 = cu.c < e.full ? F::kVB / 2 : 0u;
    return a;
}

// Registers of one unit.
template <int FMT, int LG>
struct UnitRegs {
    uint4 v[StreamFmt<FMT>::kVB / 16];                          // nibbles
    uint4 ix[StreamFmt<FMT>::kIB > 0 ? StreamFmt<FMT>::kIB / 16 : 1];  // positions (sparse formats)
    uint32_t sz[unit_groups<FMT, LG>()];                        // {s, z} word of each group
    uint32_t xo;                                                 // shared-memory offset of the unit's x
    uint32_t slot;
};

// Loads lane row r's unit of the pair at the cursor. Nibble rows are 32-byte (2:4, dense) or 16-byte
// (1:4) aligned, position rows 16-byte (2:4) or 8-byte (1:4) aligned, {s, z} rows 16-byte aligned; a half
// unit's 16- or 8-byte {s, z} load reaches into the row's zero padding, which the sz pitch, rounded up to
// 16 bytes, always holds (g = 256 has no half units: K is then a multiple of 256).
template <int FMT, int LG>
__device__ __forceinline__ void load_unit(const CtaLayer* tab, const PairCursor& cu, int r, uint32_t pstride,
                                          UnitRegs<FMT, LG>& t) {
    const CtaLayer e = tab[cu.l];
    const UnitAddr a = unit_addr<FMT, LG>(e, cu, r, pstride);
    t.xo = a.xo;
    t.slot = a.slot;
    if constexpr (FMT == SGEMV_FMT_SPARSE14) {
        t.v[0] = ldg_stream_v4(a.vp);
        t.v[1] = ldg_stream_v4(a.vp + a.h2);
        const uint2 i0 = ldg_stream_v2(a.ip);
        const uint2 i1 = ldg_stream_v2(a.ip + (a.h2 >> 1));
        t.ix[0] = make_uint4(i0.x, i0.y, i1.x, i1.y);
    } else {
        const U8 v0 = ldg_stream_v8(a.vp);
        const U8 v1 = ldg_stream_v8(a.vp + a.h2);
        t.v[0] = v0.lo;
        t.v[1] = v0.hi;
        t.v[2] = v1.lo;
        t.v[3] = v1.hi;
        if constexpr (FMT == SGEMV_FMT_SPARSE24) {
            t.ix[0] = ldg_stream_v4(a.ip);
            t.ix[1] = ldg_stream_v4(a.ip + (a.h2 >> 1));
        }
    }
    constexpr int NG = unit_groups<FMT, LG>();
    if constexpr (NG == 4) {
        const uint4 q = ldg_stream_v4(a.sp);
        t.sz[0] = q.x;
        t.sz[1] = q.y;
        t.sz[2] = q.z;
        t.sz[3] = q.w;
    } else if constexpr (NG == 2) {
        const uint2 q = ldg_stream_v2(a.sp);
        t.sz[0] = q.x;
        t.sz[1] = q.y;
    } else {
        t.sz[0] = ldg_stream_u32(a.sp);
    }
}

// One 64-column chunk (32 kept) of a 2:4 row for every batch row, added into accA (even blocks) and
// accB (odd blocks, scaled by 16). x stored as byte planes.
template <int B>
__device__ __forceinline__ void chunk24(const uint4 v, const uint32_t i0, const uint32_t i1, const GroupParams& gp,
                                        const uint8_t* xp, const uint32_t xbs, float (&accA)[B], float (&accB)[B]) {
    const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
    const uint32_t i2[2] = {i0, i1};
#pragma unroll
    for (int u = 0; u < 2; ++u) {
        // i2[u]: positions of vals words 2u (low 16 bits) and 2u+1 (high 16 bits)
        // (a low or high product without an addend: the fill constant supplies the 0x4040)
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
}

// One 64-column chunk (16 blocks, 16 kept) of a 1:4 row, added into accA / accB (x16).
//   w0, w1: nibbles (word h: blocks 8h .. 8h+7, one per slot); ix: the 16 blocks' positions.
// Selectors: m_t = fields of blocks t, 4+t, 8+t, 12+t (bytes 0..3) plus the fill constant; byte k of
// m_t * 0x11 is the selector (nibbles p, p+4) for block 4k+t, brought down to bits 0-7 by the low or a
// high product (prmt reads only its low nibbles here: one activation per block).
template <int B>
__device__ __forceinline__ void chunk14(const uint32_t w0, const uint32_t w1, const uint32_t ix, const GroupParams& gp,
                                        const uint8_t* xp, const uint32_t xbs, float (&accA)[B], float (&accB)[B]) {
    uint32_t S[4][4];  // [t][k]: selector of block 4k+t
#pragma unroll
    for (int t = 0; t < 4; ++t) {
        const uint32_t m = and_or(ix >> (2 * t), 0x03030303u, kSelFill);
        S[t][0] = sel_lo(m);
        S[t][1] = __umulhi(m, 0x11000000u);
        S[t][2] = __umulhi(m, 0x00110000u);
        S[t][3] = __umulhi(m, 0x00001100u);
    }
    const uint32_t w2[2] = {w0, w1};
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        uint32_t d[4];  // d[i] = {q of block 8h+i, q of block 8h+i+4} - z (x16 for odd i)
        dequant_word(w2[h], gp.zA, gp.zB, d);
#pragma unroll
        for (int b = 0; b < B; ++b) {
            const uint8_t* xw = xp + b * xbs + 64 * h;  // 16-byte pieces 4h..4h+3: blocks 8h..8h+7
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
}

// One 64-column chunk of a dense row, added into accA / accB (x16). va = columns 0..31, vb = 32..63;
// x stored as fp16.
template <int B>
__device__ __forceinline__ void chunkd(const uint4 va, const uint4 vb, const GroupParams& gp, const uint8_t* xp,
                                       const uint32_t xbs, float (&accA)[B], float (&accB)[B]) {
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
}

template <int FMT, int B, int LG>
__device__ __forceinline__ void compute_unit(const UnitRegs<FMT, LG>& t, const uint8_t* smem, uint32_t xbs,
                                             float (&part)[B]) {
    constexpr int NG = unit_groups<FMT, LG>();
    constexpr int CPG = StreamFmt<FMT>::kChunks / NG;  // chunks per group
    const uint8_t* xp = smem + t.xo;
#pragma unroll
    for (int grp = 0; grp < NG; ++grp) {
        const GroupParams gp = group_params_nat(t.sz[grp]);
        float accA[B], accB[B];
#pragma unroll
        for (int b = 0; b < B; ++b) accA[b] = accB[b] = 0.0f;
#pragma unroll
        for (int ch = 0; ch < CPG; ++ch) {
            const int k = grp * CPG + ch;
            if constexpr (FMT == SGEMV_FMT_SPARSE24) {
                const uint4 ixk = t.ix[k >> 1];
                chunk24<B>(t.v[k], (k & 1) ? ixk.z : ixk.x, (k & 1) ? ixk.w : ixk.y, gp, xp + 128 * k, xbs, accA, accB);
            } else if constexpr (FMT == SGEMV_FMT_SPARSE14) {
                const uint4 vk = t.v[k >> 1];
                const uint32_t ixw = k == 0 ? t.ix[0].x : (k == 1 ? t.ix[0].y : (k == 2 ? t.ix[0].z : t.ix[0].w));
                chunk14<B>((k & 1) ? vk.z : vk.x, (k & 1) ? vk.w : vk.y, ixw, gp, xp + 128 * k, xbs, accA, accB);
            } else {
                chunkd<B>(t.v[2 * k], t.v[2 * k + 1], gp, xp + 128 * k, xbs, accA, accB);
            }
        }
#pragma unroll
        for (int b = 0; b < B; ++b) part[b] = fmaf(gp.s, fmaf(accB[b], 0.0625f, accA[b]), part[b]);
    }
}

// The copy-engine form of stage_x (launches of several layers): thread 0 has issued one bulk copy of
// each layer's x per batch row into the raw buffer at xraw_off; every thread waits for them (bounded:
// a wait that gives up stores SGEMV_ERR_TIMEOUT in the status word and x is then invalid) and moves its
// pieces from the raw buffer into the unit layout below.
template <int FMT, int B>
__device__ __forceinline__ void stage_x_from_raw(const StreamGroup& g, uint8_t* smem) {
    using F = StreamFmt<FMT>;
    constexpr int kPU = F::kCols / 8;  // 16-byte pieces per unit
    if (!mbar_wait(reinterpret_cast<uint64_t*>(smem + g.xbar_off), 0) && g.status)
        atomicExch(g.status, SGEMV_ERR_TIMEOUT);
    uint32_t ro = g.xraw_off;
    for (int l = 0; l < g.n_layers; ++l) {
        const StreamLayer& L = g.layer[l];
        const int per_row = L.cpr * kPU;
        const int kp = L.k / 8;
        for (int b = 0; b < B; ++b) {
            const uint4* src = reinterpret_cast<const uint4*>(smem + ro);
            for (int v = threadIdx.x; v < per_row; v += kThreads) {
                const uint4 q = v < kp ? src[v] : make_uint4(0, 0, 0, 0);
                *reinterpret_cast<uint4*>(smem + L.xoff + b * g.xbs + (v / kPU) * F::kXU + (v % kPU) * 16) =
                    F::kPlanes ? byte_planes(q) : q;
            }
            ro += 2u * static_cast<uint32_t>(L.k);
        }
    }
}

// x of every layer into shared memory: 16-byte pieces (sparse formats: two 4-column blocks as byte
// planes; dense: 8 fp16), unit c of batch row b of layer l at b * xbs + xoff + c * kXU; zero beyond K up
// to the end of the last unit.
template <int FMT, int B>
__device__ __forceinline__ void stage_x(const StreamGroup& g, uint8_t* smem) {
    using F = StreamFmt<FMT>;
    constexpr int kPU = F::kCols / 8;  // 16-byte pieces per unit
    for (int l = 0; l < g.n_layers; ++l) {
        const StreamLayer& L = g.layer[l];
        const int per_row = L.cpr * kPU;  // 16-byte pieces per batch row, padded to whole units
        const int kp = L.k / 8;
        const uint4* xg = reinterpret_cast<const uint4*>(L.x);
        uint8_t* xs = smem + L.xoff;
#pragma unroll
        for (int b = 0; b < B; ++b) {
            for (int v0 = threadIdx.x; v0 < per_row; v0 += 4 * kThreads) {
                uint4 rg[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int v = v0 + q * kThreads;
                    rg[q] = v < kp ? __ldg(xg + static_cast<size_t>(b) * kp + v) : make_uint4(0, 0, 0, 0);
                }
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int v = v0 + q * kThreads;
                    if (v < per_row)
                        *reinterpret_cast<uint4*>(xs + b * g.xbs + (v / kPU) * F::kXU + (v % kPU) * 16) =
                            F::kPlanes ? byte_planes(rg[q]) : rg[q];
                }
            }
        }
    }
}

// kCopyX: x arrives by the copy engine (the plan's xraw_off is set); a separate instance, so that the
// launches that stage x with plain loads keep their code as it is.
template <int FMT, int B, int LG, bool kCopyX>
__global__ void __launch_bounds__(kThreads, 1) stream_kernel(const __grid_constant__ StreamGroup g) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int cta = blockIdx.x;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int r = lane >> 3;  // row of the pair handled by this lane
    const int j = lane & 7;   // pair of the warp's 8
    // The next kernel in the stream may be scheduled now; it reads its own inputs only after this
    // grid has completed (its own griddepcontrol.wait).
    pdl_launch_dependents();
    CtaLayer* tab = reinterpret_cast<CtaLayer*>(smem + g.tab_off);
    uint64_t* xbar = reinterpret_cast<uint64_t*>(smem + g.xbar_off);
    if (threadIdx.x == 0) {
        build_table(g, cta, tab);
        if constexpr (kCopyX) {
            mbar_init(xbar, 1);
            mbar_fence_init();
        }
    }
    if (warp == kWarps - 1) {
        // While the previous kernel in the stream finishes, have L2 fetch the rows of this CTA's first
        // round of the first layer (a hint without architectural effect: nothing is read before the wait
        // below). Prefetching more floods the memory system just when x and the first units are needed.
        const StreamLayer& L = g.layer[0];
        const int nr = cta_nrows(L, cta);
        if (nr > 0) {
            GemvParams p;
            p.vals = L.vals;
            p.idx = L.idx;
            p.sz = L.sz;
            p.vals_pitch = L.vals_pitch;
            p.idx_pitch = L.idx_pitch;
            p.sz_pitch = L.sz_pitch;
            const int nq = (1 * kPairsPerRound + L.cpr - 1) / L.cpr;  // quads of the first rounds
            prefetch_layer<FMT != SGEMV_FMT_DENSE>(p, cta_row_begin(L, cta), min(nr, 4 * nq), lane);
        }
    }
    __syncthreads();  // the layer table
    const int nl = g.n_layers;
    const uint32_t ptotal = tab[nl].pbase;
    // Everything this kernel reads (x, and the packed weights too: a packer may precede it) may be
    // written by the previous kernel in the stream.
    pdl_wait();

    // The lane's units: pairs p0, p0 + 128, ... below ptotal, row r of each. Two register buffers: the
    // next unit is in flight while the current one is computed.
    const uint32_t p0 = static_cast<uint32_t>(8 * warp + j);
    const int n = p0 < ptotal ? static_cast<int>((ptotal - p0 + kPairsPerRound - 1) / kPairsPerRound) : 0;
    // x first: every unit needs it, and its loads would otherwise queue behind the weight loads. With
    // several layers the copy engine fetches every layer's x at once (one bulk copy per layer and batch
    // row) while the lanes issue their first weight loads.
    PairCursor cu;
    UnitRegs<FMT, LG> buf[2];
    if constexpr (kCopyX) {
        if (threadIdx.x == 0) {
            mbar_arrive_expect_tx(xbar, g.xraw_bytes);
            uint32_t ro = g.xraw_off;
            for (int l = 0; l < nl; ++l) {
                const StreamLayer& L = g.layer[l];
                for (int b = 0; b < B; ++b) {
                    bulk_g2s(smem + ro, L.x + static_cast<size_t>(b) * L.k, 2u * static_cast<uint32_t>(L.k), xbar);
                    ro += 2u * static_cast<uint32_t>(L.k);
                }
            }
        }
    } else {
        stage_x<FMT, B>(g, smem);
    }
    if (n > 0) {
        cursor_set(nl, tab, p0, cu);
        load_unit<FMT, LG>(tab, cu, r, g.pstride, buf[0]);
    }
    if constexpr (kCopyX) stage_x_from_raw<FMT, B>(g, smem);
    __syncthreads();  // x staged

    float* part = reinterpret_cast<float*>(smem + g.part_off);
    const uint32_t bstride = 4u * g.pstride;
    auto finish = [&](const UnitRegs<FMT, LG>& t) {
        float acc[B];
#pragma unroll
        for (int b = 0; b < B; ++b) acc[b] = 0.0f;
        compute_unit<FMT, B, LG>(t, smem, g.xbs, acc);
        if (t.slot != kNoSlot) {
#pragma unroll
            for (int b = 0; b < B; ++b) part[b * bstride + t.slot] = acc[b];
        }
    };
    int i = 0;
    for (; i + 2 <= n; i += 2) {
        cursor_advance(nl, tab, cu);
        load_unit<FMT, LG>(tab, cu, r, g.pstride, buf[1]);
        finish(buf[0]);
        if (i + 2 < n) {
            cursor_advance(nl, tab, cu);
            load_unit<FMT, LG>(tab, cu, r, g.pstride, buf[0]);
        }
        finish(buf[1]);
    }
    if (i < n) finish(buf[0]);
    __syncthreads();  // every unit sum is in shared memory

    // Row sums in a fixed order: 8 lanes per row (4 rows per warp), lane jj adds the row's units jj,
    // jj + 8, ..., then a 3-step shuffle tree.
    int nrow_all = 0;
    for (int l = 0; l < nl; ++l) nrow_all += tab[l].nrows;
    const int jj = lane & 7;
    for (int i0 = 4 * warp; i0 < nrow_all; i0 += 4 * kWarps) {
        const int i = i0 + (lane >> 3);
        int l = 0, rr = i;
        while (l < nl - 1 && rr >= tab[l].nrows) {
            rr -= tab[l].nrows;
            ++l;
        }
        const bool on = i < nrow_all;
        const CtaLayer& e = tab[l];
        const uint32_t base =
            static_cast<uint32_t>(rr & 3) * g.pstride + e.pbase + static_cast<uint32_t>((rr >> 2) * e.cpr);
#pragma unroll
        for (int b = 0; b < B; ++b) {
            float v = 0.0f;
            if (on)
                for (int c = jj; c < e.cpr; c += 8) v += part[b * bstride + base + c];
            v += __shfl_xor_sync(0xFFFFFFFFu, v, 4);
            v += __shfl_xor_sync(0xFFFFFFFFu, v, 2);
            v += __shfl_xor_sync(0xFFFFFFFFu, v, 1);
            if (on && jj == 0) {
                const StreamLayer& L = g.layer[l];
                L.y[static_cast<size_t>(b) * L.n + cta_row_begin(L, cta) + rr] = __float2half_rn(v);
            }
        }
    }
}

}  // namespace sgemv
