// Streaming INT4 GEMV kernel for GB300 (sm_103a): the SparseGemv of the paper "Efficient LLM-based
// Advertising via Model Compression and Parallel Verification" (§3.3 "Revised Kernel") over the 2:4
// "2bit-CSR" format (and, with the same skeleton, the 1:4 and dense INT4 formats).
//
// Work split (one persistent CTA of 16 warps per SM):
//   * CTA c owns a contiguous, balanced range of output rows of every layer of the launch (±1 row).
//   * The CTA's rows x K are cut into units of 256 columns (one 128-column half unit ends a row whose K
//     is an odd multiple of 128); the units of all layers of the launch form ONE flat list, row after
//     row, layer after layer. Lane L of the CTA takes units L, L + 512, L + 1024, ... so every round of
//     the CTA reads one contiguous stretch of each section (32 KB of nibbles per round for 2:4), every
//     lane has the same number of units (±1), and the addresses of a lane's next unit follow from its
//     current one by a few additions.
//   * Each unit's weights go straight from HBM into registers (256-bit streaming loads), the next
//     unit's while the current one is computed. Nothing is read before the dependent-launch wait (a
//     packer or the previous layer may precede the kernel), but one warp first asks L2 to prefetch the
//     CTA's rows of the first layer, so they stream from HBM while the previous kernel finishes.
//   * x of every layer of the launch is staged once into shared memory (fp16 as stored, 16 bytes of
//     padding after every 512, so that the 32 lanes of a warp, which read consecutive units, hit 8
//     different bank groups): the paper's block-level cooperative activation load with a conflict-free
//     layout (§3.3 "Accelerate Memory Access").
//   * A unit's fp32 sum goes to its own slot in shared memory. When every unit is done, each row's
//     slots are added in a fixed order (lane-strided sums, then a shuffle tree) and y is written once:
//     y does not depend on scheduling, run to run.
//
// Per 8 kept elements (one 32-bit word of nibbles, one 16-bit word of positions) and batch row:
//   * dequantisation (§3.3 "Reduce Computational Burden", lop3): one AND-OR per nibble pair gives
//     half2 {1024+q0, 1024+q1} (or 1024+16q for the odd nibbles), one HSUB2 removes 1024+z exactly;
//   * the two 2-bit positions p0, p1 of a block become the byte-permute selector (2p0, 2p0+1, 2p1,
//     2p1+1) = (p0 + 256 p1) * 0x22 + 0x1010: one mask for two blocks, then one multiply-add (low or
//     high product) per block; one PRMT gathers the block's two activations {x[p0], x[p1]};
//   * products (q - z) * x are exact in fp32 (mixed-precision FMA, fp16 sources, fp32 accumulate); the
//     group scale is applied once per 64 columns.
// No tensor cores: a batch <= 8 GEMV is no dense contraction. The only waits on other threads are CTA
// barriers that every thread reaches, so the kernel cannot hang.
#pragma once

#include "gemv_kernel.cuh"

namespace sgemv {

// Selector of the block whose positions sit in bits 0-1 (p0) and 8-9 (p1) of m, for x stored as
// fp16 pairs {x0, x1}, {x2, x3}: nibbles (2p0, 2p0+1, 2p1, 2p1+1).
__device__ __forceinline__ uint32_t sel_nat_lo(uint32_t m) {
    uint32_t d;
    asm("mad.lo.u32 %0, %1, 0x22, 0x1010;" : "=r"(d) : "r"(m));
    return d;
}
// The same for the block whose positions sit in bits 16-17 and 24-25: hi32(m * 0x220000) is exactly
// (p0 + 256 p1) * 0x22, since the low block's fields add less than 2^16 * 0x220000 / 2^32.
__device__ __forceinline__ uint32_t sel_nat_hi(uint32_t m) {
    uint32_t d;
    asm("mad.hi.u32 %0, %1, 0x220000, 0x1010;" : "=r"(d) : "r"(m));
    return d;
}

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

// Per-layer numbers of this CTA, kept in shared memory.
struct CtaLayer {
    int row_begin, nrows;
    uint32_t ubase;        // first unit of the layer in the CTA's flat list
};

// A lane's position in the flat unit list.
struct UnitCursor {
    uint32_t u;            // flat unit index
    uint32_t uend;         // end of the current layer's units
    int l;                 // layer
    int r, c;              // row within the CTA's rows of layer l, unit within the row
};

// The CTA's rows and first unit of every layer; tab has n_layers + 1 entries (the last holds only ubase,
// the CTA's total number of units).
__host__ __device__ __forceinline__ void build_table(const StreamGroup& g, int cta, CtaLayer* tab) {
    uint32_t ub = 0;
    for (int l = 0; l < g.n_layers; ++l) {
        const StreamLayer& L = g.layer[l];
        CtaLayer e;
        e.row_begin = cta * L.rows_base + min(cta, L.rows_rem);
        e.nrows = cta < L.nctas ? L.rows_base + (cta < L.rows_rem ? 1 : 0) : 0;
        e.ubase = ub;
        ub += static_cast<uint32_t>(e.nrows * L.cpr);
        tab[l] = e;
    }
    tab[g.n_layers].row_begin = tab[g.n_layers].nrows = 0;
    tab[g.n_layers].ubase = ub;
}

__host__ __device__ __forceinline__ void cursor_set(const StreamGroup& g, const CtaLayer* tab, uint32_t utotal,
                                                    uint32_t u, UnitCursor& cu) {
    cu.u = u;
    int l = 0;
    while (l + 1 < g.n_layers && u >= tab[l + 1].ubase) ++l;
    cu.l = l;
    cu.uend = l + 1 < g.n_layers ? tab[l + 1].ubase : utotal;
    const uint32_t q = u - tab[l].ubase;
    const uint32_t cpr = static_cast<uint32_t>(g.layer[l].cpr);
    cu.r = static_cast<int>(q / cpr);
    cu.c = static_cast<int>(q - static_cast<uint32_t>(cu.r) * cpr);
}

__host__ __device__ __forceinline__ void cursor_advance(const StreamGroup& g, const CtaLayer* tab, uint32_t utotal,
                                                        UnitCursor& cu) {
    const uint32_t u = cu.u + kThreads;
    if (u >= cu.uend) {
        if (u < utotal) cursor_set(g, tab, utotal, u, cu);
        else cu.u = u;
        return;
    }
    const StreamLayer& L = g.layer[cu.l];
    cu.u = u;
    cu.c += L.dc;
    cu.r += L.dr;
    if (cu.c >= L.cpr) {
        cu.c -= L.cpr;
        ++cu.r;
    }
}

// Registers of one unit (2:4): 256 columns = 4 chunks of 64 columns (32 kept each).
struct UnitRegs24 {
    uint4 v[4];            // nibbles: chunk k in v[k] (4 words)
    uint4 ix[2];           // positions: chunk k in 32-bit words 2k, 2k+1 (ix[k/2].{x,y} or .{z,w})
    uint32_t sz[4];        // {s, z} word of each chunk's group
    uint32_t xo;           // shared-memory offset of the unit's x (batch row 0)
    uint32_t slot;         // unit index (its sum goes to slot b * ustride + slot)
};

// Where the unit at the cursor lives: its nibbles, positions and chunk-0 {s, z} word in global memory,
// its x in shared memory (batch row 0); full = false for the half unit that ends a row with
// K % 256 == 128.
struct UnitAddr {
    const uint8_t* vp;
    const uint8_t* ip;
    const uint8_t* sp;
    uint32_t xo;
    bool full;
};
__host__ __device__ __forceinline__ UnitAddr unit_addr(const StreamGroup& g, const CtaLayer* tab, const UnitCursor& cu) {
    const StreamLayer& L = g.layer[cu.l];
    const size_t row = static_cast<size_t>(tab[cu.l].row_begin + cu.r);
    const uint32_t c = static_cast<uint32_t>(cu.c);
    UnitAddr a;
    a.vp = L.vals + row * L.vals_pitch + c * 64u;
    a.ip = L.idx + row * L.idx_pitch + c * 32u;
    a.sp = L.sz + row * L.sz_pitch + (((c * kUnitCols) >> L.log2g) << 2);
    a.xo = L.xoff + c * kXUnitBytes;
    a.full = cu.c < L.full;
    return a;
}

// Loads the unit at the cursor. Nibble rows are 32-byte aligned (K/4 bytes, K a multiple of 128),
// position rows only 16-byte aligned (K/8 bytes). A half unit leaves its second half zero: zero codes
// with a zero {s, z} word contribute exactly 0 against the zero x padding.
__device__ __forceinline__ void load_unit24(const StreamGroup& g, const CtaLayer* tab, const UnitCursor& cu,
                                            UnitRegs24& t) {
    const StreamLayer& L = g.layer[cu.l];
    const UnitAddr a = unit_addr(g, tab, cu);
    t.xo = a.xo;
    t.slot = cu.u;
    const U8 v0 = ldg_stream_v8(a.vp);
    t.v[0] = v0.lo;
    t.v[1] = v0.hi;
    t.ix[0] = ldg_stream_v4(a.ip);
    t.sz[0] = ldg_stream_u32(a.sp);
    t.sz[1] = ldg_stream_u32(a.sp + L.so1);
    if (a.full) {
        const U8 v1 = ldg_stream_v8(a.vp + 32);
        t.v[2] = v1.lo;
        t.v[3] = v1.hi;
        t.ix[1] = ldg_stream_v4(a.ip + 16);
        t.sz[2] = ldg_stream_u32(a.sp + L.so2);
        t.sz[3] = ldg_stream_u32(a.sp + L.so3);
    } else {
        t.v[2] = t.v[3] = make_uint4(0, 0, 0, 0);
        t.ix[1] = make_uint4(0, 0, 0, 0);
        t.sz[2] = t.sz[3] = 0;
    }
}

// One 64-column chunk (32 kept) of a 2:4 row for every batch row, added into part[b]. x stored as fp16.
template <int B>
__device__ __forceinline__ void chunk24(const uint4 v, const uint32_t i0, const uint32_t i1, const uint32_t szw,
                                        const uint8_t* xp, const uint32_t xbs, float (&part)[B]) {
    const GroupParams gp = group_params_nat(szw);
    float accA[B], accB[B];
#pragma unroll
    for (int b = 0; b < B; ++b) accA[b] = accB[b] = 0.0f;
    const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
    const uint32_t i2[2] = {i0, i1};
#pragma unroll
    for (int u = 0; u < 2; ++u) {
        // i2[u]: positions of vals words 2u (low 16 bits) and 2u+1 (high 16 bits)
        uint32_t S[2][4];
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            const uint32_t m = (i2[u] >> (2 * t)) & 0x03030303u;
            S[0][t] = sel_nat_lo(m);
            S[1][t] = sel_nat_hi(m);
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

template <int B>
__device__ __forceinline__ void compute_unit24(const UnitRegs24& t, const uint8_t* smem, uint32_t xbs,
                                               float (&part)[B]) {
    const uint8_t* xp = smem + t.xo;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const uint4 ixk = t.ix[k >> 1];
        const uint32_t i0 = (k & 1) ? ixk.z : ixk.x;
        const uint32_t i1 = (k & 1) ? ixk.w : ixk.y;
        chunk24<B>(t.v[k], i0, i1, t.sz[k], xp + 128 * k, xbs, part);
    }
}

// x of every layer into shared memory: 16-byte pieces, unit c of batch row b of layer l at
// b * xbs + xoff + c * 528; zero beyond K up to the end of the last unit.
template <int B>
__device__ __forceinline__ void stage_x(const StreamGroup& g, uint8_t* smem) {
    for (int l = 0; l < g.n_layers; ++l) {
        const StreamLayer& L = g.layer[l];
        const int per_row = L.cpr * (kUnitCols / 8);  // 16-byte pieces per batch row, padded to whole units
        const int kp = L.k / 8;
        const int total = B * per_row;
        const uint4* xg = reinterpret_cast<const uint4*>(L.x);
        for (int i0 = threadIdx.x; i0 < total; i0 += 4 * kThreads) {
            uint4 r[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int i = i0 + q * kThreads;
                const int b = (B == 1) ? 0 : i / per_row;
                const int v = i - b * per_row;
                r[q] = make_uint4(0, 0, 0, 0);
                if (i < total && v < kp) r[q] = __ldg(xg + static_cast<size_t>(b) * kp + v);
            }
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int i = i0 + q * kThreads;
                if (i < total) {
                    const int b = (B == 1) ? 0 : i / per_row;
                    const int v = i - b * per_row;
                    *reinterpret_cast<uint4*>(smem + b * g.xbs + L.xoff + (v >> 5) * kXUnitBytes + (v & 31) * 16) = r[q];
                }
            }
        }
    }
}

template <int FMT, int B>
__global__ void __launch_bounds__(kThreads, 1) stream_kernel(const __grid_constant__ StreamGroup g) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int cta = blockIdx.x;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // The next kernel in the stream may be scheduled now; it reads its own inputs only after this
    // grid has completed (its own griddepcontrol.wait).
    pdl_launch_dependents();
    CtaLayer* tab = reinterpret_cast<CtaLayer*>(smem + g.tab_off);
    if (threadIdx.x == 0) build_table(g, cta, tab);
    if (warp == kWarps - 1) {
        // While the previous kernel in the stream finishes, have L2 fetch this CTA's rows of the first
        // layer (a hint without architectural effect: nothing is read before the wait below).
        const StreamLayer& L = g.layer[0];
        const int rb = cta * L.rows_base + min(cta, L.rows_rem);
        const int nr = cta < L.nctas ? L.rows_base + (cta < L.rows_rem ? 1 : 0) : 0;
        if (nr > 0) {
            GemvParams p;
            p.vals = L.vals;
            p.idx = L.idx;
            p.sz = L.sz;
            p.vals_pitch = L.vals_pitch;
            p.idx_pitch = L.idx_pitch;
            p.sz_pitch = L.sz_pitch;
            prefetch_layer<FMT != SGEMV_FMT_DENSE>(p, rb, nr, lane);
        }
    }
    __syncthreads();  // the layer table
    const uint32_t utotal = tab[g.n_layers].ubase;
    // Everything this kernel reads (x, and the packed weights too: a packer may precede it) may be
    // written by the previous kernel in the stream.
    pdl_wait();

    // Two register buffers: the next unit is in flight while the current one is computed.
    UnitCursor cu;
    UnitRegs24 buf[2];
    const uint32_t u0 = static_cast<uint32_t>(threadIdx.x);
    const bool any = u0 < utotal;
    if (any) {
        cursor_set(g, tab, utotal, u0, cu);
        load_unit24(g, tab, cu, buf[0]);
        cursor_advance(g, tab, utotal, cu);
    }
    stage_x<B>(g, smem);
    __syncthreads();  // x staged

    float* part = reinterpret_cast<float*>(smem + g.part_off);
    if (any) {
        for (;;) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const bool more = cu.u < utotal;
                if (more) {
                    load_unit24(g, tab, cu, buf[h ^ 1]);
                    cursor_advance(g, tab, utotal, cu);
                }
                float acc[B];
#pragma unroll
                for (int b = 0; b < B; ++b) acc[b] = 0.0f;
                compute_unit24<B>(buf[h], smem, g.xbs, acc);
#pragma unroll
                for (int b = 0; b < B; ++b) part[b * g.ustride + buf[h].slot] = acc[b];
                if (!more) goto done;
            }
        }
    }
done:
    __syncthreads();  // every unit sum is in shared memory

    // Row sums in a fixed order: lane j adds units j, j+32, ... of the row, then a shuffle tree.
    int nrow_all = 0;
    for (int l = 0; l < g.n_layers; ++l) nrow_all += tab[l].nrows;
    for (int i = warp; i < nrow_all; i += kWarps) {
        int l = 0, r = i;
        while (r >= tab[l].nrows) {
            r -= tab[l].nrows;
            ++l;
        }
        const StreamLayer& L = g.layer[l];
        const uint32_t base = tab[l].ubase + static_cast<uint32_t>(r * L.cpr);
#pragma unroll
        for (int b = 0; b < B; ++b) {
            float v = 0.0f;
            for (int c = lane; c < L.cpr; c += 32) v += part[b * g.ustride + base + c];
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
            if (lane == 0) L.y[static_cast<size_t>(b) * L.n + tab[l].row_begin + r] = __float2half_rn(v);
        }
    }
}

}  // namespace sgemv
