// GPU packer: fp16 W[N][K] -> INT4 + 2:4 or 1:4 "2bit-CSR" (or dense INT4), byte layout of packed format v1.
//
// This is the offline compression step of the paper "Efficient LLM-based Advertising via Model
// Compression and Parallel Verification": 2:4 or 1:4 semi-structured pruning by importance (§3.2
// "Sparsification", Eq. 3 in its magnitude-only form; Table 1 for the 1:4 tier), group-wise INT4 weight-only quantisation with a
// per-layer group size (§3.2 "Adaptive Group-Wise Quantization"), and the 2bit-CSR index with
// uint16_t words filled least-significant first (§3.3 "Sparse Index Structure", "Reduce Computational
// Burden").
//
// One thread handles 16 dense columns (4 blocks) of a row: it prunes the blocks, reduces min/max over
// the kept values of its group with warp shuffles (a group is g/16 consecutive lanes), quantises, and
// writes one nibble word + one position word (2:4), half a nibble word + one position byte (1:4) or
// two nibble words (dense). Arithmetic is
// IEEE binary32 with explicit round-to-nearest operations and no contraction (this file is compiled
// with -fmad=false), so the bytes are deterministic and match any other correct implementation of the
// same definition. min/max are order independent, so the thread layout cannot change the result.
#include "common.cuh"

namespace sgemv {

namespace {

__device__ __forceinline__ float h2f(uint16_t h) { return __half2float(__ushort_as_half(h)); }

// Rank-based top-2 of a 4-block: element i is kept iff fewer than two elements rank ahead of it
// (larger magnitude, or equal magnitude at a lower column).
__device__ __forceinline__ void prune_block(const uint16_t (&w)[4], int& p0, int& p1) {
    uint16_t m[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) m[i] = w[i] & 0x7FFFu;
    int found = 0;
    p0 = 0;
    p1 = 1;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        int ahead = 0;
#pragma unroll
        for (int jj = 0; jj < 4; ++jj)
            if (jj != i && (m[jj] > m[i] || (m[jj] == m[i] && jj < i))) ++ahead;
        if (ahead < 2) {
            if (found == 0) p0 = i; else p1 = i;
            ++found;
        }
    }
}

// 1:4: the single best-ranked element (largest magnitude, ties to the lower column).
__device__ __forceinline__ int prune_block_1of4(const uint16_t (&w)[4]) {
    int best = 0;
#pragma unroll
    for (int i = 1; i < 4; ++i)
        if ((w[i] & 0x7FFFu) > (w[best] & 0x7FFFu)) best = i;
    return best;
}

__device__ __forceinline__ int quantise(float v, float s, float z) {
    float q = __fadd_rn(rintf(__fdiv_rn(v, s)), z);
    q = fminf(fmaxf(q, 0.0f), 15.0f);
    return static_cast<int>(q);
}

__device__ void zero_bytes(uint8_t* base, uint64_t begin, uint64_t end) {
    for (uint64_t i = begin + blockIdx.x * blockDim.x + threadIdx.x; i < end;
         i += static_cast<uint64_t>(gridDim.x) * blockDim.x)
        base[i] = 0;
}

__global__ void __launch_bounds__(256) pack_kernel(const PackParams p) {
    const sgemv_layout& L = p.L;
    const int n = L.n, k = L.k, g = L.group;
    const bool sparse = (L.format == SGEMV_FMT_SPARSE24);
    const bool sparse14 = (L.format == SGEMV_FMT_SPARSE14);
    uint8_t* out = p.packed;

    // Header and the fixed regions: header words, header padding, section tails, row offsets.
    if (blockIdx.x == 0 && threadIdx.x < 16) {
        uint32_t hdr[16];
        hdr[0] = kMagic;
        hdr[1] = kVersion;
        hdr[2] = static_cast<uint32_t>(L.format);
        hdr[3] = static_cast<uint32_t>(n);
        hdr[4] = static_cast<uint32_t>(k);
        hdr[5] = static_cast<uint32_t>(g);
        const uint64_t offs[5] = {L.off_vals, L.off_idx, L.off_sz, L.off_rowptr, L.total_bytes};
        for (int i = 0; i < 5; ++i) {
            hdr[6 + 2 * i] = static_cast<uint32_t>(offs[i] & 0xFFFFFFFFu);
            hdr[7 + 2 * i] = static_cast<uint32_t>(offs[i] >> 32);
        }
        reinterpret_cast<uint32_t*>(out)[threadIdx.x] = hdr[threadIdx.x];
    }
    zero_bytes(out, 64, L.off_vals);
    zero_bytes(out, L.off_vals + static_cast<uint64_t>(n) * L.vals_pitch, L.off_idx);
    zero_bytes(out, L.off_idx + static_cast<uint64_t>(n) * L.idx_pitch, L.off_sz);
    zero_bytes(out, L.off_sz + static_cast<uint64_t>(n) * L.sz_pitch, L.off_rowptr);
    const uint64_t rowptr_bytes = (sparse || sparse14) ? 4ull * (n + 1) : 0ull;
    zero_bytes(out, L.off_rowptr + rowptr_bytes, L.total_bytes);
    if (sparse || sparse14) {
        int32_t* rp = reinterpret_cast<int32_t*>(out + L.off_rowptr);
        const int kept = sparse ? k / 2 : k / 4;
        for (int64_t r = blockIdx.x * blockDim.x + threadIdx.x; r <= n; r += static_cast<int64_t>(gridDim.x) * blockDim.x)
            rp[r] = static_cast<int32_t>(r * kept);
    }

    const int nchunks = k / 16;                // 16 dense columns per thread
    const int lanes_per_group = g / 16;        // 4, 8 or 16 consecutive lanes
    const uint32_t sz_row_bytes = 4u * static_cast<uint32_t>(k / g);
    bool nonfinite = false;

    for (int row = blockIdx.x; row < n; row += gridDim.x) {
        const uint16_t* wrow = p.w + static_cast<size_t>(row) * k;
        for (int c0 = 0; c0 < nchunks; c0 += blockDim.x) {
            const int c = c0 + threadIdx.x;
            const bool active = c < nchunks;  // whole groups are active or inactive together
            uint16_t h[16];
            if (active) {
                const uint4 a = reinterpret_cast<const uint4*>(wrow)[2 * c];
                const uint4 b = reinterpret_cast<const uint4*>(wrow)[2 * c + 1];
                const uint32_t u[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    h[2 * i] = static_cast<uint16_t>(u[i] & 0xFFFFu);
                    h[2 * i + 1] = static_cast<uint16_t>(u[i] >> 16);
                }
            } else {
#pragma unroll
                for (int i = 0; i < 16; ++i) h[i] = 0;
            }
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                if ((h[i] & 0x7C00u) == 0x7C00u) nonfinite = true;
                if ((h[i] & 0x7FFFu) == 0) h[i] = 0;  // -0 -> +0
            }
            // kept values in kept order; positions for the sparse index
            uint16_t kv[16];
            int pos[8];
            int nk;
            if (sparse) {
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                    const uint16_t blk[4] = {h[4 * t], h[4 * t + 1], h[4 * t + 2], h[4 * t + 3]};
                    int p0, p1;
                    prune_block(blk, p0, p1);
                    pos[2 * t] = p0;
                    pos[2 * t + 1] = p1;
                    kv[2 * t] = blk[p0];
                    kv[2 * t + 1] = blk[p1];
                }
                nk = 8;
            } else if (sparse14) {
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                    const uint16_t blk[4] = {h[4 * t], h[4 * t + 1], h[4 * t + 2], h[4 * t + 3]};
                    const int pb = prune_block_1of4(blk);
                    pos[t] = pb;
                    kv[t] = blk[pb];
                }
                nk = 4;
            } else {
#pragma unroll
                for (int i = 0; i < 16; ++i) kv[i] = h[i];
                nk = 16;
            }
            float mn = 0.0f, mx = 0.0f;
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                if (i < nk) {
                    const float v = h2f(kv[i]);
                    mn = fminf(mn, v);
                    mx = fmaxf(mx, v);
                }
            }
            for (int off = 1; off < lanes_per_group; off <<= 1) {
                mn = fminf(mn, __shfl_xor_sync(0xFFFFFFFFu, mn, off));
                mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, off));
            }
            const float rng = __fsub_rn(mx, mn);
            __half s16 = __float2half_rn(__fdiv_rn(rng, 15.0f));
            if ((__half_as_ushort(s16) & 0x7FFFu) == 0) s16 = __ushort_as_half(0x3C00u);
            const float s = __half2float(s16);
            float zf = rintf(__fdiv_rn(-mn, s));
            zf = fminf(fmaxf(zf, 0.0f), 15.0f);
            const int zi = static_cast<int>(zf);
            const float z = static_cast<float>(zi);
            if (!active) continue;
            const size_t rbase_v = L.off_vals + static_cast<size_t>(row) * L.vals_pitch;
            if (sparse) {
                uint32_t vw = 0;
                uint32_t iw = 0;
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                    vw |= static_cast<uint32_t>(quantise(h2f(kv[2 * t]), s, z)) << (4 * t);
                    vw |= static_cast<uint32_t>(quantise(h2f(kv[2 * t + 1]), s, z)) << (4 * (t + 4));
                    iw |= static_cast<uint32_t>(pos[2 * t]) << (2 * t);
                    iw |= static_cast<uint32_t>(pos[2 * t + 1]) << (8 + 2 * t);
                }
                *reinterpret_cast<uint32_t*>(out + rbase_v + 4 * static_cast<size_t>(c)) = vw;
                *reinterpret_cast<uint16_t*>(out + L.off_idx + static_cast<size_t>(row) * L.idx_pitch + 2 * static_cast<size_t>(c)) =
                    static_cast<uint16_t>(iw);
            } else if (sparse14) {
                // blocks 4c..4c+3: slots 4(c%2)..4(c%2)+3 of vals word c/2 (its 16-bit half c%2) and
                // bits 8(c%2)..8(c%2)+7 of idx word c/2 (its byte c%2)
                uint32_t vh = 0;
                uint32_t ib = 0;
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                    vh |= static_cast<uint32_t>(quantise(h2f(kv[t]), s, z)) << (4 * t);
                    ib |= static_cast<uint32_t>(pos[t]) << (2 * t);
                }
                *reinterpret_cast<uint16_t*>(out + rbase_v + 2 * static_cast<size_t>(c)) = static_cast<uint16_t>(vh);
                out[L.off_idx + static_cast<size_t>(row) * L.idx_pitch + static_cast<size_t>(c)] = static_cast<uint8_t>(ib);
            } else {
#pragma unroll
                for (int hw = 0; hw < 2; ++hw) {  // word 2c+hw: columns 16c + 8hw .. +7
                    uint32_t vw = 0;
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        vw |= static_cast<uint32_t>(quantise(h2f(kv[8 * hw + 2 * i]), s, z)) << (4 * i);
                        vw |= static_cast<uint32_t>(quantise(h2f(kv[8 * hw + 2 * i + 1]), s, z)) << (4 * (i + 4));
                    }
                    *reinterpret_cast<uint32_t*>(out + rbase_v + 8 * static_cast<size_t>(c) + 4 * hw) = vw;
                }
            }
            if ((threadIdx.x % lanes_per_group) == 0) {
                const uint32_t word = static_cast<uint32_t>(__half_as_ushort(s16)) |
                                      (static_cast<uint32_t>(__half_as_ushort(__float2half_rn(z))) << 16);
                *reinterpret_cast<uint32_t*>(out + L.off_sz + static_cast<size_t>(row) * L.sz_pitch +
                                             4 * static_cast<size_t>(c / lanes_per_group)) = word;
            }
        }
        // zero padding at the end of the row's sz entries
        for (uint32_t b = sz_row_bytes + threadIdx.x; b < L.sz_pitch; b += blockDim.x)
            out[L.off_sz + static_cast<size_t>(row) * L.sz_pitch + b] = 0;
    }
    if (nonfinite && p.status) atomicCAS(reinterpret_cast<int*>(p.status), 0, SGEMV_ERR_NONFINITE);
}

}  // namespace

cudaError_t launch_pack(const PackParams& p, int grid, cudaStream_t s) {
    pack_kernel<<<grid, 256, 0, s>>>(p);
    return cudaPeekAtLastError();
}

}  // namespace sgemv
