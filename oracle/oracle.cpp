// CPU oracle for the INT4 + 2:4 "2bit-CSR" SparseGemv.
//
// TEST INFRASTRUCTURE ONLY. This file is the plain, slow, obviously-correct statement of what the GPU
// library computes. It is used by the tests, by the smoke check and by the CPU baseline of the bench.
// The product never links, loads or calls it, and it shares no code with the CUDA path.
//
// Source of the method: the paper "Efficient LLM-based Advertising via Model Compression and Parallel
// Verification":
//   - group-wise INT4 weight-only quantisation, one group size per layer (§1 "Our Main Idea",
//     §3.2 "Adaptive Group-Wise Quantization");
//   - 2:4 and 1:4 semi-structured pruning by importance (§3.2 "Sparsification", Eq. 3 with a constant
//     activation norm and no gradient term, i.e. magnitude; Table 1 for the 1:4 tier);
//   - the 2bit-CSR index with uint16_t words in least-significant-first order (§1 Contributions,
//     §3.3 "Sparse Index Structure", §3.3 "Reduce Computational Burden");
//   - the decode-time product y = W x (§3.3 "Computational Acceleration").
// The byte layout and the readings of open points are those of the packed format, version 1.
//
// Every function follows the definition step by step, one element at a time:
//   pack    : prune each 4-block, quantise each group, write the sections;
//   dequant : read the sections back into a dense fp64 matrix;
//   gemv    : y[b][i] = sum over kept elements of (q - z) * s * x[b][col], in fp64.
//
// Arithmetic: binary32 IEEE operations for quantisation (compile with -ffp-contract=off), binary64
// for the product. The fp16 <-> binary32 conversions are written here from the IEEE 754 definition.
//
// Parity status: every function here is pinned by tests under tests/ (closed forms, invariants,
// brute force and exactly-representable cases); none is "parity unpinned".

#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>

#ifdef _OPENMP
#include <omp.h>
#endif

namespace {

// ---------------------------------------------------------------------------------------------
// Status codes (same numeric values as the library's; defined here on their own).
enum {
    ORC_OK = 0,
    ORC_ERR_ARG = -1,
    ORC_ERR_SHAPE = -2,
    ORC_ERR_FORMAT = -4,
    ORC_ERR_NONFINITE = -6,
};

enum { ORC_FMT_SPARSE24 = 1, ORC_FMT_DENSE = 2, ORC_FMT_SPARSE14 = 3 };

const uint32_t ORC_MAGIC = 0x564D4753u;  // bytes "SGMV"
const uint32_t ORC_VERSION = 1;

// ---------------------------------------------------------------------------------------------
// IEEE 754 binary16 <-> binary32, from the definition.

float half_bits_to_float(uint16_t h) {
    const uint32_t sign = (h >> 15) & 1u;
    const uint32_t exp = (h >> 10) & 0x1Fu;
    const uint32_t man = h & 0x3FFu;
    double mag;
    if (exp == 0) {
        mag = std::ldexp((double)man, -24);  // subnormal: man * 2^-24
    } else if (exp == 31) {
        if (man != 0) return std::nanf("");
        mag = INFINITY;
    } else {
        mag = std::ldexp((double)(1024u + man), (int)exp - 25);  // (1 + man/1024) * 2^(exp-15)
    }
    float f = (float)mag;  // exact: every binary16 value is a binary32 value
    return sign ? -f : f;
}

// Round a binary32 value to the nearest binary16 value, ties to even.
uint16_t float_to_half_bits(float f) {
    uint32_t u;
    std::memcpy(&u, &f, 4);
    const uint16_t sign = (uint16_t)((u >> 16) & 0x8000u);
    if (std::isnan(f)) return (uint16_t)(sign | 0x7E00u);
    double a = std::fabs((double)f);
    if (a == 0.0) return sign;
    // binary16: smallest subnormal 2^-24, largest finite 65504, spacing 2^(e-10) in [2^e, 2^(e+1)).
    int e;
    std::frexp(a, &e);            // a = m * 2^e, m in [0.5, 1)  =>  a in [2^(e-1), 2^e)
    int ulp_exp = (e - 1) - 10;   // spacing of binary16 numbers around a
    if (ulp_exp < -24) ulp_exp = -24;  // subnormal range has fixed spacing 2^-24
    double units = std::ldexp(a, -ulp_exp);  // exact: a scaled by a power of two
    double fl = std::floor(units);
    double rem = units - fl;
    double n;
    if (rem > 0.5) n = fl + 1.0;
    else if (rem < 0.5) n = fl;
    else n = (std::fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;  // tie: to even
    double r = std::ldexp(n, ulp_exp);
    if (r > 65504.0) return (uint16_t)(sign | 0x7C00u);  // overflow to infinity
    // encode r (exactly representable in binary16 now)
    if (r < std::ldexp(1.0, -14)) {
        uint16_t man = (uint16_t)std::ldexp(r, 24);  // subnormal (or 2^-14 exactly handled below)
        return (uint16_t)(sign | man);
    }
    int re;
    double rm = std::frexp(r, &re);  // r = rm * 2^re, rm in [0.5, 1)
    uint16_t exp = (uint16_t)(re - 1 + 15);
    uint16_t man = (uint16_t)(std::ldexp(rm, 11) - 1024.0);
    return (uint16_t)(sign | (exp << 10) | man);
}

// ---------------------------------------------------------------------------------------------
// Layout (packed format v1, sections 3 and 4).

struct Layout {
    int format;
    int64_t n, k, g;
    uint64_t vals_pitch, idx_pitch, sz_pitch;
    uint64_t off_vals, off_idx, off_sz, off_rowptr, total;
};

uint64_t round_up(uint64_t v, uint64_t m) { return (v + m - 1) / m * m; }

int make_layout(int format, int64_t n, int64_t k, int64_t g, Layout* L) {
    if (format != ORC_FMT_SPARSE24 && format != ORC_FMT_DENSE && format != ORC_FMT_SPARSE14)
        return ORC_ERR_FORMAT;
    if (n < 1 || n > (1 << 24)) return ORC_ERR_SHAPE;
    if (k < 128 || k > (1 << 20) || k % 128 != 0) return ORC_ERR_SHAPE;
    if (g != 64 && g != 128 && g != 256) return ORC_ERR_SHAPE;
    if (k % g != 0) return ORC_ERR_SHAPE;
    // row_ptr is int32 (section 7.4): its last entry, N times the kept elements of a row, must fit
    const int64_t kept = format == ORC_FMT_SPARSE24 ? k / 2 : (format == ORC_FMT_SPARSE14 ? k / 4 : 0);
    if (n * kept > INT32_MAX) return ORC_ERR_SHAPE;
    L->format = format;
    L->n = n;
    L->k = k;
    L->g = g;
    if (format == ORC_FMT_SPARSE24) {
        L->vals_pitch = (uint64_t)k / 4;  // K/2 kept nibbles
        L->idx_pitch = (uint64_t)k / 8;   // K/2 kept x 2 bits
    } else if (format == ORC_FMT_SPARSE14) {
        L->vals_pitch = (uint64_t)k / 8;  // K/4 kept nibbles
        L->idx_pitch = (uint64_t)k / 16;  // K/4 kept x 2 bits
    } else {
        L->vals_pitch = (uint64_t)k / 2;  // K nibbles
        L->idx_pitch = 0;
    }
    L->sz_pitch = round_up(4 * (uint64_t)(k / g), 16);
    uint64_t rowptr_bytes = (format == ORC_FMT_DENSE) ? 0 : 4 * (uint64_t)(n + 1);
    L->off_vals = 256;
    L->off_idx = L->off_vals + round_up((uint64_t)n * L->vals_pitch, 256);
    L->off_sz = L->off_idx + round_up((uint64_t)n * L->idx_pitch, 256);
    L->off_rowptr = L->off_sz + round_up((uint64_t)n * L->sz_pitch, 256);
    L->total = L->off_rowptr + round_up(rowptr_bytes, 256);
    return ORC_OK;
}

void put_u32(uint8_t* p, uint32_t v) { std::memcpy(p, &v, 4); }
void put_u64(uint8_t* p, uint64_t v) { std::memcpy(p, &v, 8); }
uint32_t get_u32(const uint8_t* p) { uint32_t v; std::memcpy(&v, p, 4); return v; }
uint64_t get_u64(const uint8_t* p) { uint64_t v; std::memcpy(&v, p, 8); return v; }

// Read and check the header of a packed buffer; fills L.
int read_header(const uint8_t* buf, uint64_t bytes, Layout* L) {
    if (buf == nullptr || bytes < 64) return ORC_ERR_ARG;
    if (get_u32(buf + 0) != ORC_MAGIC || get_u32(buf + 4) != ORC_VERSION) return ORC_ERR_FORMAT;
    int rc = make_layout((int)get_u32(buf + 8), get_u32(buf + 12), get_u32(buf + 16), get_u32(buf + 20), L);
    if (rc != ORC_OK) return rc;
    if (get_u64(buf + 24) != L->off_vals || get_u64(buf + 32) != L->off_idx ||
        get_u64(buf + 40) != L->off_sz || get_u64(buf + 48) != L->off_rowptr ||
        get_u64(buf + 56) != L->total)
        return ORC_ERR_FORMAT;
    if (bytes < L->total) return ORC_ERR_ARG;
    return ORC_OK;
}

// ---------------------------------------------------------------------------------------------
// Pruning (packed format v1, section 5): keep the two largest magnitudes of a 4-block, ties to the lower
// column; report the kept positions in ascending order.

void prune_block(const uint16_t w[4], int* p0, int* p1) {
    uint16_t mag[4];
    for (int i = 0; i < 4; ++i) mag[i] = (uint16_t)(w[i] & 0x7FFFu);  // |w| on the fp16 bits
    bool kept[4];
    for (int i = 0; i < 4; ++i) {
        int better = 0;  // how many elements rank ahead of element i
        for (int j = 0; j < 4; ++j) {
            if (j == i) continue;
            if (mag[j] > mag[i] || (mag[j] == mag[i] && j < i)) ++better;
        }
        kept[i] = better < 2;
    }
    int found = 0;
    for (int i = 0; i < 4; ++i) {
        if (!kept[i]) continue;
        if (found == 0) *p0 = i; else *p1 = i;
        ++found;
    }
}

// 1:4: keep the single best-ranked value of a 4-block (same ranking: magnitude, ties to the lower
// column).
int prune_block_1of4(const uint16_t w[4]) {
    int best = 0;
    for (int i = 1; i < 4; ++i)
        if ((w[i] & 0x7FFFu) > (w[best] & 0x7FFFu)) best = i;  // strictly larger: ties keep the lower
    return best;
}

// ---------------------------------------------------------------------------------------------
// Group quantisation (packed format v1, section 6). vals: the kept values of one group, as fp16 bits.

struct GroupQ {
    uint16_t s16, z16;
    std::vector<uint8_t> q;
};

GroupQ quantise_group(const std::vector<uint16_t>& vals) {
    float mn = 0.0f, mx = 0.0f;
    for (uint16_t h : vals) {
        float v = half_bits_to_float(h);
        if (v < mn) mn = v;
        if (v > mx) mx = v;
    }
    float r = mx - mn;
    uint16_t s16 = float_to_half_bits(r / 15.0f);
    if ((s16 & 0x7FFFu) == 0) s16 = 0x3C00u;  // 1.0
    float s = half_bits_to_float(s16);
    float zf = std::rint(-mn / s);
    if (zf < 0.0f) zf = 0.0f;
    if (zf > 15.0f) zf = 15.0f;
    int z = (int)zf;
    GroupQ out;
    out.s16 = s16;
    out.z16 = float_to_half_bits((float)z);
    for (uint16_t h : vals) {
        float v = half_bits_to_float(h);
        float qf = std::rint(v / s) + (float)z;
        if (qf < 0.0f) qf = 0.0f;
        if (qf > 15.0f) qf = 15.0f;
        out.q.push_back((uint8_t)(int)qf);
    }
    return out;
}

}  // namespace

extern "C" {

// binary16 <-> binary32 (exposed so the tests can pin them against an independent library).
float orc_half_to_float(uint16_t h) { return half_bits_to_float(h); }
uint16_t orc_float_to_half(float f) { return float_to_half_bits(f); }

// Section offsets and sizes. out[0..8] = vals_pitch, idx_pitch, sz_pitch, off_vals, off_idx,
// off_sz, off_rowptr, total_bytes, kept_per_row.
int orc_layout(int format, int64_t n, int64_t k, int64_t g, uint64_t* out) {
    Layout L;
    int rc = make_layout(format, n, k, g, &L);
    if (rc != ORC_OK) return rc;
    if (out == nullptr) return ORC_ERR_ARG;
    out[0] = L.vals_pitch;
    out[1] = L.idx_pitch;
    out[2] = L.sz_pitch;
    out[3] = L.off_vals;
    out[4] = L.off_idx;
    out[5] = L.off_sz;
    out[6] = L.off_rowptr;
    out[7] = L.total;
    out[8] = (format == ORC_FMT_SPARSE24) ? (uint64_t)k / 2 : (format == ORC_FMT_SPARSE14) ? (uint64_t)k / 4 : (uint64_t)k;
    return ORC_OK;
}

// Pack W (fp16 bits, [n][k] row-major) into out (out_bytes >= total). Every byte of out[0, total)
// is written.
int orc_pack(int format, int64_t n, int64_t k, int64_t g, const uint16_t* w, uint8_t* out,
             uint64_t out_bytes) {
    Layout L;
    int rc = make_layout(format, n, k, g, &L);
    if (rc != ORC_OK) return rc;
    if (w == nullptr || out == nullptr || out_bytes < L.total) return ORC_ERR_ARG;
    for (int64_t i = 0; i < n * k; ++i)
        if ((w[i] & 0x7C00u) == 0x7C00u) return ORC_ERR_NONFINITE;  // inf or NaN

    std::memset(out, 0, L.total);
    put_u32(out + 0, ORC_MAGIC);
    put_u32(out + 4, ORC_VERSION);
    put_u32(out + 8, (uint32_t)format);
    put_u32(out + 12, (uint32_t)n);
    put_u32(out + 16, (uint32_t)k);
    put_u32(out + 20, (uint32_t)g);
    put_u64(out + 24, L.off_vals);
    put_u64(out + 32, L.off_idx);
    put_u64(out + 40, L.off_sz);
    put_u64(out + 48, L.off_rowptr);
    put_u64(out + 56, L.total);

    const bool sparse = (format == ORC_FMT_SPARSE24);
    const bool sparse14 = (format == ORC_FMT_SPARSE14);
    std::vector<uint16_t> row(k);
    for (int64_t r = 0; r < n; ++r) {
        for (int64_t c = 0; c < k; ++c) {
            uint16_t h = w[r * k + c];
            row[c] = ((h & 0x7FFFu) == 0) ? (uint16_t)0 : h;  // -0 -> +0
        }
        // Kept elements of the row, in kept order, with their dense columns.
        std::vector<uint16_t> kv;
        std::vector<int64_t> kc;
        std::vector<int> kpos;  // in-block position (sparse only)
        for (int64_t t = 0; t < k / 4; ++t) {
            if (sparse) {
                int p0 = 0, p1 = 0;
                prune_block(&row[4 * t], &p0, &p1);
                kv.push_back(row[4 * t + p0]); kc.push_back(4 * t + p0); kpos.push_back(p0);
                kv.push_back(row[4 * t + p1]); kc.push_back(4 * t + p1); kpos.push_back(p1);
            } else if (sparse14) {
                int p = prune_block_1of4(&row[4 * t]);
                kv.push_back(row[4 * t + p]); kc.push_back(4 * t + p); kpos.push_back(p);
            } else {
                for (int p = 0; p < 4; ++p) { kv.push_back(row[4 * t + p]); kc.push_back(4 * t + p); }
            }
        }
        // Quantise group by group; a kept element belongs to the group of its dense column.
        std::vector<uint8_t> q(kv.size());
        uint8_t* sz_row = out + L.off_sz + (uint64_t)r * L.sz_pitch;
        std::vector<std::vector<size_t>> group_members((size_t)(k / g));
        for (size_t e = 0; e < kv.size(); ++e) group_members[(size_t)(kc[e] / g)].push_back(e);
        for (int64_t G = 0; G < k / g; ++G) {
            const std::vector<size_t>& members = group_members[(size_t)G];
            std::vector<uint16_t> gv;
            for (size_t e : members) gv.push_back(kv[e]);
            GroupQ gq = quantise_group(gv);
            for (size_t m = 0; m < members.size(); ++m) q[members[m]] = gq.q[m];
            uint32_t word = (uint32_t)gq.s16 | ((uint32_t)gq.z16 << 16);
            put_u32(sz_row + 4 * G, word);
        }
        // vals and idx words.
        uint8_t* vals_row = out + L.off_vals + (uint64_t)r * L.vals_pitch;
        if (sparse) {
            uint8_t* idx_row = out + L.off_idx + (uint64_t)r * L.idx_pitch;
            for (int64_t u = 0; u < k / 16; ++u) {  // word u: blocks 4u .. 4u+3
                uint32_t vw = 0;
                uint16_t iw = 0;
                for (int i = 0; i < 4; ++i) {
                    int64_t blk = 4 * u + i;
                    size_t e_first = (size_t)(2 * blk), e_second = (size_t)(2 * blk + 1);
                    vw |= (uint32_t)q[e_first] << (4 * i);
                    vw |= (uint32_t)q[e_second] << (4 * (i + 4));
                    iw |= (uint16_t)(kpos[e_first] << (2 * i));
                    iw |= (uint16_t)(kpos[e_second] << (8 + 2 * i));
                }
                put_u32(vals_row + 4 * u, vw);
                std::memcpy(idx_row + 2 * u, &iw, 2);
            }
        } else if (sparse14) {
            uint8_t* idx_row = out + L.off_idx + (uint64_t)r * L.idx_pitch;
            for (int64_t u = 0; u < k / 32; ++u) {  // word u: blocks 8u .. 8u+7, one kept each
                uint32_t vw = 0;
                uint16_t iw = 0;
                for (int i = 0; i < 8; ++i) {
                    size_t e = (size_t)(8 * u + i);
                    vw |= (uint32_t)q[e] << (4 * i);
                    iw |= (uint16_t)(kpos[e] << (2 * i));
                }
                put_u32(vals_row + 4 * u, vw);
                std::memcpy(idx_row + 2 * u, &iw, 2);
            }
        } else {
            for (int64_t u = 0; u < k / 8; ++u) {  // word u: columns 8u .. 8u+7
                uint32_t vw = 0;
                for (int i = 0; i < 4; ++i) {
                    vw |= (uint32_t)q[(size_t)(8 * u + 2 * i)] << (4 * i);
                    vw |= (uint32_t)q[(size_t)(8 * u + 2 * i + 1)] << (4 * (i + 4));
                }
                put_u32(vals_row + 4 * u, vw);
            }
        }
    }
    if (sparse || sparse14) {
        for (int64_t r = 0; r <= n; ++r) {
            int32_t v = (int32_t)(r * (sparse ? k / 2 : k / 4));
            std::memcpy(out + L.off_rowptr + 4 * r, &v, 4);
        }
    }
    return ORC_OK;
}

// ---------------------------------------------------------------------------------------------
// Decoding one kept element straight from the sections (packed format v1, section 7).

namespace {

struct Kept {
    int64_t col;
    int q;
};

// Kept element e (0-based, in kept order) of row r.
Kept kept_element(const uint8_t* buf, const Layout& L, int64_t r, int64_t e) {
    const uint8_t* vals_row = buf + L.off_vals + (uint64_t)r * L.vals_pitch;
    Kept out;
    if (L.format == ORC_FMT_SPARSE24) {
        int64_t blk = e / 2;
        int second = (int)(e % 2);
        int64_t u = blk / 4;
        int i = (int)(blk % 4);
        uint32_t vw = get_u32(vals_row + 4 * u);
        int slot = i + 4 * second;
        out.q = (int)((vw >> (4 * slot)) & 0xFu);
        uint16_t iw;
        std::memcpy(&iw, buf + L.off_idx + (uint64_t)r * L.idx_pitch + 2 * u, 2);
        int p = (int)((iw >> (2 * i + 8 * second)) & 3u);
        out.col = 4 * blk + p;
    } else if (L.format == ORC_FMT_SPARSE14) {
        int64_t blk = e;  // one kept element per block
        int64_t u = blk / 8;
        int i = (int)(blk % 8);
        uint32_t vw = get_u32(vals_row + 4 * u);
        out.q = (int)((vw >> (4 * i)) & 0xFu);
        uint16_t iw;
        std::memcpy(&iw, buf + L.off_idx + (uint64_t)r * L.idx_pitch + 2 * u, 2);
        int p = (int)((iw >> (2 * i)) & 3u);
        out.col = 4 * blk + p;
    } else {
        int64_t u = e / 8;
        int m = (int)(e % 8);  // column 8u + m
        int slot = (m % 2 == 0) ? m / 2 : m / 2 + 4;
        uint32_t vw = get_u32(vals_row + 4 * u);
        out.q = (int)((vw >> (4 * slot)) & 0xFu);
        out.col = e;
    }
    return out;
}

void group_params(const uint8_t* buf, const Layout& L, int64_t r, int64_t G, double* s, double* z) {
    uint32_t word = get_u32(buf + L.off_sz + (uint64_t)r * L.sz_pitch + 4 * G);
    *s = (double)half_bits_to_float((uint16_t)(word & 0xFFFFu));
    *z = (double)half_bits_to_float((uint16_t)(word >> 16));
}

int64_t kept_per_row(const Layout& L) {
    return L.format == ORC_FMT_SPARSE24 ? L.k / 2 : L.format == ORC_FMT_SPARSE14 ? L.k / 4 : L.k;
}

}  // namespace

// Dequantise a packed buffer into a dense fp64 matrix w_hat[n][k] (zeros at dropped positions).
int orc_dequant(const uint8_t* buf, uint64_t bytes, double* w_hat) {
    Layout L;
    int rc = read_header(buf, bytes, &L);
    if (rc != ORC_OK) return rc;
    if (w_hat == nullptr) return ORC_ERR_ARG;
    std::memset(w_hat, 0, sizeof(double) * (size_t)(L.n * L.k));
    for (int64_t r = 0; r < L.n; ++r) {
        for (int64_t e = 0; e < kept_per_row(L); ++e) {
            Kept kp = kept_element(buf, L, r, e);
            double s, z;
            group_params(buf, L, r, kp.col / L.g, &s, &z);
            w_hat[r * L.k + kp.col] += ((double)kp.q - z) * s;
        }
    }
    return ORC_OK;
}

// The unpacked representation used by the round-trip tests: q[n][kept], col[n][kept] (int32),
// s16/z16 [n][k/g].
int orc_unpack(const uint8_t* buf, uint64_t bytes, uint8_t* q, int32_t* col, uint16_t* s16,
               uint16_t* z16) {
    Layout L;
    int rc = read_header(buf, bytes, &L);
    if (rc != ORC_OK) return rc;
    int64_t kpr = kept_per_row(L);
    for (int64_t r = 0; r < L.n; ++r) {
        for (int64_t e = 0; e < kpr; ++e) {
            Kept kp = kept_element(buf, L, r, e);
            if (q) q[r * kpr + e] = (uint8_t)kp.q;
            if (col) col[r * kpr + e] = (int32_t)kp.col;
        }
        for (int64_t G = 0; G < L.k / L.g; ++G) {
            uint32_t word = get_u32(buf + L.off_sz + (uint64_t)r * L.sz_pitch + 4 * G);
            if (s16) s16[r * (L.k / L.g) + G] = (uint16_t)(word & 0xFFFFu);
            if (z16) z16[r * (L.k / L.g) + G] = (uint16_t)(word >> 16);
        }
    }
    return ORC_OK;
}

// y[b][rows[i]] for the listed rows (or all rows if rows == nullptr, nrows ignored):
//   y[b][r]      = sum_e (q_e - z) * s * x[b][col_e]        (binary64)
//   absdot[b][r] = sum_e |(q_e - z) * s * x[b][col_e]|      (for the tolerance)
// Output arrays are [batch][nr] where nr = nrows (or n). x is fp16 bits [batch][k].
int orc_gemv_rows(const uint8_t* buf, uint64_t bytes, const uint16_t* x, int batch,
                  const int32_t* rows, int64_t nrows, double* y, double* absdot, int nthreads) {
    Layout L;
    int rc = read_header(buf, bytes, &L);
    if (rc != ORC_OK) return rc;
    if (x == nullptr || y == nullptr || batch < 1) return ORC_ERR_ARG;
    int64_t nr = rows ? nrows : L.n;
    for (int64_t i = 0; rows && i < nr; ++i)
        if (rows[i] < 0 || rows[i] >= L.n) return ORC_ERR_ARG;
    std::vector<double> xd((size_t)batch * (size_t)L.k);
    for (size_t i = 0; i < xd.size(); ++i) xd[i] = (double)half_bits_to_float(x[i]);
    const int64_t kpr = kept_per_row(L);
    (void)nthreads;
#ifdef _OPENMP
    if (nthreads < 1) nthreads = 1;
#pragma omp parallel for schedule(dynamic, 4) num_threads(nthreads)
#endif
    for (int64_t i = 0; i < nr; ++i) {
        int64_t r = rows ? rows[i] : i;
        for (int b = 0; b < batch; ++b) {
            double acc = 0.0, aacc = 0.0;
            for (int64_t e = 0; e < kpr; ++e) {
                Kept kp = kept_element(buf, L, r, e);
                double s, z;
                group_params(buf, L, r, kp.col / L.g, &s, &z);
                double term = ((double)kp.q - z) * s * xd[(size_t)b * (size_t)L.k + (size_t)kp.col];
                acc += term;
                aacc += std::fabs(term);
            }
            y[(size_t)b * (size_t)nr + (size_t)i] = acc;
            if (absdot) absdot[(size_t)b * (size_t)nr + (size_t)i] = aacc;
        }
    }
    return ORC_OK;
}

int orc_gemv(const uint8_t* buf, uint64_t bytes, const uint16_t* x, int batch, double* y,
             double* absdot, int nthreads) {
    return orc_gemv_rows(buf, bytes, x, batch, nullptr, 0, y, absdot, nthreads);
}

int orc_openmp_available(void) {
#ifdef _OPENMP
    return 1;
#else
    return 0;
#endif
}

}  // extern "C"
