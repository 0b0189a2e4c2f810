// Host-only check of the streaming GEMV kernel's index arithmetic, built with the library's own planner
// (plan_stream), CTA table (build_table), pair cursor (cursor_set, cursor_advance) and unit addresses
// (unit_addr), for the 2:4, 1:4 and dense formats, single layers and groups of layers over ragged and
// full-size shapes and seeded random groups, every group size and batch 1..3 (larger batches run the
// tiled kernel). For every CTA and every one of its 512 lanes it walks the lane's units exactly as the
// kernel does and checks that:
//   * every unit of every row of every layer is visited exactly once, by the CTA that owns the row, and
//     rows beyond the CTA's rows (a short last quad) load an existing row and store no sum;
//   * every weight load (per unit 64 bytes of nibbles in two loads, the positions in two, and one 16-, 8-
//     or 4-byte {s, z} load) stays inside its row and section with its vector width's alignment, and
//     brings the words of the unit's own columns and groups;
//   * the unit's x (512 bytes per batch row) and its sum slot stay inside their shared-memory regions,
//     the row sums read exactly the slots the units wrote, and the regions (x, layer table, unit sums,
//     and for groups of layers the copy engine's raw x and its mbarrier) do not overlap and fit the
//     device, with every x copy 16-byte aligned.
// No GPU is needed: the device code is compiled but never launched (tests/host/stub_launchers.cu).
#include <cstdio>
#include <cstdlib>
#include <vector>

#include "stream_kernel.cuh"

using namespace sgemv;

static int fails = 0;
static int g_copy_x = 0;  // groups whose x the copy engine fetches
static uint32_t g_max_pairs = 0;  // pairs of the busiest CTA in the last walk
#define CHECK(c, ...) do { if (!(c)) { if (fails < 20) { printf("FAIL %s:%d: ", __FILE__, __LINE__); printf(__VA_ARGS__); printf("\n"); } ++fails; } } while (0)

struct Shape {
    int n, k, g;
};
static int g_fmt = SGEMV_FMT_SPARSE24;  // format of the groups being checked

// Shared memory of a streaming launch, restated: x of every layer (528 bytes per 256-column unit and
// batch row), the layer table (9 entries of 64 bytes), then fp32 unit sums [B][4 rows][pairs] for the CTA
// with most pairs.
static uint64_t smem_needed(const std::vector<Shape>& shapes, int B) {
    auto r16 = [](uint64_t v) { return (v + 15) / 16 * 16; };
    const uint64_t uc = g_fmt == SGEMV_FMT_DENSE ? 128 : 256;
    uint64_t x = 0, pairs = 0;
    for (const Shape& s : shapes) {
        const uint64_t cpr = (s.k + uc - 1) / uc, nq = (s.n + 3) / 4, ctas = nq < 152 ? nq : 152;
        x += cpr * (2 * uc + 16);
        pairs += (nq / ctas + (nq % ctas ? 1 : 0)) * cpr;  // quads of the busiest CTA
    }
    return r16(r16(B * x) + 9 * 64) + 4ull * B * 4 * ((pairs + 3) / 4 * 4);
}

template <int FMT, int LG>
static void walk(const StreamGroup& g, const std::vector<Shape>& shapes, const std::vector<sgemv_layout>& L,
                 const std::vector<sgemv_layer>& table, int B, int grid) {
    const int nl = static_cast<int>(shapes.size());
    const uint64_t x_end = static_cast<uint64_t>(B) * g.xbs;
    std::vector<std::vector<int>> cov(nl), rowcov(nl);
    for (int i = 0; i < nl; ++i) {
        cov[i].assign(static_cast<size_t>(shapes[i].n) * g.layer[i].cpr, 0);
        rowcov[i].assign(shapes[i].n, 0);
    }
    std::vector<CtaLayer> tab(kStreamMaxLayers + 1);
    g_max_pairs = 0;
    for (int cta = 0; cta < 152; ++cta) {
        build_table(g, cta, tab.data());
        const uint32_t ptotal = tab[nl].pbase;
        g_max_pairs = std::max(g_max_pairs, ptotal);
        CHECK(ptotal <= g.pstride, "pairs %u > pstride %u", ptotal, g.pstride);
        for (int l = 0; l < nl; ++l) {
            const CtaLayer& e = tab[l];
            const int rb = cta_row_begin(g.layer[l], cta);
            CHECK(e.nrows == 0 || (e.nrows > 0 && rb + e.nrows <= shapes[l].n), "cta rows");
            if (cta >= grid) CHECK(e.nrows == 0, "CTA beyond the grid owns rows");
            for (int r = 0; r < e.nrows; ++r) rowcov[l][rb + r] += 1;
            if (cta == 0 && l == 0 && e.nrows > 0) {
                // the L2 prefetch ranges of the first layer, widened to 16 bytes, stay inside their sections
                const uint64_t begins[3] = {L[0].off_vals + rb * L[0].vals_pitch, L[0].off_idx + rb * L[0].idx_pitch,
                                            L[0].off_sz + rb * L[0].sz_pitch};
                const uint64_t lens[3] = {e.nrows * L[0].vals_pitch, e.nrows * L[0].idx_pitch, e.nrows * L[0].sz_pitch};
                const uint64_t lo[3] = {L[0].off_vals, L[0].off_idx, L[0].off_sz};
                const uint64_t hi[3] = {L[0].off_idx, L[0].off_sz, L[0].off_rowptr};
                for (int q = 0; q < 3; ++q) {
                    const uint64_t a0 = begins[q] & ~15ull, a1 = (begins[q] + lens[q] + 15) & ~15ull;
                    CHECK(a0 >= lo[q] && a1 <= hi[q], "prefetch range %d", q);
                }
            }
        }
        std::vector<int> slotcov(static_cast<size_t>(4) * g.pstride, 0);
        for (int warp = 0; warp < kWarps; ++warp)
            for (int lane = 0; lane < 32; ++lane) {
                const int r = lane >> 3, j = lane & 7;
                const uint32_t p0 = static_cast<uint32_t>(8 * warp + j);
                const int n = p0 < ptotal ? static_cast<int>((ptotal - p0 + kPairsPerRound - 1) / kPairsPerRound) : 0;
                PairCursor cu;
                if (n > 0) cursor_set(nl, tab.data(), p0, cu);
                for (int i = 0; i < n; ++i) {
                    const uint32_t p = p0 + static_cast<uint32_t>(i) * kPairsPerRound;
                    CHECK(cu.p == p && p < ptotal, "cursor p %u expected %u", cu.p, p);
                    int l = 0;
                    while (l + 1 < nl && p >= tab[l + 1].pbase) ++l;
                    const int cpr = g.layer[l].cpr;
                    const int q = static_cast<int>((p - tab[l].pbase) / cpr), c = static_cast<int>((p - tab[l].pbase) % cpr);
                    CHECK(cu.l == l && cu.q == q && cu.c == c, "cursor (l %d q %d c %d) expected (%d %d %d)", cu.l, cu.q,
                          cu.c, l, q, c);
                    const int row = 4 * q + r;
                    const bool ok = row < tab[l].nrows;
                    const int lrow = ok ? row : tab[l].nrows - 1;
                    CHECK(lrow >= 0, "load row");
                    const uint64_t grow = static_cast<uint64_t>(cta_row_begin(g.layer[l], cta) + lrow);
                    if (ok) cov[l][grow * cpr + c] += 1;
                    using F = StreamFmt<FMT>;
                    const UnitAddr a = unit_addr<FMT, LG>(tab[l], cu, r, g.pstride);
                    const bool full = (c + 1) * F::kCols <= shapes[l].k;
                    CHECK(a.h2 == (full ? F::kVB / 2 : 0u), "half offset");
                    const uint64_t base = reinterpret_cast<uint64_t>(table[l].packed_dev);
                    const uint64_t vo = reinterpret_cast<uint64_t>(a.vp) - base;
                    const uint64_t io = reinterpret_cast<uint64_t>(a.ip) - base;
                    const uint64_t so = reinterpret_cast<uint64_t>(a.sp) - base;
                    const uint64_t vend = L[l].off_vals + (grow + 1) * L[l].vals_pitch;
                    const uint64_t vhalf = F::kVB / 2;  // bytes of each of the two nibble loads
                    CHECK(vo == L[l].off_vals + grow * L[l].vals_pitch + static_cast<uint64_t>(c) * F::kVB, "vals addr");
                    CHECK(vo % vhalf == 0 && vo + vhalf <= vend && vo + a.h2 + vhalf <= vend && (vo + a.h2) % vhalf == 0,
                          "vals bounds");
                    if constexpr (F::kIB > 0) {
                        const uint64_t iend = L[l].off_idx + (grow + 1) * L[l].idx_pitch;
                        const uint64_t ihalf = F::kIB / 2;
                        CHECK(io == L[l].off_idx + grow * L[l].idx_pitch + static_cast<uint64_t>(c) * F::kIB, "idx addr");
                        CHECK(io % ihalf == 0 && io + ihalf <= iend && io + a.h2 / 2 + ihalf <= iend, "idx bounds");
                    }
                    constexpr int NG = unit_groups<FMT, LG>(), CPG = F::kChunks / NG;
                    const uint64_t sbytes = 4 * NG;
                    const uint64_t srow = L[l].off_sz + grow * L[l].sz_pitch;
                    CHECK(so % sbytes == 0 && so >= srow && so + sbytes <= srow + L[l].sz_pitch, "sz bounds");
                    for (int grp = 0; grp < NG; ++grp) {
                        if (grp * CPG * 64 >= shapes[l].k - c * F::kCols) continue;  // a half unit's missing groups read padding
                        const uint64_t want = srow + ((static_cast<uint64_t>(c) * F::kCols + 64 * grp * CPG) >> LG) * 4;
                        CHECK(so + 4 * grp == want, "sz word of group %d", grp);
                        CHECK(want + 4 <= srow + 4ull * (shapes[l].k / shapes[l].g), "sz word beyond the row's groups");
                    }
                    CHECK(a.xo == g.layer[l].xoff + static_cast<uint32_t>(c) * F::kXU &&
                              static_cast<uint64_t>(B - 1) * g.xbs + a.xo + 2 * F::kCols <= x_end, "x read");
                    if (ok) {
                        CHECK(a.slot == static_cast<uint32_t>(r) * g.pstride + p, "slot");
                        // the row sum of row `row` reads slot (row & 3) * pstride + pbase + (row >> 2) * cpr + c
                        const uint32_t rs = static_cast<uint32_t>(row & 3) * g.pstride + tab[l].pbase +
                                            static_cast<uint32_t>((row >> 2) * cpr + c);
                        CHECK(rs == a.slot, "row-sum slot");
                        if (a.slot < slotcov.size()) slotcov[a.slot] += 1;
                    } else {
                        CHECK(a.slot == kNoSlot, "phantom row has a slot");
                    }
                    if (i + 1 < n) cursor_advance(nl, tab.data(), cu);
                }
            }
        for (size_t s = 0; s < slotcov.size(); ++s) CHECK(slotcov[s] <= 1, "slot %zu written %d times", s, slotcov[s]);
        // x staging: piece v of batch row b of layer l goes to b * xbs + xoff + (v / pu) * kXU + (v % pu) * 16
        for (int l = 0; l < nl; ++l) {
            constexpr int pu = StreamFmt<FMT>::kCols / 8;
            const int per_row = g.layer[l].cpr * pu;
            const uint64_t last = static_cast<uint64_t>(B - 1) * g.xbs + g.layer[l].xoff +
                                  static_cast<uint64_t>((per_row - 1) / pu) * StreamFmt<FMT>::kXU + ((per_row - 1) % pu) * 16 + 16;
            CHECK(last <= x_end, "x staging");
        }
    }
    for (int l = 0; l < nl; ++l) {
        for (size_t i = 0; i < cov[l].size(); ++i) CHECK(cov[l][i] == 1, "layer %d unit %zu covered %d", l, i, cov[l][i]);
        for (int r = 0; r < shapes[l].n; ++r) CHECK(rowcov[l][r] == 1, "layer %d row %d covered %d", l, r, rowcov[l][r]);
    }
}

// One group of layers (same batch and group size); packed buffers at distinct fake addresses.
static void check(const std::vector<Shape>& shapes, int B) {
    const bool expect_fit = smem_needed(shapes, B) <= 232448;
    const int nl = static_cast<int>(shapes.size());
    std::vector<sgemv_layer> table(nl);
    std::vector<sgemv_layout> L(nl);
    for (int i = 0; i < nl; ++i) {
        if (compute_layout(g_fmt, shapes[i].n, shapes[i].k, shapes[i].g, &L[i]) != SGEMV_OK) {
            printf("layout fail\n");
            ++fails;
            return;
        }
        table[i].layout = L[i];
        table[i].packed_dev = reinterpret_cast<const void*>(0x100000000ull * (i + 1));
        table[i].x_dev = reinterpret_cast<const void*>(0x10000000000ull + 0x100000000ull * i);
        table[i].y_dev = reinterpret_cast<void*>(0x20000000000ull + 0x100000000ull * i);
    }
    DeviceInfo di;
    di.sm_count = 152;
    di.max_smem_optin = 232448;
    StreamGroup g;
    int grid = 0;
    uint32_t smem = 0;
    const int rc = plan_stream(table.data(), nl, B, di, &g, &grid, &smem);
    if (!expect_fit) {
        CHECK(rc == SGEMV_ERR_SHAPE, "expected no fit, rc %d", rc);
        return;
    }
    CHECK(rc == SGEMV_OK, "plan rc %d (n %d k %d, %d layers, B %d)", rc, shapes[0].n, shapes[0].k, nl, B);
    if (rc) return;
    CHECK(smem <= static_cast<uint32_t>(di.max_smem_optin), "smem %u", smem);
    CHECK(grid >= 1 && grid <= di.sm_count, "grid %d", grid);
    const uint64_t x_end = static_cast<uint64_t>(B) * g.xbs;
    CHECK(sizeof(CtaLayer) == kCtaLayerBytes && g.tab_off % 16 == 0 && g.tab_off >= x_end, "table");
    CHECK(g.part_off >= g.tab_off + (kStreamMaxLayers + 1) * sizeof(CtaLayer) && g.part_off % 16 == 0, "sums overlap");
    CHECK(g.part_off + 4ull * B * 4 * g.pstride <= smem, "sums beyond smem");
    // x by the copy engine (groups of several layers, when it fits): raw copies after the sums, the
    // mbarrier after them; each copy 16-byte aligned at both ends with a size that is a multiple of 16,
    // and the pieces the transform reads inside the copy of their layer and batch row
    if (g.xraw_off) {
        ++g_copy_x;
        CHECK(nl >= kCopyXMinLayers, "copy-engine x for fewer layers than its minimum");
        CHECK(g.xraw_off >= g.part_off + 4ull * B * 4 * g.pstride && g.xraw_off % 16 == 0, "raw x region");
        uint64_t ro = g.xraw_off;
        for (int i = 0; i < nl; ++i)
            for (int b = 0; b < B; ++b) {
                const uint64_t bytes = 2ull * shapes[i].k;
                const uint64_t src = reinterpret_cast<uint64_t>(table[i].x_dev) + b * bytes;
                CHECK(ro % 16 == 0 && bytes % 16 == 0 && src % 16 == 0, "x copy alignment");
                // the transform reads pieces v < K / 8 of 16 bytes from ro
                CHECK(ro + 16ull * (shapes[i].k / 8) <= g.xraw_off + g.xraw_bytes, "x piece beyond its copy");
                ro += bytes;
            }
        CHECK(ro == g.xraw_off + g.xraw_bytes, "raw x bytes");
        CHECK(g.xbar_off == g.xraw_off + g.xraw_bytes && g.xbar_off % 8 == 0 && g.xbar_off + 8 <= smem,
              "x barrier");
        CHECK(g.xraw_bytes < (1u << 20), "transaction count beyond the mbarrier's range");
    } else if (nl >= kCopyXMinLayers) {
        uint64_t raw = 0, largest = 0;
        for (int i = 0; i < nl; ++i) {
            raw += 2ull * B * shapes[i].k;
            largest = std::max<uint64_t>(largest, 2ull * shapes[i].k);
        }
        CHECK(largest > kCopyXMaxCopy || raw > kCopyXMaxBytes ||
                  ((g.part_off + 4ull * B * 4 * g.pstride + 15) / 16 * 16) + raw + 8 > 232448,
              "copy-engine x left out although it fits its limits");
    }
    CHECK(g.xbs % 16 == 0, "x stride");
    for (int i = 0; i < nl; ++i) {
        const StreamLayer& S = g.layer[i];
        const int uc = stream_unit_cols(g_fmt);
        CHECK(S.cpr == (shapes[i].k + uc - 1) / uc && S.full == shapes[i].k / uc, "cpr");
        CHECK(S.dq == kPairsPerRound / S.cpr && S.dc == kPairsPerRound % S.cpr, "steps");
        CHECK(S.xoff + static_cast<uint64_t>(S.cpr) * stream_x_unit_bytes(g_fmt) <= g.xbs && S.xoff % 16 == 0, "x region");
    }
    const int lg = g.log2g;
    if (g_fmt == SGEMV_FMT_SPARSE24) {
        if (lg == 6) walk<SGEMV_FMT_SPARSE24, 6>(g, shapes, L, table, B, grid);
        else if (lg == 7) walk<SGEMV_FMT_SPARSE24, 7>(g, shapes, L, table, B, grid);
        else walk<SGEMV_FMT_SPARSE24, 8>(g, shapes, L, table, B, grid);
    } else if (g_fmt == SGEMV_FMT_SPARSE14) {
        if (lg == 6) walk<SGEMV_FMT_SPARSE14, 6>(g, shapes, L, table, B, grid);
        else if (lg == 7) walk<SGEMV_FMT_SPARSE14, 7>(g, shapes, L, table, B, grid);
        else walk<SGEMV_FMT_SPARSE14, 8>(g, shapes, L, table, B, grid);
    } else {
        if (lg == 6) walk<SGEMV_FMT_DENSE, 6>(g, shapes, L, table, B, grid);
        else if (lg == 7) walk<SGEMV_FMT_DENSE, 7>(g, shapes, L, table, B, grid);
        else walk<SGEMV_FMT_DENSE, 8>(g, shapes, L, table, B, grid);
    }
}

int main() {
    const int shapes[][2] = {{1, 128}, {7, 640}, {152, 1152}, {153, 2176}, {300, 1152}, {1024, 1024}, {38917, 128},
                             {38917, 384},
                             {4096, 4096}, {11008, 4096}, {4096, 11008}, {2000, 5120}, {999, 9216}, {600, 12288},
                             {200, 9216}, {32000, 4096}, {28672, 8192}, {8192, 28672}, {160, 131072}};
    int configs = 0;
    for (int fmt : {SGEMV_FMT_SPARSE24, SGEMV_FMT_SPARSE14, SGEMV_FMT_DENSE}) {
    g_fmt = fmt;
    for (auto& s : shapes)
        for (int g : {64, 128, 256})
            for (int B = 1; B <= kStreamMaxBatch; ++B) {
                if (s[1] % g) continue;
                if ((long long)s[0] * s[1] > 60000000LL && B != 1 && B != kStreamMaxBatch) continue;
                check({{s[0], s[1], g}}, B);
                ++configs;
            }
    // groups: the 7B decode step, a mixed group with ragged K and few-row layers, eight layers
    for (int B : {1, 2, kStreamMaxBatch}) {
        for (int g : {64, 128, 256}) {
            check({{4096, 4096, g}, {11008, 4096, g}, {4096, 11008, g}}, B);
            // the rotated quad partition spreads the three layers' extra quads: the busiest CTA of the
            // 7B step has 701 pairs (6 + 18 + 6 base quads, extras of the first and last layer), not 717
            if (g_fmt != SGEMV_FMT_DENSE) CHECK(g_max_pairs == 701, "7B step: busiest CTA %u pairs", g_max_pairs);
            check({{7, 640 / 128 * 128 + (g == 256 ? 128 : 0), g}, {300, 1280, g}, {1, 2304 + (g == 256 ? 256 : 0), g},
                   {2000, 9216, g}, {152, 256, g}}, B);
            check({{4096, 4096, g}, {4096, 4096, g}, {4096, 4096, g}, {4096, 4096, g}, {11008, 4096, g},
                   {11008, 4096, g}, {4096, 11008 + (g == 256 ? 256 : 0), g}, {155, 1280, g}}, B);
            configs += 3;
        }
        // a group may not mix group sizes
        std::vector<sgemv_layer> table(2);
        for (int i = 0; i < 2; ++i) {
            compute_layout(g_fmt, 256, 1024, i ? 64 : 128, &table[i].layout);
            table[i].packed_dev = reinterpret_cast<const void*>(0x100000000ull * (i + 1));
            table[i].x_dev = table[i].y_dev = reinterpret_cast<void*>(0x10000000000ull + 0x100000000ull * i);
        }
        DeviceInfo di;
        di.sm_count = 152;
        di.max_smem_optin = 232448;
        StreamGroup sg;
        int grid;
        uint32_t smem;
        CHECK(plan_stream(table.data(), 2, B, di, &sg, &grid, &smem) == SGEMV_ERR_ARG, "mixed group sizes accepted");
    }
    }
    // seeded random groups (splitmix64): 1-8 layers of one group size, N up to 3000 (few-row layers
    // included), K a multiple of the group size up to 12288, batch 1-3, each format
    uint64_t st = 0x5eed5eedull;
    auto next = [&st]() {
        uint64_t z = (st += 0x9E3779B97F4A7C15ull);
        z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
        z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
        return z ^ (z >> 31);
    };
    for (int t = 0; t < 240; ++t) {
        g_fmt = t % 3 == 0 ? SGEMV_FMT_SPARSE24 : (t % 3 == 1 ? SGEMV_FMT_SPARSE14 : SGEMV_FMT_DENSE);
        const int g = 64 << (next() % 3);
        const int nl = 1 + static_cast<int>(next() % 8);
        const int B = 1 + static_cast<int>(next() % kStreamMaxBatch);
        std::vector<Shape> grp;
        for (int i = 0; i < nl; ++i) {
            const int n = next() % 4 == 0 ? 1 + static_cast<int>(next() % 160) : 1 + static_cast<int>(next() % 3000);
            const int kmax = 12288 / std::max(g, 128);
            const int k = std::max(g, 128) * (1 + static_cast<int>(next() % kmax));
            grp.push_back({n, k, g});
        }
        check(grp, B);
        ++configs;
    }
    CHECK(g_copy_x > 0, "no group fetched x with the copy engine");
    printf("%d configs (%d with x by the copy engine), %d failures\n", configs, g_copy_x, fails);
    return fails ? 1 : 0;
}
