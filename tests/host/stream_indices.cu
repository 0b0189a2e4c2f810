// Host-only check of the streaming GEMV kernel's index arithmetic, built with the library's own planner
// (plan_stream), CTA table (build_table), unit cursor (cursor_set, cursor_advance) and addresses
// (unit_addr), for single layers and groups of layers over ragged and full-size shapes, every group size
// and batch 1..8. For every CTA and every one of its 512 lanes it walks the lane's units exactly as the
// kernel does and checks that:
//   * every unit of every row of every layer is visited exactly once, by the CTA that owns the row;
//   * every weight load (two 32-byte nibble loads, two 16-byte position loads and four 4-byte {s, z}
//     loads for a full unit; half of them for the half unit ending a row with K % 256 == 128) is the one
//     of its (row, columns), stays inside its row and section, and has its vector width's alignment;
//   * the unit's x (512 bytes per batch row) and its sum slot stay inside their shared-memory regions,
//     and the regions (x, layer table, unit sums) do not overlap and fit the device.
// No GPU is needed: the device code is compiled but never launched (tests/host/stub_launchers.cu).
#include <cstdio>
#include <cstdlib>
#include <vector>

#include "stream_kernel.cuh"

using namespace sgemv;

static int fails = 0;
#define CHECK(c, ...) do { if (!(c)) { if (fails < 20) { printf("FAIL %s:%d: ", __FILE__, __LINE__); printf(__VA_ARGS__); printf("\n"); } ++fails; } } while (0)

struct Shape {
    int n, k, g;
};

// Shared memory of a streaming launch, restated: x of every layer (528 bytes per 256-column unit and
// batch row), the layer table (9 entries of 12 bytes), then fp32 unit sums for the CTA with most units.
static uint64_t smem_needed(const std::vector<Shape>& shapes, int B) {
    auto r16 = [](uint64_t v) { return (v + 15) / 16 * 16; };
    uint64_t x = 0, units = 0;
    for (const Shape& s : shapes) {
        const uint64_t cpr = (s.k + 255) / 256, ctas = s.n < 152 ? s.n : 152;
        x += cpr * 528;
        units += (s.n / ctas + (s.n % ctas ? 1 : 0)) * cpr;
    }
    return r16(r16(B * x) + 9 * 12) + 4ull * B * ((units + 3) / 4 * 4);
}

// One group of layers (same batch); packed buffers at distinct fake addresses.
static void check(const std::vector<Shape>& shapes, int B) {
    const bool expect_fit = smem_needed(shapes, B) <= 232448;
    const int nl = static_cast<int>(shapes.size());
    std::vector<sgemv_layer> table(nl);
    std::vector<sgemv_layout> L(nl);
    for (int i = 0; i < nl; ++i) {
        if (compute_layout(SGEMV_FMT_SPARSE24, shapes[i].n, shapes[i].k, shapes[i].g, &L[i]) != SGEMV_OK) {
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
    CHECK(g.tab_off >= x_end && g.tab_off % 16 == 0, "table overlaps x");
    CHECK(g.part_off >= g.tab_off + (kStreamMaxLayers + 1) * sizeof(CtaLayer) && g.part_off % 16 == 0, "sums overlap");
    CHECK(g.part_off + 4ull * B * g.ustride <= smem, "sums beyond smem");
    CHECK(g.xbs % 16 == 0, "x stride");
    std::vector<std::vector<int>> cov(nl);
    std::vector<std::vector<int>> rowcov(nl);
    for (int i = 0; i < nl; ++i) {
        const StreamLayer& S = g.layer[i];
        CHECK(S.cpr == (shapes[i].k + 255) / 256 && S.full == shapes[i].k / 256, "cpr");
        CHECK(S.xoff + static_cast<uint64_t>(S.cpr) * kXUnitBytes <= g.xbs && S.xoff % 16 == 0, "x region");
        cov[i].assign(static_cast<size_t>(shapes[i].n) * S.cpr, 0);
        rowcov[i].assign(shapes[i].n, 0);
    }
    std::vector<CtaLayer> tab(kStreamMaxLayers + 1);
    for (int cta = 0; cta < di.sm_count; ++cta) {
        build_table(g, cta, tab.data());
        const uint32_t utotal = tab[nl].ubase;
        CHECK(utotal <= g.ustride, "units %u > ustride %u", utotal, g.ustride);
        for (int l = 0; l < nl; ++l) {
            const CtaLayer& e = tab[l];
            CHECK(e.nrows == 0 || (e.nrows > 0 && e.row_begin + e.nrows <= shapes[l].n), "cta rows");
            if (cta >= grid) CHECK(e.nrows == 0, "CTA beyond the grid owns rows");
            for (int r = 0; r < e.nrows; ++r) rowcov[l][e.row_begin + r] += 1;
            if (cta == 0 && l == 0 && e.nrows > 0) {
                // the L2 prefetch ranges of the first layer, widened to 16 bytes, stay inside their sections
                const uint64_t begins[3] = {L[0].off_vals + e.row_begin * L[0].vals_pitch,
                                            L[0].off_idx + e.row_begin * L[0].idx_pitch,
                                            L[0].off_sz + e.row_begin * L[0].sz_pitch};
                const uint64_t lens[3] = {e.nrows * L[0].vals_pitch, e.nrows * L[0].idx_pitch, e.nrows * L[0].sz_pitch};
                const uint64_t lo[3] = {L[0].off_vals, L[0].off_idx, L[0].off_sz};
                const uint64_t hi[3] = {L[0].off_idx, L[0].off_sz, L[0].off_rowptr};
                for (int q = 0; q < 3; ++q) {
                    const uint64_t a0 = begins[q] & ~15ull, a1 = (begins[q] + lens[q] + 15) & ~15ull;
                    CHECK(a0 >= lo[q] && a1 <= hi[q], "prefetch range %d", q);
                }
            }
        }
        for (uint32_t lane = 0; lane < static_cast<uint32_t>(kThreads) && lane < utotal; ++lane) {
            UnitCursor cu;
            cursor_set(g, tab.data(), utotal, lane, cu);
            uint32_t expect_u = lane;
            while (cu.u < utotal) {
                CHECK(cu.u == expect_u, "cursor u %u expected %u", cu.u, expect_u);
                // reference (layer, row, unit) of flat unit u
                int l = 0;
                while (l + 1 < nl && cu.u >= tab[l + 1].ubase) ++l;
                const uint32_t q = cu.u - tab[l].ubase;
                const int cpr = g.layer[l].cpr;
                const int r = static_cast<int>(q / cpr), c = static_cast<int>(q % cpr);
                CHECK(cu.l == l && cu.r == r && cu.c == c, "cursor (l %d r %d c %d) expected (%d %d %d)", cu.l, cu.r,
                      cu.c, l, r, c);
                CHECK(r < tab[l].nrows, "row beyond the CTA's rows");
                const uint64_t row = static_cast<uint64_t>(tab[l].row_begin + r);
                cov[l][row * cpr + c] += 1;
                const UnitAddr a = unit_addr(g, tab.data(), cu);
                const bool full = (c + 1) * 256 <= shapes[l].k;
                CHECK(a.full == full, "full flag");
                const uint64_t base = reinterpret_cast<uint64_t>(table[l].packed_dev);
                const uint64_t vo = reinterpret_cast<uint64_t>(a.vp) - base;
                const uint64_t io = reinterpret_cast<uint64_t>(a.ip) - base;
                const uint64_t so = reinterpret_cast<uint64_t>(a.sp) - base;
                const uint64_t vbytes = full ? 64 : 32, ibytes = full ? 32 : 16;
                CHECK(vo == L[l].off_vals + row * L[l].vals_pitch + static_cast<uint64_t>(c) * 64, "vals addr");
                CHECK(vo % 32 == 0 && vo + vbytes <= L[l].off_vals + (row + 1) * L[l].vals_pitch, "vals bounds");
                CHECK(io == L[l].off_idx + row * L[l].idx_pitch + static_cast<uint64_t>(c) * 32, "idx addr");
                CHECK(io % 16 == 0 && io + ibytes <= L[l].off_idx + (row + 1) * L[l].idx_pitch, "idx bounds");
                const int lg = g.layer[l].log2g;
                const uint32_t so_k[4] = {0, g.layer[l].so1, g.layer[l].so2, g.layer[l].so3};
                for (int kk = 0; kk < (full ? 4 : 2); ++kk) {
                    const uint64_t want = L[l].off_sz + row * L[l].sz_pitch + ((static_cast<uint64_t>(c) * 256 + 64 * kk) >> lg) * 4;
                    CHECK(so + so_k[kk] == want, "sz addr chunk %d", kk);
                    CHECK(want % 4 == 0 && want + 4 <= L[l].off_sz + row * L[l].sz_pitch + 4ull * (shapes[l].k / shapes[l].g),
                          "sz bounds");
                }
                const uint64_t xlast = static_cast<uint64_t>(B - 1) * g.xbs + a.xo + 512;
                CHECK(a.xo == g.layer[l].xoff + static_cast<uint32_t>(c) * kXUnitBytes && xlast <= x_end, "x read");
                CHECK(cu.u < g.ustride, "slot");
                cursor_advance(g, tab.data(), utotal, cu);
                expect_u += kThreads;
            }
        }
        // x staging: piece v of batch row b of layer l goes to b * xbs + xoff + (v / 32) * 528 + (v % 32) * 16
        for (int l = 0; l < nl; ++l) {
            const int per_row = g.layer[l].cpr * 32;
            const uint64_t last = static_cast<uint64_t>(B - 1) * g.xbs + g.layer[l].xoff +
                                  static_cast<uint64_t>((per_row - 1) >> 5) * kXUnitBytes + ((per_row - 1) & 31) * 16 + 16;
            CHECK(last <= x_end, "x staging");
        }
    }
    for (int l = 0; l < nl; ++l) {
        for (size_t i = 0; i < cov[l].size(); ++i) CHECK(cov[l][i] == 1, "layer %d unit %zu covered %d", l, i, cov[l][i]);
        for (int r = 0; r < shapes[l].n; ++r) CHECK(rowcov[l][r] == 1, "layer %d row %d covered %d", l, r, rowcov[l][r]);
    }
}

int main() {
    const int shapes[][2] = {{1, 128}, {7, 640}, {152, 1152}, {153, 2176}, {300, 1152}, {1024, 1024},
                             {4096, 4096}, {11008, 4096}, {4096, 11008}, {2000, 5120}, {999, 9216}, {600, 12288},
                             {200, 9216}, {32000, 4096}, {28672, 8192}, {8192, 28672}, {160, 131072}};
    int configs = 0;
    for (auto& s : shapes)
        for (int g : {64, 128, 256})
            for (int B = 1; B <= 8; ++B) {
                if (s[1] % g) continue;
                if ((long long)s[0] * s[1] > 60000000LL && B != 1 && B != 8) continue;
                check({{s[0], s[1], g}}, B);
                ++configs;
            }
    // groups: the 7B decode step, a mixed group with ragged K and few-row layers, eight layers
    for (int B : {1, 2, 8}) {
        check({{4096, 4096, 128}, {11008, 4096, 128}, {4096, 11008, 128}}, B);
        check({{7, 640, 64}, {300, 1152, 128}, {1, 2304, 256}, {2000, 9216, 128}, {152, 128, 64}}, B);
        check({{4096, 4096, 64}, {4096, 4096, 128}, {4096, 4096, 256}, {4096, 4096, 128}, {11008, 4096, 64},
               {11008, 4096, 256}, {4096, 11008, 128}, {155, 1152, 64}}, B);
        configs += 3;
    }
    printf("%d configs, %d failures\n", configs, fails);
    return fails ? 1 : 0;
}
