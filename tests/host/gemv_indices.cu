// Host-only check of the GEMV kernel's index arithmetic, built with the library's own planner
// (plan_gemv), task geometry (TaskSpace, warp_run, cta_rows) and load cursors (Loader<FMT>), for the 2:4,
// 1:4 and dense formats over ragged and full-size shapes, every group size and batch 1..8. For every
// CTA, pass, x tile, warp and lane it checks that:
//   * every weight load address is the one of its (row, column) and stays inside its row and section,
//     with the alignment of its vector width; the L2 prefetch ranges stay inside their sections;
//   * every existing (row, 64-column chunk) is loaded exactly once and every task is run exactly once;
//     every row belongs to exactly one CTA, and CTAs beyond a layer's grid own none;
//   * x staging and x reads stay inside the x tile, accumulator indices inside the accumulators, and
//     the shared-memory plan fits the device.
// No GPU is needed: the device code is compiled but never launched (tests/host/stub_launchers.cu).
#include <cstdio>
#include <cstdlib>
#include <utility>
#include <vector>
#include "gemv_kernel.cuh"

using namespace sgemv;

static int fails = 0;
static int g_splits = 0;  // configurations planned with split-K
#define CHECK(c, ...) do { if (!(c)) { if (fails < 20) { printf("FAIL %s:%d: ", __FILE__, __LINE__); printf(__VA_ARGS__); printf("\n"); } ++fails; } } while (0)

template <int FMT>
void check(int n, int k, int g, int B) {
    constexpr bool sp = FMT == SGEMV_FMT_SPARSE24;
    sgemv_layout L;
    if (compute_layout(FMT, n, k, g, &L) != SGEMV_OK) { printf("layout fail\n"); ++fails; return; }
    DeviceInfo di; di.sm_count = 152; di.max_smem_optin = 232448;
    GemvParams p; int grid; uint32_t smem;
    int rc = plan_gemv(L, (void*)0x100000000ull, (void*)0x200000000ull, B, (void*)0x300000000ull, nullptr, di, &p, &grid, &smem);
    CHECK(rc == SGEMV_OK, "plan rc %d", rc);
    if (rc) return;
    CHECK(smem <= (uint32_t)di.max_smem_optin, "smem %u", smem);
    CHECK(p.sm_acc >= p.sm_x + (uint32_t)B * p.x_b_stride, "x overlaps acc");
    CHECK(smem >= p.sm_acc + (uint32_t)(B * p.pass_rows * 4), "acc beyond smem");
    CHECK(p.pass_rows % 4 == 0, "pass_rows");
    CHECK(p.xt == k || p.xt % kTaskCols == 0, "xt");
    CHECK(p.x_b_stride % 16 == 0 && p.sm_x % 16 == 0 && p.sm_acc % 4 == 0, "align");
    std::vector<int> row_cov(n, 0);
    std::vector<int> chunk_cov((size_t)n * (k / 64), 0);
    CHECK(grid == p.nctas * p.split, "grid");
    CHECK(p.split == split_factor(n, k, di) && grid <= di.sm_count, "split");
    CHECK(p.split == 1 || k >= kSplitMinK, "split below the K threshold");
    if (p.split > 1) ++g_splits;
    for (int cta = 0; cta < grid; ++cta) {
        int row_begin, nrows, kbeg, kend;
        cta_work(p, cta, row_begin, nrows, kbeg, kend);
        CHECK(row_begin + nrows <= n, "cta rows");
        CHECK(kbeg % kTaskCols == 0 && kbeg < kend && kend <= k, "k slice %d %d", kbeg, kend);
        if (nrows <= 0) continue;
        const int rank = cta % p.split;
        if (p.split == 1) {
            const uint64_t rows = std::min(nrows, p.pass_rows);
            // the kernel widens each range to 16-byte boundaries; it must stay inside its section
            const uint64_t begins[3] = {L.off_vals + row_begin * L.vals_pitch, L.off_idx + row_begin * L.idx_pitch,
                                        L.off_sz + row_begin * L.sz_pitch};
            const uint64_t lens[3] = {rows * L.vals_pitch, sp || FMT == SGEMV_FMT_SPARSE14 ? rows * L.idx_pitch : 0,
                                      rows * L.sz_pitch};
            const uint64_t sec_lo[3] = {L.off_vals, L.off_idx, L.off_sz};
            const uint64_t sec_hi[3] = {L.off_idx, L.off_sz, L.off_rowptr};
            for (int q = 0; q < 3; ++q) {
                if (lens[q] == 0) continue;
                const uint64_t a0 = begins[q] & ~15ull, a1 = (begins[q] + lens[q] + 15) & ~15ull;
                CHECK(a0 >= sec_lo[q] && a1 <= sec_hi[q] && a1 <= L.total_bytes, "prefetch range %d", q);
            }
            CHECK(L.off_vals % 256 == 0 && L.off_idx % 256 == 0 && L.off_sz % 256 == 0, "section align");
            CHECK(rows * L.vals_pitch < (1ull << 32), "prefetch size");
        }
        const int ntile = (kend - kbeg + p.xt - 1) / p.xt;
        const int npass = (nrows + p.pass_rows - 1) / p.pass_rows;
        for (int pass = 0; pass < npass; ++pass) {
            const int prow0 = pass * p.pass_rows, prows = std::min(p.pass_rows, nrows - prow0);
            if (rank == 0)  // the rows of a cluster are written once, by its rank 0
                for (int rr = 0; rr < prows; ++rr) row_cov[row_begin + prow0 + rr] += 1;
            for (int tile = 0; tile < ntile; ++tile) {
                TaskSpace ts;
                ts.set(prow0, prows, kbeg + tile * p.xt, std::min(p.xt, kend - kbeg - tile * p.xt));
                CHECK(ts.tcols > 0 && ts.tcols % 128 == 0, "tile cols");
                const int units = ts.tcols / 8, punits = ts.nblk * (kTaskCols / 8);
                CHECK(ts.nblk * kTaskCols <= ((p.xt + kTaskCols - 1) / kTaskCols) * kTaskCols, "pad");
                for (int b = 0; b < B; ++b) {
                    const int v = units - 1;
                    CHECK((uint64_t)b * k + ts.tc0 + (uint64_t)v * 8 + 8 <= (uint64_t)B * k, "x src");
                    const int pv = punits - 1;
                    CHECK(b * p.x_b_stride + (pv >> 4) * kXLaneBytes + (pv & 15) * 16 + 16 <= (uint32_t)B * p.x_b_stride, "x dst");
                }
                std::vector<int> task_cov(ts.ntasks, 0);
                for (int w = 0; w < kWarps; ++w) {
                    int tb, te;
                    warp_run(ts.ntasks, w, tb, te);
                    CHECK(tb >= 0 && te <= ts.ntasks && tb <= te, "run");
                    if (tb == te) continue;
                    Loader<FMT> lds[32];
                    for (int lane = 0; lane < 32; ++lane) lds[lane].start(p, ts, row_begin, lane >> 3, lane & 7, tb);
                    int cquad = tb / ts.nblk, cblk = tb - cquad * ts.nblk;
                    for (int t = tb; t < te; ++t) {
                        task_cov[t] += 1;
                        CHECK(lds[0].quad == t / ts.nblk && lds[0].blk == t % ts.nblk, "loader cursor");
                        CHECK(cquad == t / ts.nblk && cblk == t % ts.nblk, "compute cursor");
                        const bool full = lds[0].full(ts);
                        for (int lane = 0; lane < 32; ++lane) {
                            const int r = lane >> 3, j = lane & 7;
                            Loader<FMT>& ld = lds[lane];
                            CHECK(ld.full(ts) == full, "full not warp-uniform");
                            const int rr = cquad * 4 + r;
                            // compute side reads x for both chunks whatever the task
                            const uint32_t xoff = (B - 1) * p.x_b_stride + (cblk * 8 + j) * kXLaneBytes + 256;
                            CHECK(xoff <= (uint32_t)B * p.x_b_stride, "x read");
                            if (rr < prows) CHECK((B - 1) * p.pass_rows + rr < B * p.pass_rows, "acc");
                            const bool on = full || ld.lane_on(ts, j);
                            const int cc = cblk * kTaskCols + j * kLaneCols;
                            const bool exists = rr < prows && cc < ts.tcols;
                            CHECK(on == exists, "lane_on t=%d lane=%d", t, lane);
                            if (!on) continue;
                            CHECK(cc + kLaneCols <= ts.tcols, "lane in tile");
                            const uint64_t grow = row_begin + ts.prow0 + rr;
                            const uint64_t gcol = ts.tc0 + cc;
                            CHECK(grow < (uint64_t)n, "grow");
                            const uint64_t vo = (uint64_t)(ld.vp - (const uint8_t*)0x100000000ull);
                            const uint64_t io = (uint64_t)(ld.ip - (const uint8_t*)0x100000000ull);
                            const uint64_t s0 = (uint64_t)(ld.sp0 - (const uint8_t*)0x100000000ull);
                            const uint64_t s1 = (uint64_t)(ld.sp1 - (const uint8_t*)0x100000000ull);
                            const uint64_t vcols = FMT == SGEMV_FMT_SPARSE24 ? 4 : (FMT == SGEMV_FMT_SPARSE14 ? 8 : 2);
                            const uint64_t vbytes = 128 / vcols, valign = FMT == SGEMV_FMT_SPARSE14 ? 16 : 32;
                            CHECK(vo == L.off_vals + grow * L.vals_pitch + gcol / vcols, "vals addr");
                            CHECK(vo % valign == 0 && vo + vbytes <= L.off_vals + (grow + 1) * L.vals_pitch, "vals");
                            if (FMT == SGEMV_FMT_SPARSE24)
                                CHECK(io == L.off_idx + grow * L.idx_pitch + gcol / 8 && io % 16 == 0 &&
                                      io + 16 <= L.off_idx + (grow + 1) * L.idx_pitch, "idx");
                            if (FMT == SGEMV_FMT_SPARSE14)
                                CHECK(io == L.off_idx + grow * L.idx_pitch + gcol / 16 && io % 8 == 0 &&
                                      io + 8 <= L.off_idx + (grow + 1) * L.idx_pitch, "idx14");
                            CHECK(s0 == L.off_sz + grow * L.sz_pitch + ((gcol >> p.log2g) << 2), "sz0 addr");
                            CHECK(s1 == L.off_sz + grow * L.sz_pitch + (((gcol + 64) >> p.log2g) << 2), "sz1 addr");
                            CHECK(s1 + 4 <= L.off_sz + grow * L.sz_pitch + 4 * (k / g), "sz");
                            chunk_cov[grow * (k / 64) + gcol / 64] += 1;
                            chunk_cov[grow * (k / 64) + gcol / 64 + 1] += 1;
                        }
                        for (int lane = 0; lane < 32; ++lane) lds[lane].advance(p, ts, row_begin, lane >> 3, lane & 7);
                        if (++cblk == ts.nblk) { ++cquad; cblk = 0; }
                    }
                }
                for (int t = 0; t < ts.ntasks; ++t) CHECK(task_cov[t] == 1, "task %d covered %d", t, task_cov[t]);
            }
        }
    }
    for (int u = p.nctas; u < p.nctas + 160; ++u) {
        int rb, nr;
        cta_rows(p, u, rb, nr);
        CHECK(nr == 0, "row unit %d beyond the layer's grid owns rows", u);
    }
    for (int r = 0; r < n; ++r) CHECK(row_cov[r] == 1, "row %d covered %d", r, row_cov[r]);
    for (size_t i = 0; i < chunk_cov.size(); ++i) CHECK(chunk_cov[i] == 1, "chunk %zu covered %d", i, chunk_cov[i]);
}

int main() {
    const int shapes[][2] = {{1, 128}, {7, 640}, {152, 1152}, {153, 2176}, {300, 1152}, {1024, 1024}, {4096, 4096},
                             {11008, 4096}, {4096, 11008}, {2000, 5120}, {38917, 128}, {8192, 28672}, {999, 9216},
                             {600, 12288}, {200, 9216}, {32000, 4096}, {28672, 8192},
                             // few rows and a short K: no split
                             {1, 4096}, {3, 2304}, {19, 8192}, {37, 11008}, {76, 2048}, {75, 4096},
                             // few rows and a long K: split-K by clusters of 8, 4 and 2 (uneven block shares
                             // included)
                             {1, 32768}, {3, 33792}, {19, 65536}, {37, 40960}, {76, 32768}, {75, 36864}};
    int configs = 0;
    for (auto& s : shapes)
        for (int g : {64, 128, 256})
            for (int B = 1; B <= 8; ++B) {
                if (s[1] % g) continue;
                if ((long long)s[0] * s[1] > 60000000LL && B != 1 && B != 8) continue;
                check<SGEMV_FMT_SPARSE24>(s[0], s[1], g, B);
                check<SGEMV_FMT_DENSE>(s[0], s[1], g, B);
                check<SGEMV_FMT_SPARSE14>(s[0], s[1], g, B);
                configs += 3;
            }
    // the format's limits: K = 2^20 (many x tiles), N = 2^24 (hundreds of accumulator passes per CTA)
    for (int B : {1, 8})
        for (int g : {64, 256}) {
            check<SGEMV_FMT_SPARSE24>(5, 1 << 20, g, B);
            check<SGEMV_FMT_DENSE>(5, 1 << 20, g, B);
            check<SGEMV_FMT_SPARSE14>(5, 1 << 20, g, B);
            configs += 3;
        }
    check<SGEMV_FMT_SPARSE24>(1 << 24, 128, 64, 1);
    check<SGEMV_FMT_DENSE>(1 << 24, 128, 64, 1);
    check<SGEMV_FMT_SPARSE14>(1 << 24, 128, 64, 1);
    configs += 3;
    CHECK(g_splits > 0, "no configuration was split");
    printf("%d configs (%d split over K), %d failures\n", configs, g_splits, fails);
    return fails ? 1 : 0;
}
