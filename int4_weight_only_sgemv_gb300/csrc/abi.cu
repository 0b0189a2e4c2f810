// Host side of the C ABI declared in include/sgemv.h: argument checks, the packed layout, launch
// geometry of the GEMV kernels, and the per-layer dispatch of sgemv_run_stack.
#include <algorithm>
#include <cstring>
#include <mutex>

#include "common.cuh"

namespace sgemv {

namespace {

uint64_t round_up(uint64_t v, uint64_t m) { return (v + m - 1) / m * m; }

int ilog2(int v) {
    int r = 0;
    while ((1 << r) < v) ++r;
    return r;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned32(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 31u) == 0; }

}  // namespace

int compute_layout(int format, int n, int k, int group, sgemv_layout* out) {
    if (out == nullptr) return SGEMV_ERR_ARG;
    if (format != SGEMV_FMT_SPARSE24 && format != SGEMV_FMT_DENSE && format != SGEMV_FMT_SPARSE14)
        return SGEMV_ERR_ARG;
    if (n < 1 || n > (1 << 24)) return SGEMV_ERR_SHAPE;
    if (k < 128 || k > (1 << 20) || k % 128 != 0) return SGEMV_ERR_SHAPE;
    if (group != 64 && group != 128 && group != 256) return SGEMV_ERR_SHAPE;
    if (k % group != 0) return SGEMV_ERR_SHAPE;
    // row_ptr is int32 (packed format v1, section 7.4): N times the kept elements of a row must fit
    const int64_t kept = format == SGEMV_FMT_SPARSE24 ? k / 2 : (format == SGEMV_FMT_SPARSE14 ? k / 4 : 0);
    if (static_cast<int64_t>(n) * kept > INT32_MAX) return SGEMV_ERR_SHAPE;
    sgemv_layout L;
    std::memset(&L, 0, sizeof(L));
    L.format = format;
    L.n = n;
    L.k = k;
    L.group = group;
    const bool sparse = (format != SGEMV_FMT_DENSE);
    const uint64_t kk = static_cast<uint64_t>(k);
    L.vals_pitch = format == SGEMV_FMT_SPARSE24 ? kk / 4 : (format == SGEMV_FMT_SPARSE14 ? kk / 8 : kk / 2);
    L.idx_pitch = format == SGEMV_FMT_SPARSE24 ? kk / 8 : (format == SGEMV_FMT_SPARSE14 ? kk / 16 : 0);
    L.sz_pitch = round_up(4ull * static_cast<uint64_t>(k / group), 16);
    const uint64_t nn = static_cast<uint64_t>(n);
    L.off_vals = 256;
    L.off_idx = L.off_vals + round_up(nn * L.vals_pitch, 256);
    L.off_sz = L.off_idx + round_up(nn * L.idx_pitch, 256);
    L.off_rowptr = L.off_sz + round_up(nn * L.sz_pitch, 256);
    L.total_bytes = L.off_rowptr + round_up(sparse ? 4 * (nn + 1) : 0, 256);
    *out = L;
    return SGEMV_OK;
}

bool layout_equal(const sgemv_layout& a, const sgemv_layout& b) {
    return a.format == b.format && a.n == b.n && a.k == b.k && a.group == b.group &&
           a.vals_pitch == b.vals_pitch && a.idx_pitch == b.idx_pitch && a.sz_pitch == b.sz_pitch &&
           a.off_vals == b.off_vals && a.off_idx == b.off_idx && a.off_sz == b.off_sz &&
           a.off_rowptr == b.off_rowptr && a.total_bytes == b.total_bytes;
}

int device_info(DeviceInfo* out) {
    static std::mutex mu;
    static DeviceInfo cache[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return SGEMV_ERR_CUDA;
    std::lock_guard<std::mutex> lock(mu);
    if (cache[dev].sm_count == 0) {
        DeviceInfo di;
        if (cudaDeviceGetAttribute(&di.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&di.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
            return SGEMV_ERR_CUDA;
        for (int i = 0; i < 3; ++i)
            if (query_max_clusters(2 << i, &di.max_clusters[i]) != cudaSuccess) return SGEMV_ERR_CUDA;
        cache[dev] = di;
    }
    *out = cache[dev];
    return SGEMV_OK;
}

namespace {

// Validates the caller's layout against the one recomputed from (format, n, k, group).
int check_layout(const sgemv_layout* layout) {
    if (layout == nullptr) return SGEMV_ERR_ARG;
    sgemv_layout ref;
    const int rc = compute_layout(layout->format, layout->n, layout->k, layout->group, &ref);
    if (rc != SGEMV_OK) return rc == SGEMV_ERR_ARG ? SGEMV_ERR_FORMAT : rc;
    return layout_equal(ref, *layout) ? SGEMV_OK : SGEMV_ERR_FORMAT;
}

bool is_sparse(int format) { return format == SGEMV_FMT_SPARSE24 || format == SGEMV_FMT_SPARSE14; }

// Byte ranges [a, a + na) and [b, b + nb) overlap.
bool overlap(const void* a, size_t na, const void* b, size_t nb) {
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + nb && b0 < a0 + na;
}

// want_sparse: the entry point reads sparse layouts (sgemv_run) or dense ones (sgemv_run_dense).
int check_run_args(const sgemv_layout* layout, bool want_sparse, const void* packed, const void* x, int batch,
                   const void* y, const int32_t* status) {
    const int rc = check_layout(layout);
    if (rc != SGEMV_OK) return rc;
    if (is_sparse(layout->format) != want_sparse) return SGEMV_ERR_FORMAT;
    if (packed == nullptr || x == nullptr || y == nullptr) return SGEMV_ERR_ARG;
    if (batch < 1 || batch > 8) return SGEMV_ERR_ARG;
    if (!aligned32(packed) || !aligned16(x) || !aligned16(y) || (reinterpret_cast<uintptr_t>(status) & 3u))
        return SGEMV_ERR_ALIGN;
    // y is written while x and the packed layer are read: it may overlap neither
    const size_t xb = 2ull * batch * static_cast<size_t>(layout->k), yb = 2ull * batch * static_cast<size_t>(layout->n);
    if (overlap(y, yb, x, xb) || overlap(y, yb, packed, layout->total_bytes)) return SGEMV_ERR_ARG;
    return SGEMV_OK;
}

}  // namespace


// Launch geometry and shared-memory plan of one GEMV (see gemv_kernel.cuh).
int split_factor(int n, int k, const DeviceInfo& di) {
    if (k < kSplitMinK) return 1;
    const int nblk = (k + kTaskCols - 1) / kTaskCols;
    for (int s = kMaxSplit, i = 2; s >= 2; s >>= 1, --i)
        if (n * s <= di.sm_count && s <= nblk && n <= di.max_clusters[i]) return s;
    return 1;
}

int plan_gemv(const sgemv_layout& L, const void* packed, const void* x, int batch, void* y, int32_t* status,
              const DeviceInfo& di, GemvParams* pp, int* grid, uint32_t* smem) {
    const uint8_t* base = static_cast<const uint8_t*>(packed);
    GemvParams p;
    std::memset(&p, 0, sizeof(p));
    p.vals = base + L.off_vals;
    p.idx = base + L.off_idx;
    p.sz = base + L.off_sz;
    p.vals_pitch = static_cast<uint32_t>(L.vals_pitch);
    p.idx_pitch = static_cast<uint32_t>(L.idx_pitch);
    p.sz_pitch = static_cast<uint32_t>(L.sz_pitch);
    p.x = static_cast<const __half*>(x);
    p.y = static_cast<__half*>(y);
    p.status = status;
    p.n = L.n;
    p.k = L.k;
    p.log2g = ilog2(L.group);
    p.split = split_factor(L.n, L.k, di);
    const int g = std::min(di.sm_count / p.split, L.n);  // row units (CTAs, or clusters with split-K)
    p.nctas = g;
    p.rows_base = L.n / g;
    p.rows_rem = L.n % g;
    // x tile: as many columns as fit the budget, a multiple of the task width (or all of K).
    int xt = static_cast<int>(kXTileBudget / (static_cast<uint32_t>(batch) * kXLaneBytes)) * kLaneCols;
    xt = std::max(kTaskCols, xt / kTaskCols * kTaskCols);
    p.xt = std::min(L.k, xt);
    const int rows_max = p.rows_base + (p.rows_rem > 0 ? 1 : 0);
    p.pass_rows = std::min(kMaxPassRows, (rows_max + 3) / 4 * 4);
    // staged over whole 1024-column blocks (zero padded): never more than the budget, a multiple of 1024
    p.x_b_stride = static_cast<uint32_t>((p.xt + kTaskCols - 1) / kTaskCols * (kTaskCols / kLaneCols)) * kXLaneBytes;
    const uint32_t x_bytes = static_cast<uint32_t>(batch) * p.x_b_stride;
    const uint32_t acc_bytes = static_cast<uint32_t>(batch * p.pass_rows) * 4u;
    p.sm_x = 0;
    p.sm_acc = x_bytes;
    *smem = x_bytes + acc_bytes;
    if (*smem > static_cast<uint32_t>(di.max_smem_optin)) return SGEMV_ERR_SHAPE;
    *grid = g * p.split;
    *pp = p;
    return SGEMV_OK;
}

// Plan of one streaming launch over the layers table[0 .. n) (same format, group size and batch). Fails
// with SGEMV_ERR_SHAPE when the x of every layer plus the unit sums do not fit the shared memory of a CTA.
int plan_stream(const sgemv_layer* table, int n, int batch, const DeviceInfo& di, StreamGroup* gp, int* grid,
                uint32_t* smem) {
    if (n < 1 || n > kStreamMaxLayers) return SGEMV_ERR_ARG;
    StreamGroup g;
    std::memset(&g, 0, sizeof(g));
    g.n_layers = n;
    g.log2g = ilog2(table[0].layout.group);
    const int fmt = table[0].layout.format;
    const int uc = stream_unit_cols(fmt);
    uint32_t xoff = 0, rot = 0;
    uint64_t pairs_max = 0;
    int gr = 0;
    for (int i = 0; i < n; ++i) {
        const sgemv_layout& L = table[i].layout;
        if (ilog2(L.group) != g.log2g || L.format != fmt) return SGEMV_ERR_ARG;
        const uint8_t* base = static_cast<const uint8_t*>(table[i].packed_dev);
        StreamLayer& s = g.layer[i];
        s.vals = base + L.off_vals;
        s.idx = base + L.off_idx;
        s.sz = base + L.off_sz;
        s.vals_pitch = static_cast<uint32_t>(L.vals_pitch);
        s.idx_pitch = static_cast<uint32_t>(L.idx_pitch);
        s.sz_pitch = static_cast<uint32_t>(L.sz_pitch);
        s.x = static_cast<const __half*>(table[i].x_dev);
        s.y = static_cast<__half*>(table[i].y_dev);
        s.n = L.n;
        s.k = L.k;
        const int nq = (L.n + 3) / 4;  // quads of the layer
        s.nctas = std::min(di.sm_count, nq);
        s.q_base = nq / s.nctas;
        s.q_rem = nq % s.nctas;
        // the extra quads of this layer start where the previous layer's ended (all-SM layers)
        s.q_rot = s.nctas == di.sm_count ? static_cast<int>(rot % static_cast<uint32_t>(s.nctas)) : 0;
        if (s.nctas == di.sm_count) rot = static_cast<uint32_t>(s.q_rot + s.q_rem) % static_cast<uint32_t>(s.nctas);
        s.cpr = (L.k + uc - 1) / uc;
        s.full = L.k / uc;
        s.dq = kPairsPerRound / s.cpr;
        s.dc = kPairsPerRound % s.cpr;
        s.xoff = xoff;
        xoff += static_cast<uint32_t>(s.cpr) * stream_x_unit_bytes(fmt);
        pairs_max += static_cast<uint64_t>(s.q_base + (s.q_rem > 0 ? 1 : 0)) * static_cast<uint64_t>(s.cpr);
        gr = std::max(gr, s.nctas);
    }
    g.xbs = xoff;
    const uint64_t x_bytes = static_cast<uint64_t>(batch) * xoff;
    g.tab_off = static_cast<uint32_t>(round_up(x_bytes, 16));
    const uint64_t tab_end = g.tab_off + (kStreamMaxLayers + 1) * static_cast<uint64_t>(kCtaLayerBytes);
    g.pstride = static_cast<uint32_t>(round_up(pairs_max, 4));
    g.part_off = static_cast<uint32_t>(round_up(tab_end, 16));
    uint64_t total = g.part_off + 4ull * batch * 4ull * g.pstride;
    if (total > static_cast<uint64_t>(di.max_smem_optin)) return SGEMV_ERR_SHAPE;
    // Three or more layers: their x arrives by the copy engine, one copy per layer and batch row, all in
    // flight at once, where plain loads would fetch the layers one after another. Measured on the 7B
    // decode step (µs per GEMV): 5.30 against 5.42 at batch 1, 7.35 against 7.86 at batch 2. The copy
    // engine of an SM moves a few tens of GB/s, so it loses with large copies or much x (the wide FFN
    // step, one 56 KB copy: 23.05 against 21.26) and with two layers (two rounds of loads are as fast):
    // hence the limits kCopyXMinLayers, kCopyXMaxCopy and kCopyXMaxBytes.
    if (n >= kCopyXMinLayers) {
        uint64_t raw = 0, largest = 0;
        for (int i = 0; i < n; ++i) {
            raw += 2ull * batch * static_cast<uint64_t>(table[i].layout.k);
            largest = std::max<uint64_t>(largest, 2ull * static_cast<uint64_t>(table[i].layout.k));
        }
        const uint64_t raw_off = round_up(total, 16);
        const uint64_t end = raw_off + raw + 8;
        if (largest <= kCopyXMaxCopy && raw <= kCopyXMaxBytes && end <= static_cast<uint64_t>(di.max_smem_optin)) {
            g.xraw_off = static_cast<uint32_t>(raw_off);
            g.xraw_bytes = static_cast<uint32_t>(raw);
            g.xbar_off = static_cast<uint32_t>(raw_off + raw);
            total = end;
        }
    }
    *smem = static_cast<uint32_t>(total);
    *grid = gr;
    *gp = g;
    return SGEMV_OK;
}

cudaError_t launch_stream(int format, int batch, const StreamGroup& g, int grid, uint32_t smem, cudaStream_t s) {
    const int lg = g.log2g;
    if (lg < 6 || lg > 8) return cudaErrorInvalidValue;
    switch (format) {
        case SGEMV_FMT_SPARSE24:
            return lg == 6 ? launch_stream24_g64(batch, g, grid, smem, s)
                           : (lg == 7 ? launch_stream24_g128(batch, g, grid, smem, s) : launch_stream24_g256(batch, g, grid, smem, s));
        case SGEMV_FMT_SPARSE14:
            return lg == 6 ? launch_stream14_g64(batch, g, grid, smem, s)
                           : (lg == 7 ? launch_stream14_g128(batch, g, grid, smem, s) : launch_stream14_g256(batch, g, grid, smem, s));
        case SGEMV_FMT_DENSE:
            return lg == 6 ? launch_streamd_g64(batch, g, grid, smem, s)
                           : (lg == 7 ? launch_streamd_g128(batch, g, grid, smem, s) : launch_streamd_g256(batch, g, grid, smem, s));
        default:
            return cudaErrorInvalidValue;
    }
}

namespace {

// The streaming kernel serves the layers that need no split over K, up to batch kStreamMaxBatch; larger
// batches run the tiled kernel, which measured faster there (its shorter loop body stays in the
// instruction cache).
bool streams(const sgemv_layout& L, const DeviceInfo& di, int batch) {
    return batch <= kStreamMaxBatch && split_factor(L.n, L.k, di) == 1;
}

cudaError_t launch_group(int format, int batch, const LayerGroup& g, int grid, uint32_t smem, cudaStream_t s) {
    return format == SGEMV_FMT_SPARSE24   ? launch_gemv_sparse(batch, g, grid, smem, s)
           : format == SGEMV_FMT_SPARSE14 ? launch_gemv_sparse14(batch, g, grid, smem, s)
                                          : launch_gemv_dense(batch, g, grid, smem, s);
}

int run_one(const sgemv_layout* layout, bool want_sparse, const void* packed, const void* x, int batch, void* y,
            int32_t* status, void* stream) {
    int rc = check_run_args(layout, want_sparse, packed, x, batch, y, status);
    if (rc != SGEMV_OK) return rc;
    DeviceInfo di;
    rc = device_info(&di);
    if (rc != SGEMV_OK) return rc;
    if (streams(*layout, di, batch)) {
        sgemv_layer one;
        one.layout = *layout;
        one.packed_dev = packed;
        one.x_dev = x;
        one.y_dev = y;
        StreamGroup sgp;
        int grid = 0;
        uint32_t smem = 0;
        if (plan_stream(&one, 1, batch, di, &sgp, &grid, &smem) == SGEMV_OK) {
            sgp.status = status;
            const cudaError_t e = launch_stream(layout->format, batch, sgp, grid, smem, static_cast<cudaStream_t>(stream));
            return e == cudaSuccess ? SGEMV_OK : SGEMV_ERR_CUDA;
        }
    }
    LayerGroup g;
    std::memset(&g, 0, sizeof(g));
    g.n_layers = 1;
    int grid = 0;
    uint32_t smem = 0;
    rc = plan_gemv(*layout, packed, x, batch, y, status, di, &g.layer[0], &grid, &smem);
    if (rc != SGEMV_OK) return rc;
    const cudaError_t e = launch_group(layout->format, batch, g, grid, smem, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? SGEMV_OK : SGEMV_ERR_CUDA;
}

// Layer l of the table can join a group that starts at layer g0: same format, and no data flows between
// it and any earlier member (its x overlaps no member's y, its y overlaps no member's x or y).
bool can_join(const sgemv_layer* table, int g0, int l, int batch) {
    const sgemv_layer& c = table[l];
    if (c.layout.format != table[g0].layout.format || l - g0 >= kMaxGroup) return false;
    const size_t cx = 2ull * batch * c.layout.k, cy = 2ull * batch * c.layout.n;
    for (int i = g0; i < l; ++i) {
        const sgemv_layer& m = table[i];
        const size_t mx = 2ull * batch * m.layout.k, my = 2ull * batch * m.layout.n;
        if (overlap(c.x_dev, cx, m.y_dev, my) || overlap(c.y_dev, cy, m.x_dev, mx) ||
            overlap(c.y_dev, cy, m.y_dev, my))
            return false;
    }
    return true;
}

}  // namespace

}  // namespace sgemv

using namespace sgemv;

extern "C" {

int sgemv_abi_version(void) { return 1; }

const char* sgemv_status_str(int status) {
    switch (status) {
        case SGEMV_OK: return "SGEMV_OK";
        case SGEMV_ERR_ARG: return "SGEMV_ERR_ARG";
        case SGEMV_ERR_SHAPE: return "SGEMV_ERR_SHAPE";
        case SGEMV_ERR_ALIGN: return "SGEMV_ERR_ALIGN";
        case SGEMV_ERR_FORMAT: return "SGEMV_ERR_FORMAT";
        case SGEMV_ERR_CUDA: return "SGEMV_ERR_CUDA";
        case SGEMV_ERR_NONFINITE: return "SGEMV_ERR_NONFINITE";
        case SGEMV_ERR_TIMEOUT: return "SGEMV_ERR_TIMEOUT";
        default: return "SGEMV_ERR_UNKNOWN";
    }
}

int sgemv_layout_query(int format, int n, int k, int group, sgemv_layout* out) {
    return compute_layout(format, n, k, group, out);
}

int sgemv_pack(const sgemv_layout* layout, const void* w_dev, void* packed_dev, int32_t* status_dev, void* stream) {
    int rc = check_layout(layout);
    if (rc != SGEMV_OK) return rc;
    if (w_dev == nullptr || packed_dev == nullptr) return SGEMV_ERR_ARG;
    if (!aligned16(w_dev) || !aligned32(packed_dev) || (status_dev && (reinterpret_cast<uintptr_t>(status_dev) & 3u)))
        return SGEMV_ERR_ALIGN;
    DeviceInfo di;
    rc = device_info(&di);
    if (rc != SGEMV_OK) return rc;
    PackParams p;
    p.w = static_cast<const uint16_t*>(w_dev);
    p.packed = static_cast<uint8_t*>(packed_dev);
    p.status = status_dev;
    p.L = *layout;
    p.log2g = 0;
    while ((1 << p.log2g) < layout->group) ++p.log2g;
    const int grid = std::max(1, std::min(layout->n, 8 * di.sm_count));
    return launch_pack(p, grid, static_cast<cudaStream_t>(stream)) == cudaSuccess ? SGEMV_OK : SGEMV_ERR_CUDA;
}

int sgemv_run(const sgemv_layout* layout, const void* packed_dev, const void* x_dev, int batch, void* y_dev,
              int32_t* status_dev, void* stream) {
    return run_one(layout, true, packed_dev, x_dev, batch, y_dev, status_dev, stream);
}

int sgemv_run_dense(const sgemv_layout* layout, const void* packed_dev, const void* x_dev, int batch, void* y_dev,
                    int32_t* status_dev, void* stream) {
    return run_one(layout, false, packed_dev, x_dev, batch, y_dev, status_dev, stream);
}

int sgemv_run_stack(const sgemv_layer* table, int n_layers, int batch, int32_t* status_dev, void* stream) {
    if (table == nullptr || n_layers < 1) return SGEMV_ERR_ARG;
    for (int i = 0; i < n_layers; ++i) {
        const sgemv_layer& l = table[i];
        const int rc = check_run_args(&l.layout, is_sparse(l.layout.format), l.packed_dev, l.x_dev, batch, l.y_dev,
                                      status_dev);
        if (rc != SGEMV_OK) return rc;
    }
    DeviceInfo di;
    int rc = device_info(&di);
    if (rc != SGEMV_OK) return rc;
    // consecutive independent layers of the same format run as one launch
    for (int g0 = 0; g0 < n_layers;) {
        if (streams(table[g0].layout, di, batch)) {
            StreamGroup sgp;
            int grid = 0;
            uint32_t smem = 0;
            if (plan_stream(table + g0, 1, batch, di, &sgp, &grid, &smem) == SGEMV_OK) {
                int g1 = g0 + 1;
                while (g1 < n_layers && g1 - g0 < kStreamMaxLayers && streams(table[g1].layout, di, batch) &&
                       table[g1].layout.group == table[g0].layout.group && can_join(table, g0, g1, batch)) {
                    StreamGroup trial;
                    int gt = 0;
                    uint32_t st = 0;
                    if (plan_stream(table + g0, g1 - g0 + 1, batch, di, &trial, &gt, &st) != SGEMV_OK) break;
                    sgp = trial;
                    grid = gt;
                    smem = st;
                    ++g1;
                }
                sgp.status = status_dev;
                const cudaError_t e =
                    launch_stream(table[g0].layout.format, batch, sgp, grid, smem, static_cast<cudaStream_t>(stream));
                if (e != cudaSuccess) return SGEMV_ERR_CUDA;
                g0 = g1;
                continue;
            }
        }
        int g1 = g0 + 1;
        // a layer split over K by clusters runs alone (a launch has one cluster shape)
        const auto splits = [&](int i) { return split_factor(table[i].layout.n, table[i].layout.k, di) > 1; };
        while (g1 < n_layers && !splits(g0) && !splits(g1) && can_join(table, g0, g1, batch)) ++g1;
        LayerGroup g;
        std::memset(&g, 0, sizeof(g));
        g.n_layers = g1 - g0;
        int grid = 0;
        uint32_t smem = 0;
        for (int i = g0; i < g1; ++i) {
            const sgemv_layer& l = table[i];
            int gi = 0;
            uint32_t si = 0;
            rc = plan_gemv(l.layout, l.packed_dev, l.x_dev, batch, l.y_dev, status_dev, di, &g.layer[i - g0], &gi, &si);
            if (rc != SGEMV_OK) return rc;
            grid = std::max(grid, gi);
            smem = std::max(smem, si);
        }
        const cudaError_t e = launch_group(table[g0].layout.format, batch, g, grid, smem,
                                           static_cast<cudaStream_t>(stream));
        if (e != cudaSuccess) return SGEMV_ERR_CUDA;
        g0 = g1;
    }
    return SGEMV_OK;
}

int sgemv_header_read(const void* header_host, uint64_t bytes, sgemv_layout* out) {
    if (header_host == nullptr || out == nullptr || bytes < 64) return SGEMV_ERR_ARG;
    const uint8_t* h = static_cast<const uint8_t*>(header_host);
    uint32_t w[6];
    uint64_t o[5];
    std::memcpy(w, h, 24);
    std::memcpy(o, h + 24, 40);
    if (w[0] != kMagic || w[1] != kVersion) return SGEMV_ERR_FORMAT;
    sgemv_layout L;
    const int rc = compute_layout(static_cast<int>(w[2]), static_cast<int>(w[3]), static_cast<int>(w[4]),
                                  static_cast<int>(w[5]), &L);
    if (rc != SGEMV_OK) return rc == SGEMV_ERR_ARG ? SGEMV_ERR_FORMAT : rc;
    if (o[0] != L.off_vals || o[1] != L.off_idx || o[2] != L.off_sz || o[3] != L.off_rowptr || o[4] != L.total_bytes)
        return SGEMV_ERR_FORMAT;
    *out = L;
    return SGEMV_OK;
}

int sgemv_header_check(const sgemv_layout* layout, const void* header_host, uint64_t bytes) {
    if (layout == nullptr) return SGEMV_ERR_ARG;
    sgemv_layout L;
    const int rc = sgemv_header_read(header_host, bytes, &L);
    if (rc == SGEMV_ERR_ARG) return rc;
    if (rc != SGEMV_OK) return SGEMV_ERR_FORMAT;
    return layout_equal(L, *layout) ? SGEMV_OK : SGEMV_ERR_FORMAT;
}

}  // extern "C"
