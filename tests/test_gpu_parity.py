"""GPU parity of the C-ABI library against the CPU oracle (needs a GB300).

Bars (from the packed-format definition and the method of the paper "Efficient LLM-based Advertising
via Model Compression and Parallel Verification", §3.2-§3.3; formats 2:4, 1:4 and dense):
  * packing is bit-exact: the GPU-packed buffer equals the oracle's byte for byte;
  * outputs: |y_gpu - y_oracle| <= 4e-3 * sum_j |ŵ_ij x_j| + 2^-24 per element, where y_oracle is the
    fp64 sum and 2^-24 is the spacing of fp16 subnormals (the output format's resolution near 0);
  * the integer-exact case (every product and partial sum an exactly representable integer) must match
    the oracle exactly after fp16 rounding.
Small shapes span several CTAs, ragged row counts, ragged 512-column slabs and several x tiles; the
full-size configurations are checked bit-exactly for packing and on sampled rows for the GEMV, in the
launch configuration the bench times.
"""

import numpy as np
import pytest

import oracle
import synth

pytestmark = pytest.mark.gpu

TOL_REL = 4e-3
TOL_ABS = 2.0 ** -24
SP, DN, S14 = 1, 2, 3


@pytest.fixture(scope="module")
def env():
    import torch
    import __graft_entry__
    __graft_entry__.build()
    import int4_weight_only_sgemv_gb300 as sg
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    return sg, torch


def _gpu_pack(env, w, fmt, g):
    sg, torch = env
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    layout, packed = sg.pack(torch.from_numpy(w).cuda(), fmt, g, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return layout, packed


def _gpu_gemv(env, layout, packed, x):
    sg, torch = env
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    y = sg.gemv(layout, packed, torch.from_numpy(x).cuda(), status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0, sg.sgemv_status_str(int(status.item()))
    return y.cpu().numpy()


def _assert_close(y_gpu, y_ref, absdot):
    err = np.abs(y_gpu.astype(np.float64) - y_ref)
    tol = TOL_REL * absdot + TOL_ABS
    bad = ~(err <= tol)
    assert not bad.any(), (f"{int(bad.sum())} of {bad.size} outside tolerance; worst err/tol "
                           f"{float(np.max(err / tol)):.3f}")


SMALL = [(1, 128), (7, 640), (152, 1152), (153, 2176), (300, 1152), (1024, 1024), (999, 9216)]


@pytest.mark.parametrize("fmt", [SP, DN, S14])
@pytest.mark.parametrize("g", [64, 128, 256])
@pytest.mark.parametrize("n,k", SMALL)
def test_pack_bit_exact(env, fmt, g, n, k):
    if k % g:
        pytest.skip("K not a multiple of g")
    dist = "t3" if (n + g) % 2 else "normal"
    w = synth.weights(n, k, "pack", fmt, g, n, k, dist=dist)
    _, packed = _gpu_pack(env, w, fmt, g)
    assert np.array_equal(packed.cpu().numpy(), oracle.pack(w, fmt, g))


def test_pack_ties_zeros_and_signed_zero(env):
    rng = np.random.default_rng(5)
    alphabet = np.array([0.0, -0.0, 1.0, -1.0, 0.5, -0.5, 2.0 ** -24, -(2.0 ** -20)], dtype=np.float16)
    w = alphabet[rng.integers(0, len(alphabet), (64, 1024))]
    w[3] = 0.0
    w[4] = -0.0
    w[5, :128] = 2.0 ** -24  # a group whose scale underflows
    for fmt in (SP, DN, S14):
        for g in (64, 256):
            _, packed = _gpu_pack(env, w, fmt, g)
            assert np.array_equal(packed.cpu().numpy(), oracle.pack(w, fmt, g))


@pytest.mark.parametrize("fmt", [SP, DN, S14])
@pytest.mark.parametrize("batch", [1, 2, 3, 4, 5, 6, 7, 8])
@pytest.mark.parametrize("n,k,g", [(300, 1152, 128), (153, 2176, 64), (999, 9216, 256), (7, 640, 128)])
def test_gemv_parity(env, fmt, batch, n, k, g):
    w = synth.weights(n, k, "gemv", fmt, n, k, g)
    x = synth.activations(batch, k, "gemv", fmt, n, k, g, batch)
    layout, packed = _gpu_pack(env, w, fmt, g)
    y = _gpu_gemv(env, layout, packed, x)
    y_ref, absdot = oracle.gemv(oracle.pack(w, fmt, g), x)
    _assert_close(y, y_ref, absdot)


@pytest.mark.parametrize("fmt", [SP, DN, S14])
@pytest.mark.parametrize("g", [64, 128, 256])
@pytest.mark.parametrize("batch", [1, 3, 8])
def test_gemv_integer_exact(env, fmt, g, batch):
    n, k = 333, 2048
    w, x = synth.integer_exact_case(n, k, g, batch, "gpu-exact", fmt, g, batch, kept=1 if fmt == S14 else 2)
    if fmt == DN:
        rng = np.random.default_rng(g + batch)
        wd = w.astype(np.float64)
        fill = rng.integers(-8, 8, wd.shape).astype(np.float64)
        wd[wd == 0] = fill[wd == 0]
        w = wd.astype(np.float16)
    layout, packed = _gpu_pack(env, w, fmt, g)
    y = _gpu_gemv(env, layout, packed, x)
    y_ref, _ = oracle.gemv(oracle.pack(w, fmt, g), x)
    assert np.array_equal(y, y_ref.astype(np.float16))


def test_many_passes_and_x_tiles(env):
    """N large enough that a CTA holds more rows than its shared-memory accumulator (several passes), and
    B*K large enough for several x tiles."""
    for (n, k, batch) in [(38917, 128, 1), (38917, 384, 2), (600, 12288, 8), (200, 9216, 5)]:
        for fmt in (SP, DN, S14):
            w = synth.weights(n, k, "tiles", fmt, n, k)
            x = synth.activations(batch, k, "tiles", fmt, n, k)
            layout, packed = _gpu_pack(env, w, fmt, 128)
            y = _gpu_gemv(env, layout, packed, x)
            y_ref, absdot = oracle.gemv(oracle.pack(w, fmt, 128), x)
            _assert_close(y, y_ref, absdot)


def test_special_activations(env):
    n, k = 256, 1024
    w = synth.weights(n, k, "special")
    for fmt in (SP, DN, S14):
        layout, packed = _gpu_pack(env, w, fmt, 128)
        ref_buf = oracle.pack(w, fmt, 128)
        x0 = np.zeros((2, k), dtype=np.float16)
        assert np.all(_gpu_gemv(env, layout, packed, x0) == 0)
        # large activations (outliers): fp32 accumulation must not overflow; y may exceed fp16 range
        xl = (synth.activations(2, k, "special-large").astype(np.float32) * 3000).astype(np.float16)
        y = _gpu_gemv(env, layout, packed, xl)
        y_ref, absdot = oracle.gemv(ref_buf, xl)
        finite = np.abs(y_ref) < 65504
        _assert_close(y[finite], y_ref[finite], absdot[finite])
        assert np.all(np.isinf(y[~finite]) & (np.sign(y[~finite]) == np.sign(y_ref[~finite])))


@pytest.mark.parametrize("fmt", [SP, DN, S14])
@pytest.mark.parametrize("batch", [1, 3, 8])
def test_outlier_columns(env, fmt, batch):
    """A few activation columns of magnitude 500-3000 among N(0, 1) ones, with heavy-tailed weights: the
    products of the outliers must neither overflow nor swamp the small columns' contributions, in rows
    whose other chunks hold only ordinary activations."""
    n, k = 600, 4096
    w = synth.weights(n, k, "outlier", fmt, batch, dist="t3")
    x = synth.activations(batch, k, "outlier", fmt, batch).astype(np.float32)
    rng = np.random.default_rng(batch + 10 * fmt)
    cols = rng.choice(k, 12, replace=False)
    x[:, cols] = rng.choice([-1, 1], (batch, 12)) * rng.uniform(500, 3000, (batch, 12))
    x = x.astype(np.float16)
    layout, packed = _gpu_pack(env, w, fmt, 128)
    y = _gpu_gemv(env, layout, packed, x)
    y_ref, absdot = oracle.gemv(oracle.pack(w, fmt, 128), x)
    _assert_close(y, y_ref, absdot)


@pytest.mark.parametrize("fmt", [SP, DN, S14])
def test_bounded_activations_at_32(env, fmt):
    """|x| up to exactly 32, with +-32 every 97 columns, and heavy-tailed weights at group size 64: large
    but ordinary partial sums; results must stay finite and within tolerance."""
    n, k, batch = 512, 4096, 2
    w = synth.weights(n, k, "threshold", fmt, dist="t3")
    u = synth.uniform53(synth.stream_key("threshold-x", fmt), batch * k).reshape(batch, k)
    x = ((u * 2 - 1) * 32).astype(np.float16)
    x[:, ::97] = 32.0
    x[:, 1::97] = -32.0
    layout, packed = _gpu_pack(env, w, fmt, 64)
    y = _gpu_gemv(env, layout, packed, x)
    y_ref, absdot = oracle.gemv(oracle.pack(w, fmt, 64), x)
    assert np.all(np.isfinite(y))
    _assert_close(y, y_ref, absdot)


def test_nonfinite_weights_reported(env):
    sg, torch = env
    w = synth.weights(64, 512, "nonfinite")
    w[10, 100] = np.inf
    for fmt in (SP, DN, S14):
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        sg.pack(torch.from_numpy(w).cuda(), fmt, 128, status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == sg.SGEMV_ERR_NONFINITE


def test_wrong_format_rejected_without_launch(env):
    sg, torch = env
    w = synth.weights(64, 512, "fmt")
    layout, packed = _gpu_pack(env, w, SP, 128)
    x = torch.zeros((1, 512), dtype=torch.float16, device="cuda")
    y = torch.full((1, 64), 7.0, dtype=torch.float16, device="cuda")
    with pytest.raises(sg.SgemvError) as e:
        sg.sgemv_run_dense(layout, packed, x, y)
    assert e.value.code == sg.SGEMV_ERR_FORMAT
    layout14, packed14 = _gpu_pack(env, w, S14, 128)
    with pytest.raises(sg.SgemvError) as e:
        sg.sgemv_run_dense(layout14, packed14, x, y)
    assert e.value.code == sg.SGEMV_ERR_FORMAT
    layout_d, packed_d = _gpu_pack(env, w, DN, 128)
    with pytest.raises(sg.SgemvError) as e:
        sg.sgemv_run(layout_d, packed_d, x, y)
    assert e.value.code == sg.SGEMV_ERR_FORMAT
    torch.cuda.synchronize()
    assert torch.all(y == 7.0)


@pytest.mark.parametrize("formats", [(SP, DN), (SP, S14, DN)])
def test_stack_dispatch_matches_oracle(env, formats):
    """A small layer-adaptive stack: per-layer format and group size, run through sgemv_run_stack
    (2:4 + dense, and the mixed-density {2:4, 1:4, dense} policy)."""
    sg, torch = env
    table = synth.stack_table(n_blocks=3, seed=3, scale=8, formats=formats)
    layers, refs = [], []
    for i, (name, n, k, fmt, g) in enumerate(table):
        w = synth.weights(n, k, "stack", i, name)
        x = synth.activations(1, k, "stack", i, name)
        layout, packed = _gpu_pack(env, w, fmt, g)
        xt = torch.from_numpy(x).cuda()
        yt = torch.empty((1, n), dtype=torch.float16, device="cuda")
        layers.append((layout, packed, xt, yt))
        refs.append(oracle.gemv(oracle.pack(w, fmt, g), x))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    sg.sgemv_run_stack(layers, 1, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert {fmt for (_, _, _, fmt, _) in table} == set(formats)
    for (layout, packed, xt, yt), (y_ref, absdot) in zip(layers, refs):
        _assert_close(yt.cpu().numpy(), y_ref, absdot)


@pytest.mark.parametrize("fmt", [SP, S14, DN])
def test_grouped_independent_layers(env, fmt):
    """Independent layers of one format run as one grouped launch (the dispatch groups them): layers with
    fewer rows than SMs (their own, narrower CTA partition) next to wide ones, different K, g and x tiles."""
    sg, torch = env
    shapes = [(7, 640, 64), (300, 1152, 128), (1, 2304, 256), (2000, 9216, 128), (152, 128, 64)]
    batch = 3
    layers, refs = [], []
    for i, (n, k, g) in enumerate(shapes):
        w = synth.weights(n, k, "group", fmt, i)
        x = synth.activations(batch, k, "group", fmt, i)
        layout, packed = _gpu_pack(env, w, fmt, g)
        yt = torch.full((batch, n), 7.0, dtype=torch.float16, device="cuda")
        layers.append((layout, packed, torch.from_numpy(x).cuda(), yt))
        refs.append(oracle.gemv(oracle.pack(w, fmt, g), x))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    sg.sgemv_run_stack(layers, batch, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for (layout, packed, xt, yt), (y_ref, absdot) in zip(layers, refs):
        _assert_close(yt.cpu().numpy(), y_ref, absdot)


def test_grouping_respects_data_flow(env):
    """Ten layers of one format: layer 3 reads layer 0's output and layer 7 writes into layer 8's input
    buffer before layer 8 reads it, so the dispatch must cut the groups there (and at 8 layers); every
    output must equal the oracle's on the input the layer actually saw."""
    sg, torch = env
    k = 1152
    n = k
    ws = [synth.weights(n, k, "flow", i) for i in range(10)]
    packs = [_gpu_pack(env, w, SP, 128) for w in ws]
    xs = [torch.from_numpy(synth.activations(2, k, "flow", i)).cuda() for i in range(10)]
    ys = [torch.empty((2, n), dtype=torch.float16, device="cuda") for _ in range(10)]
    xs[3] = ys[0]                     # layer 3 consumes layer 0
    ys[7] = xs[8]                     # layer 7 overwrites layer 8's input before layer 8 runs
    layers = [(packs[i][0], packs[i][1], xs[i], ys[i]) for i in range(10)]
    sg.sgemv_run_stack(layers, 2)
    torch.cuda.synchronize()
    outs = [y.cpu().numpy() for y in ys]
    for i in range(10):
        if i == 3:
            x_in = outs[0]
        elif i == 8:
            x_in = outs[7]
        else:
            x_in = synth.activations(2, k, "flow", i)
        y_ref, absdot = oracle.gemv(oracle.pack(ws[i], SP, 128), x_in)
        _assert_close(outs[i], y_ref, absdot)


def test_chained_layers_under_dependent_launch(env):
    """Layer i+1 reads layer i's output: the dependent-launch wait must order the two kernels."""
    sg, torch = env
    k = 2048
    ws = [synth.weights(k, k, "chain", i) for i in range(4)]
    x = synth.activations(2, k, "chain")
    layers = []
    xt = torch.from_numpy(x).cuda()
    cur = xt
    packs = []
    for i, w in enumerate(ws):
        layout, packed = _gpu_pack(env, w, (SP, DN, S14)[i % 3], 128)
        yt = torch.empty((2, k), dtype=torch.float16, device="cuda")
        layers.append((layout, packed, cur, yt))
        packs.append(oracle.pack(w, layout.format, 128))
        cur = yt
    sg.sgemv_run_stack(layers, 2)
    torch.cuda.synchronize()
    h = x
    for i, buf in enumerate(packs):
        y_gpu = layers[i][3].cpu().numpy()
        y_ref, absdot = oracle.gemv(buf, h)
        _assert_close(y_gpu, y_ref, absdot)
        h = y_gpu  # the next layer's oracle input is the GPU's fp16 output of this layer


# Full-size configurations, every output row compared with the oracle. The weights of a shape are drawn
# and packed once (on the GPU and by the oracle) and serve every batch of that shape.
SHAPES_7B = [(4096, 4096), (11008, 4096), (4096, 11008)]
SHAPES_WIDE = [(32000, 4096), (28672, 8192), (8192, 28672)]
FULL = ([("single-layer", 1024, 1024, 1, "normal", SP)]
        + [(f"7b-{n}x{k}-b1", n, k, 1, "normal", SP) for (n, k) in SHAPES_7B]
        + [(f"7b-{n}x{k}-b{b}", n, k, b, "normal", SP) for (n, k) in SHAPES_7B for b in (2, 4, 8)]
        + [(f"wide-{n}x{k}-b{b}", n, k, b, "t3", SP) for (n, k) in SHAPES_WIDE for b in (1, 8)]
        + [("7b-4096x11008-1of4-b1", 4096, 11008, 1, "normal", S14),
           ("7b-11008x4096-1of4-b8", 11008, 4096, 8, "normal", S14),
           ("7b-4096x11008-dense-b1", 4096, 11008, 1, "normal", DN)])

_full_cache = {}


def _full_layer(env, n, k, dist, fmt):
    """(layout, GPU-packed tensor, oracle bytes) of the full-size layer n x k; packing checked bit-exact."""
    key = (n, k, dist, fmt)
    if key not in _full_cache:
        if len(_full_cache) >= 2:  # keep at most two layers (host and device memory)
            _full_cache.clear()
        w = synth.weights(n, k, "full", n, k, dist=dist)
        layout, packed = _gpu_pack(env, w, fmt, 128)
        ref_buf = oracle.pack(w, fmt, 128)
        assert np.array_equal(packed.cpu().numpy(), ref_buf)
        _full_cache[key] = (layout, packed, ref_buf)
    return _full_cache[key]


@pytest.mark.parametrize("case", FULL, ids=[c[0] for c in FULL])
def test_full_size_configs(env, case):
    label, n, k, batch, dist, fmt = case
    layout, packed, ref_buf = _full_layer(env, n, k, dist, fmt)
    x = synth.activations(batch, k, "full", label)
    y = _gpu_gemv(env, layout, packed, x)
    y_ref, absdot = oracle.gemv(ref_buf, x)
    _assert_close(y, y_ref, absdot)


def test_full_layer_adaptive_stack(env):
    """The 224-layer layer-adaptive stack at its real shapes, formats and group sizes (32 blocks x
    {q, k, v, o, gate, up, down}, a seeded choice of 2:4 or dense INT4 and of g in {64, 128, 256} per
    layer), every layer packed on the GPU and run through sgemv_run_stack at batch 1 in one call, as the
    stack bench runs it. Each layer has its own x. Every output row of every layer is compared with the
    oracle; the packed bytes of one layer of each (shape, format, g) combination are compared exactly."""
    sg, torch = env
    table = synth.stack_table()
    assert len(table) == 224
    base, ref_bufs, checked = {}, {}, set()
    layers, xs = [], []
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for i, (name, n, k, fmt, g) in enumerate(table):
        if (n, k) not in base:
            base[(n, k)] = synth.weights(n, k, "stack-full", n, k)
        layout, packed = sg.pack(torch.from_numpy(base[(n, k)]).cuda(), fmt, g, status=status)
        combo = (n, k, fmt, g)
        if combo not in ref_bufs:
            ref_bufs[combo] = oracle.pack(base[(n, k)], fmt, g)
        if combo not in checked:
            torch.cuda.synchronize()
            assert np.array_equal(packed.cpu().numpy(), ref_bufs[combo]), name
            checked.add(combo)
        x = synth.activations(1, k, "stack-full", i)
        xs.append(x)
        layers.append((layout, packed, torch.from_numpy(x).cuda(),
                       torch.full((1, n), 7.0, dtype=torch.float16, device="cuda")))
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert {fmt for (_, _, _, fmt, _) in table} == {SP, DN} and {g for (*_, g) in table} == {64, 128, 256}
    sg.sgemv_run_stack(layers, 1, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for i, ((name, n, k, fmt, g), (_, _, _, yt)) in enumerate(zip(table, layers)):
        y_ref, absdot = oracle.gemv(ref_bufs[(n, k, fmt, g)], xs[i])
        _assert_close(yt.cpu().numpy(), y_ref, absdot)


# few rows and a long K: clusters of 8, 4 and 2 (uneven block shares included)
SPLIT = [(1, 32768, 128), (3, 33792, 64), (19, 65536, 256), (37, 40960, 128), (76, 32768, 64)]
# few rows and a short K: streamed without a split
FEW_ROWS = [(1, 4096, 128), (3, 2304, 64), (19, 8192, 256), (37, 11008, 128), (76, 2048, 64)]


@pytest.mark.parametrize("fmt", [SP, DN, S14])
@pytest.mark.parametrize("batch", [1, 8])
@pytest.mark.parametrize("n,k,g", SPLIT + FEW_ROWS)
def test_split_k_few_rows(env, fmt, batch, n, k, g):
    """Layers with fewer rows than SMs: with K of 32768 columns or more they run split over K by
    clusters of 2, 4 or 8 CTAs (their partial sums added through distributed shared memory), with a
    shorter K they stream unsplit; outputs within the tolerance of the oracle's."""
    w = synth.weights(n, k, "split", fmt, n, k)
    x = synth.activations(batch, k, "split", fmt, batch)
    layout, packed = _gpu_pack(env, w, fmt, g)
    y = _gpu_gemv(env, layout, packed, x)
    y_ref, absdot = oracle.gemv(oracle.pack(w, fmt, g), x)
    _assert_close(y, y_ref, absdot)


@pytest.mark.parametrize("fmt", [SP, S14])
def test_split_k_integer_exact(env, fmt):
    """Split-K on the integer-exact case: every product and partial sum is an exact integer, so the
    cluster's sums must equal the oracle's exactly."""
    n, k, g, batch = 19, 32768, 128, 3
    w, x = synth.integer_exact_case(n, k, g, batch, "split-exact", fmt, kept=1 if fmt == S14 else 2)
    layout, packed = _gpu_pack(env, w, fmt, g)
    y = _gpu_gemv(env, layout, packed, x)
    y_ref, _ = oracle.gemv(oracle.pack(w, fmt, g), x)
    assert np.array_equal(y, y_ref.astype(np.float16))


def test_split_k_layers_in_a_stack(env):
    """A stack mixing layers split over K with ordinary ones: the dispatch launches each split layer on
    its own and groups the others."""
    sg, torch = env
    shapes = [(4096, 1024, 128, SP), (19, 32768, 128, SP), (300, 1152, 128, SP), (3, 33792, 64, DN),
              (1024, 2048, 64, DN), (37, 40960, 128, S14), (19, 8192, 128, SP)]
    batch = 2
    layers, refs = [], []
    for i, (n, k, g, fmt) in enumerate(shapes):
        w = synth.weights(n, k, "split-stack", i)
        x = synth.activations(batch, k, "split-stack", i)
        layout, packed = _gpu_pack(env, w, fmt, g)
        yt = torch.full((batch, n), 7.0, dtype=torch.float16, device="cuda")
        layers.append((layout, packed, torch.from_numpy(x).cuda(), yt))
        refs.append(oracle.gemv(oracle.pack(w, fmt, g), x))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    sg.sgemv_run_stack(layers, batch, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for (layout, packed, xt, yt), (y_ref, absdot) in zip(layers, refs):
        _assert_close(yt.cpu().numpy(), y_ref, absdot)


@pytest.mark.parametrize("fmt", [SP, DN, S14])
def test_streamed_layers_reproducible(env, fmt):
    """A streamed layer sums each row in a fixed order: repeated runs, alone or grouped with other
    layers in one launch, give bit-identical y."""
    sg, torch = env
    shapes = [(4096, 4096), (11008, 4096), (4096, 11008)]
    batch = 2
    layers = []
    for i, (n, k) in enumerate(shapes):
        w = synth.weights(n, k, "repro", fmt, i)
        x = synth.activations(batch, k, "repro", fmt, i)
        layout, packed = _gpu_pack(env, w, fmt, 128)
        layers.append((layout, packed, torch.from_numpy(x).cuda(),
                       torch.empty((batch, n), dtype=torch.float16, device="cuda")))
    runs = []
    for _ in range(3):
        alone = []
        for layout, packed, xt, _ in layers:
            alone.append(sg.gemv(layout, packed, xt).cpu().numpy())
        sg.sgemv_run_stack(layers, batch)
        torch.cuda.synchronize()
        runs.append((alone, [yt.cpu().numpy() for (_, _, _, yt) in layers]))
    for alone, grouped in runs:
        for a, b, c in zip(alone, grouped, runs[0][0]):
            # the same per-row order alone or grouped: identical, and identical across runs
            assert np.array_equal(a.view(np.uint16), c.view(np.uint16))
            assert np.array_equal(b.view(np.uint16), c.view(np.uint16))


@pytest.mark.parametrize("fmt", [SP, S14, DN])
@pytest.mark.parametrize("g", [64, 128, 256])
@pytest.mark.parametrize("batch", [1, 2, 3])
def test_grouped_copy_engine_x(env, fmt, g, batch):
    """Groups of three or more independent layers of one format and group size fetch x with the copy
    engine when their x rows are at most 24 KB each and 96 KB in all: a 4-layer group with ragged K
    (K % 256 == 128 where g allows), then a 3-layer group whose last x row is too long for the copy
    engine (plain loads), both through sgemv_run_stack; every output against the oracle."""
    sg, torch = env
    ks = [1152 if g != 256 else 1280, 4096, 2176 if g == 64 else 2304, 640 if g != 256 else 768]
    groups = [[(300, k) for k in ks], [(200, 1024), (152, 2048), (96, 13312 if g != 256 else 13568)]]
    for gi, shapes in enumerate(groups):
        layers, refs = [], []
        for i, (n, k) in enumerate(shapes):
            w = synth.weights(n, k, "copyx", fmt, g, gi, i)
            x = synth.activations(batch, k, "copyx", fmt, g, gi, i)
            layout, packed = _gpu_pack(env, w, fmt, g)
            yt = torch.full((batch, n), 7.0, dtype=torch.float16, device="cuda")
            layers.append((layout, packed, torch.from_numpy(x).cuda(), yt))
            refs.append(oracle.gemv(oracle.pack(w, fmt, g), x))
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        sg.sgemv_run_stack(layers, batch, status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        for (layout, packed, xt, yt), (y_ref, absdot) in zip(layers, refs):
            _assert_close(yt.cpu().numpy(), y_ref, absdot)
