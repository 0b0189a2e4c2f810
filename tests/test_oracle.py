"""Pins for the CPU oracle, each against something other than the oracle itself.

Method source: the paper "Efficient LLM-based Advertising via Model Compression and Parallel
Verification", §3.2 (group-wise INT4 quantisation, 2:4 and 1:4 magnitude pruning) and §3.3 (2bit-CSR
index, SparseGemv). Byte layout: packed format v1.

Pins used:
  * fp16 conversions      -- numpy's IEEE binary16 conversion (exhaustive / large random sets);
  * layout                -- closed-form section sizes; the paper's 30% index ratio (golden file);
  * pruning               -- invariants of "keep the 2 (1:4: the 1) largest |w| of 4, ties to the lower
                             column", and an exhaustive small-alphabet enumeration;
  * quantisation          -- exactly representable weights round-trip exactly; the rounding error
                             bound |ŵ - w| <= 0.51 s; zero maps to zero; all-zero group closed form;
  * encoding              -- hand-worked examples for 2:4 and 1:4 (golden files); header, row_ptr,
                             zero padding;
  * GEMV                  -- exact integer case against numpy's matmul of the original W; random case
                             within the quantisation error bound of numpy's matmul of the kept W.
"""

import os

import numpy as np
import pytest

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
SP, DN, S14 = oracle.FMT_SPARSE24, oracle.FMT_DENSE, oracle.FMT_SPARSE14


# ---------------------------------------------------------------------------------------------- fp16

def test_half_to_float_exhaustive():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float32)
    got = np.array([oracle.half_to_float(int(b)) for b in bits], dtype=np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def test_float_to_half_matches_numpy():
    rng = np.random.default_rng(1)
    # wide magnitude range incl. subnormal fp16, overflow, and exact ties between fp16 neighbours
    mags = np.exp2(rng.uniform(-30, 17, 20000)).astype(np.float32)
    signs = np.where(rng.random(20000) < 0.5, -1, 1).astype(np.float32)
    vals = list(mags * signs)
    h = np.arange(0, 0x7C00, 7, dtype=np.uint16)
    lo = h.view(np.float16).astype(np.float64)
    hi = (h + 1).view(np.float16).astype(np.float64)
    ties = ((lo + hi) / 2).astype(np.float32)  # midpoints are exact in binary32
    vals += list(ties) + list(-ties)
    vals += [0.0, -0.0, 65504.0, 65519.0, 65520.0, 1e-8, 2.0 ** -25, 2.0 ** -24, 3 * 2.0 ** -26]
    vals = np.array(vals, dtype=np.float32)
    with np.errstate(over="ignore"):
        ref = vals.astype(np.float16).view(np.uint16)
    got = np.array([oracle.float_to_half(float(v)) for v in vals], dtype=np.uint16)
    assert np.array_equal(got, ref)


# ---------------------------------------------------------------------------------------------- layout

@pytest.mark.parametrize("n,k,g", [(1024, 1024, 128), (4096, 4096, 128), (11008, 4096, 128),
                                   (4096, 11008, 128), (32000, 4096, 128), (8192, 28672, 64),
                                   (3, 384, 128)])
def test_layout_closed_form(n, k, g):
    L = oracle.layout(SP, n, k, g)
    assert L["vals_pitch"] == k // 4 and L["idx_pitch"] == k // 8
    assert L["sz_pitch"] == -(-4 * (k // g) // 16) * 16
    assert L["off_vals"] == 256
    for key in ("off_vals", "off_idx", "off_sz", "off_rowptr", "total_bytes"):
        assert L[key] % 256 == 0
    up = lambda v: -(-v // 256) * 256
    assert L["off_idx"] == 256 + up(n * k // 4)
    assert L["off_sz"] == L["off_idx"] + up(n * k // 8)
    assert L["off_rowptr"] == L["off_sz"] + up(n * L["sz_pitch"])
    assert L["total_bytes"] == L["off_rowptr"] + up(4 * (n + 1))
    if g == 128 and (4 * k // g) % 16 == 0:
        # nibbles (K/4) + 2-bit positions of K/2 kept (K/8) + scales (4K/g) = 0.40625 bytes per
        # dense weight at g = 128
        assert (k // 4 + k // 8 + 4 * k // g) == 0.40625 * k
    D = oracle.layout(DN, n, k, g)
    assert D["vals_pitch"] == k // 2 and D["idx_pitch"] == 0
    assert D["off_idx"] == D["off_sz"] and D["off_rowptr"] == D["total_bytes"]
    Q = oracle.layout(S14, n, k, g)
    assert Q["vals_pitch"] == k // 8 and Q["idx_pitch"] == k // 16 and Q["kept_per_row"] == k // 4
    assert Q["off_idx"] == 256 + up(n * k // 8)
    assert Q["off_sz"] == Q["off_idx"] + up(n * k // 16)
    assert Q["off_rowptr"] == Q["off_sz"] + up(n * Q["sz_pitch"])
    assert Q["total_bytes"] == Q["off_rowptr"] + up(4 * (n + 1))


def test_index_ratio_is_the_papers_30_percent():
    with open(os.path.join(GOLDEN, "index_ratio.txt")) as f:
        ratio = float([ln.split()[1] for ln in f if ln.startswith("ratio")][0])
    for fmt in (SP, S14):
        for k in (1024, 4096, 11008 // 128 * 128, 28672):
            L = oracle.layout(fmt, 1, k, 128)
            kept = L["kept_per_row"]
            two_bit_csr = L["vals_pitch"] + L["idx_pitch"]          # INT4 + 2-bit positions
            plain_csr = L["vals_pitch"] + 2 * kept                  # INT4 + uint16_t column indices
            assert two_bit_csr / plain_csr == pytest.approx(ratio, abs=1e-12)


def test_bad_shapes_rejected():
    for fmt, n, k, g in [(SP, 0, 128, 128), (SP, 4, 100, 64), (SP, 4, 192, 128), (SP, 4, 128, 32),
                         (7, 4, 128, 128), (DN, 4, 64, 64)]:
        with pytest.raises(oracle.OracleError):
            oracle.layout(fmt, n, k, g)


def test_nonfinite_rejected():
    w = np.zeros((2, 128), dtype=np.float16)
    for bad in (np.inf, -np.inf, np.nan):
        w2 = w.copy()
        w2[1, 77] = bad
        with pytest.raises(oracle.OracleError) as e:
            oracle.pack(w2, SP, 128)
        assert e.value.code == -6


# ---------------------------------------------------------------------------------------------- pruning

def _adversarial_w(n, k, seed):
    """Random rows mixed with blocks built from a tiny alphabet so ties and zeros are common."""
    rng = np.random.default_rng(seed)
    alphabet = np.array([0.0, -0.0, 1.0, -1.0, 2.0, -2.0, 0.5], dtype=np.float16)
    w = synth.weights(n, k, "prune", seed)
    mask = rng.random((n, k)) < 0.5
    w[mask] = alphabet[rng.integers(0, len(alphabet), mask.sum())]
    return w


@pytest.mark.parametrize("seed", [0, 1])
def test_pruning_invariants(seed):
    n, k = 24, 512
    w = _adversarial_w(n, k, seed)
    buf = oracle.pack(w, SP, 128)
    cols = oracle.unpack(buf)["col"]
    mag = np.abs(w.astype(np.float32))
    for r in range(n):
        c = cols[r].reshape(-1, 2)                 # (blocks, 2) kept columns, in kept order
        blk = np.arange(k // 4)
        assert np.all(c[:, 0] // 4 == blk) and np.all(c[:, 1] // 4 == blk)   # two per block
        assert np.all(c[:, 0] < c[:, 1])                                      # p0 < p1
        for t in range(k // 4):
            kept = set(c[t].tolist())
            dropped = [4 * t + p for p in range(4) if 4 * t + p not in kept]
            for kc in kept:
                for dc in dropped:
                    assert mag[r, kc] >= mag[r, dc]
                    if mag[r, kc] == mag[r, dc]:
                        assert kc < dc                                        # tie -> lower column


@pytest.mark.parametrize("seed", [0, 1])
def test_pruning_invariants_1of4(seed):
    n, k = 24, 512
    w = _adversarial_w(n, k, seed)
    buf = oracle.pack(w, S14, 128)
    cols = oracle.unpack(buf)["col"]
    mag = np.abs(w.astype(np.float32))
    for r in range(n):
        c = cols[r]
        assert np.array_equal(c // 4, np.arange(k // 4))                     # one per block, in order
        for t in range(k // 4):
            for p in range(4):
                d = 4 * t + p
                if d == c[t]:
                    continue
                assert mag[r, c[t]] >= mag[r, d]
                if mag[r, c[t]] == mag[r, d]:
                    assert c[t] < d                                           # tie -> lower column
    # the dequantised matrix has at most one non-zero per block, where the kept column is
    w_hat = oracle.dequant(buf)
    assert np.all((w_hat.reshape(n, -1, 4) != 0).sum(-1) <= 1)


def test_pruning_exhaustive_small_alphabet():
    vals = np.array([0.0, 1.0, -1.0, 2.0, -2.0], dtype=np.float16)
    combos = np.array(np.meshgrid(*[np.arange(5)] * 4, indexing="ij")).reshape(4, -1).T  # 625 blocks
    k = 4 * 640  # 640 blocks per row, 625 used, rest zero
    w = np.zeros((1, k), dtype=np.float16)
    w[0, :4 * 625] = vals[combos].reshape(-1)
    cols = oracle.unpack(oracle.pack(w, SP, 64))["col"][0].reshape(-1, 2)
    cols14 = oracle.unpack(oracle.pack(w, S14, 64))["col"][0]
    mag = np.abs(vals[combos].astype(np.float32))
    for t in range(625):
        order = sorted(range(4), key=lambda p: (-mag[t, p], p))   # rank: magnitude desc, column asc
        assert sorted(order[:2]) == [c - 4 * t for c in cols[t]]
        assert order[0] == cols14[t] - 4 * t


# ---------------------------------------------------------------------------------------------- quantisation

def test_worked_example_bytes():
    fx = {}
    with open(os.path.join(GOLDEN, "worked_example_sparse24.txt")) as f:
        for ln in f:
            if ln.startswith("#") or not ln.strip():
                continue
            key, *rest = ln.split()
            fx[key] = rest
    w = np.zeros((1, 128), dtype=np.float16)
    for item in fx["input_nonzero"]:
        c, v = item.split(":")
        w[0, int(c)] = float(v)
    buf = oracle.pack(w, SP, 128)
    L = oracle.layout(SP, 1, 128, 128)
    vals = buf[L["off_vals"]:L["off_vals"] + 32].view(np.uint32)
    idx = buf[L["off_idx"]:L["off_idx"] + 16].view(np.uint16)
    sz = buf[L["off_sz"]:L["off_sz"] + 4].view(np.uint32)
    assert vals[0] == int(fx["vals_word0"][0], 16)
    assert np.all(vals[1:] == int(fx["vals_word_rest"][0], 16))
    assert idx[0] == int(fx["idx_word0"][0], 16)
    assert np.all(idx[1:] == int(fx["idx_word_rest"][0], 16))
    assert sz[0] == int(fx["sz_word0"][0], 16)


def test_worked_example_bytes_1of4():
    fx = {}
    with open(os.path.join(GOLDEN, "worked_example_sparse14.txt")) as f:
        for ln in f:
            if ln.startswith("#") or not ln.strip():
                continue
            key, *rest = ln.split()
            fx[key] = rest
    w = np.zeros((1, 128), dtype=np.float16)
    for t in range(16):                      # group 0: v_t = 0.0625 (t - 8) at position t % 4
        w[0, 4 * t + t % 4] = 0.0625 * (t - 8)
    w[0, 64:66] = np.float16(-0.0)           # block 16: [-0, -0, 0, 0]
    buf = oracle.pack(w, S14, 64)
    L = oracle.layout(S14, 1, 128, 64)
    assert L["vals_pitch"] == 16 and L["idx_pitch"] == 8
    vals = buf[L["off_vals"]:L["off_vals"] + 16].view(np.uint32)
    idx = buf[L["off_idx"]:L["off_idx"] + 8].view(np.uint16)
    sz = buf[L["off_sz"]:L["off_sz"] + 8].view(np.uint32)
    rp = buf[L["off_rowptr"]:L["off_rowptr"] + 8].view(np.int32)
    assert [int(v) for v in vals] == [int(h, 16) for h in fx["vals_words"]]
    assert [int(v) for v in idx] == [int(h, 16) for h in fx["idx_words"]]
    assert [int(v) for v in sz] == [int(h, 16) for h in fx["sz_words"]]
    assert [int(v) for v in rp] == [int(v) for v in fx["row_ptr"]]
    y, _ = oracle.gemv(buf, np.ones((1, 128), dtype=np.float16))
    assert y[0, 0] == float(fx["y_ones"][0])


@pytest.mark.parametrize("fmt", [SP, DN, S14])
@pytest.mark.parametrize("g", [64, 128, 256])
def test_exactly_representable_roundtrip(fmt, g):
    """W = (q - z) * s with a power-of-two s and an integer z chosen per group, and each group spanning
    the full code range: quantisation must reproduce W bit for bit (a wrong group index, nibble slot
    or position decode would not)."""
    n, k = 6, 512
    rng = np.random.default_rng(g + fmt)
    kept_per_block = {SP: 2, S14: 1}.get(fmt, 4)
    w = np.zeros((n, k))
    for r in range(n):
        for G in range(k // g):
            s = 2.0 ** int(rng.integers(-9, -2))
            z = int(rng.integers(1, 15))
            for t in range(G * g // 4, (G + 1) * g // 4):
                pos = np.sort(rng.choice(4, kept_per_block, replace=False))
                for p in pos:
                    w[r, 4 * t + p] = (int(rng.integers(0, 16)) - z) * s
            # the group's extremes: code 0 in its first block, code 15 in its second block
            w[r, G * g:G * g + 4] = [(0 - z) * s, 0.0, 0.0, 0.0]
            w[r, G * g + 4:G * g + 8] = [0.0, (15 - z) * s, 0.0, 0.0]
    w16 = w.astype(np.float16)
    assert np.array_equal(w16.astype(np.float64), w)
    if fmt != DN:  # at most kept_per_block non-zeros per block, so pruning keeps every non-zero
        assert np.all((w16.reshape(n, -1, 4) != 0).sum(-1) <= kept_per_block)
    w_hat = oracle.dequant(oracle.pack(w16, fmt, g))
    assert np.array_equal(w_hat, w)


@pytest.mark.parametrize("fmt", [SP, DN, S14])
@pytest.mark.parametrize("g,dist", [(64, "normal"), (128, "normal"), (256, "normal"), (128, "t3")])
def test_quantisation_error_bound(fmt, g, dist):
    n, k = 32, 1024
    w = synth.weights(n, k, "qbound", g, dist, dist=dist)
    buf = oracle.pack(w, fmt, g)
    w_hat = oracle.dequant(buf)
    u = oracle.unpack(buf)
    s = u["s16"].view(np.float16).astype(np.float64)     # [n][k/g]
    z = u["z16"].view(np.float16).astype(np.float64)
    assert np.all(z == np.round(z)) and np.all((z >= 0) & (z <= 15))
    assert np.all((u["q"] >= 0) & (u["q"] <= 15))
    s_col = np.repeat(s, g, axis=1)
    kept = np.zeros((n, k), dtype=bool)
    np.put_along_axis(kept, u["col"].astype(np.int64), True, axis=1)
    wf = w.astype(np.float64)
    normal_s = s_col >= 2.0 ** -14
    err = np.abs(w_hat - wf)
    assert np.all(err[kept & normal_s] <= 0.51 * s_col[kept & normal_s])
    assert np.all(w_hat[~kept] == 0.0)
    assert np.all(w_hat[kept & (wf == 0)] == 0.0)        # zero is exact
    # within a group, the code q is monotone in the value
    for r in range(4):
        for G in range(k // g):
            m = (u["col"][r] // g) == G
            v = wf[r, u["col"][r][m]]
            q = u["q"][r][m].astype(int)
            o = np.argsort(v, kind="stable")
            assert np.all(np.diff(q[o]) >= 0)


def test_all_zero_group_closed_form():
    w = np.zeros((2, 256), dtype=np.float16)
    w[1, 200] = 0.5  # second group of row 1 non-zero
    u = oracle.unpack(oracle.pack(w, SP, 128))
    assert u["s16"][0, 0] == 0x3C00 and u["z16"][0, 0] == 0 and np.all(u["q"][0] == 0)
    assert u["s16"][1, 0] == 0x3C00 and u["z16"][1, 0] == 0
    assert u["s16"][1, 1] != 0x3C00


def test_header_rowptr_padding_and_determinism():
    n, k, g = 5, 384, 128  # 4*k/g = 12 bytes -> sz rows padded to 16
    w = synth.weights(n, k, "hdr")
    buf = oracle.pack(w, SP, g)
    assert np.array_equal(buf, oracle.pack(w, SP, g))
    h = oracle.header(buf)
    L = oracle.layout(SP, n, k, g)
    assert h["magic"] == 0x564D4753 and bytes(buf[:4]) == b"SGMV" and h["version"] == 1
    assert (h["format"], h["n"], h["k"], h["g"]) == (SP, n, k, g)
    for key in ("off_vals", "off_idx", "off_sz", "off_rowptr", "total_bytes"):
        assert h[key] == L[key]
    assert buf.size == L["total_bytes"]
    assert np.all(buf[64:256] == 0)
    rp = buf[L["off_rowptr"]:L["off_rowptr"] + 4 * (n + 1)].view(np.int32)
    assert np.array_equal(rp, np.arange(n + 1) * (k // 2))
    assert np.all(buf[L["off_rowptr"] + 4 * (n + 1):] == 0)
    assert np.all(buf[L["off_vals"] + n * k // 4:L["off_idx"]] == 0)
    sz = buf[L["off_sz"]:L["off_sz"] + n * 16].reshape(n, 16)
    assert np.all(sz[:, 12:] == 0)
    buf14 = oracle.pack(w, S14, g)
    L14 = oracle.layout(S14, n, k, g)
    assert oracle.header(buf14)["format"] == S14 and buf14.size == L14["total_bytes"]
    rp = buf14[L14["off_rowptr"]:L14["off_rowptr"] + 4 * (n + 1)].view(np.int32)
    assert np.array_equal(rp, np.arange(n + 1) * (k // 4))
    assert np.all(buf14[L14["off_vals"] + n * k // 8:L14["off_idx"]] == 0)
    assert np.all(buf14[L14["off_idx"] + n * k // 16:L14["off_sz"]] == 0)


# ---------------------------------------------------------------------------------------------- GEMV

@pytest.mark.parametrize("fmt", [SP, DN, S14])
@pytest.mark.parametrize("g", [64, 128, 256])
def test_gemv_integer_exact(fmt, g):
    n, k, batch = 12, 512, 3
    w, x = synth.integer_exact_case(n, k, g, batch, "gemv-exact", fmt, g, kept=1 if fmt == S14 else 2)
    if fmt == DN:  # dense: fill the dropped slots with small integers, keep the [-8, 7] range
        rng = np.random.default_rng(g)
        wd = w.astype(np.float64)
        fill = rng.integers(-8, 8, wd.shape).astype(np.float64)
        wd[wd == 0] = fill[wd == 0]
        w = wd.astype(np.float16)
    y, absdot = oracle.gemv(oracle.pack(w, fmt, g), x)
    ref = x.astype(np.float64) @ w.astype(np.float64).T  # numpy matmul of the ORIGINAL W
    assert np.array_equal(y, ref)
    assert np.array_equal(absdot, np.abs(x.astype(np.float64)) @ np.abs(w.astype(np.float64)).T)


@pytest.mark.parametrize("fmt", [SP, DN, S14])
@pytest.mark.parametrize("g,dist", [(128, "normal"), (64, "t3")])
def test_gemv_within_quantisation_bound(fmt, g, dist):
    n, k, batch = 40, 1024, 2
    w = synth.weights(n, k, "gemv-bound", fmt, g, dist=dist)
    x = synth.activations(batch, k, "gemv-bound", fmt, g)
    buf = oracle.pack(w, fmt, g)
    u = oracle.unpack(buf)
    kept = np.zeros((n, k), dtype=bool)
    np.put_along_axis(kept, u["col"].astype(np.int64), True, axis=1)
    wk = np.where(kept, w.astype(np.float64), 0.0)
    xf = x.astype(np.float64)
    y, _ = oracle.gemv(buf, x)
    s_col = np.repeat(u["s16"].view(np.float16).astype(np.float64), g, axis=1)
    bound = np.abs(xf) @ (0.51 * s_col * kept).T + 1e-12
    assert np.all(np.abs(y - xf @ wk.T) <= bound)
    # and the row-subset entry point agrees with the full one
    rows = np.array([n - 1, 0, 17])
    y2, _ = oracle.gemv(buf, x, rows=rows)
    assert np.array_equal(y2, y[:, rows])
    # brute-force dense product of the decoded matrix
    assert np.allclose(y, xf @ oracle.dequant(buf).T, rtol=1e-12, atol=1e-12)
