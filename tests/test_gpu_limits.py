"""GPU parity at the format's limits (K = 2^20 columns; N = 2^24 rows), against the CPU oracle.

Bars as in test_gpu_parity.py: packed bytes bit-exact, outputs within 4e-3 * sum_j |ŵ_ij x_j| + 2^-24.
The N = 2^24 layer is a seeded 1024-row tile repeated on the device (rows are packed and multiplied
independently, so row r of the layer must equal row r % 1024 of the tile, byte for byte and output for
output); the oracle packs and multiplies the tile.
"""

import numpy as np
import pytest

import oracle
import synth

pytestmark = pytest.mark.gpu

TOL_REL = 4e-3
TOL_ABS = 2.0 ** -24


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


def _close(y_gpu, y_ref, absdot):
    err = np.abs(y_gpu.astype(np.float64) - np.asarray(y_ref, dtype=np.float64))
    bound = TOL_REL * np.asarray(absdot, dtype=np.float64) + TOL_ABS
    assert np.all(err <= bound), f"max excess {np.max(err - bound)}"


@pytest.mark.parametrize("fmt", [1, 3, 2])
@pytest.mark.parametrize("batch,g", [(1, 256), (8, 64)])
def test_max_k(env, fmt, batch, g):
    """K = 2^20 (the format's limit): the x tile is a small part of K, so every CTA runs many x tiles."""
    sg, torch = env
    n, k = 5, 1 << 20
    w = synth.weights(n, k, "max-k", fmt, g)
    x = synth.activations(batch, k, "max-k", fmt, batch)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    layout, packed = sg.pack(torch.from_numpy(w).cuda(), fmt, g, status=status)
    ref = oracle.pack(w, fmt, g)
    assert np.array_equal(packed.cpu().numpy(), ref)
    y = sg.gemv(layout, packed, torch.from_numpy(x).cuda(), status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    y_ref, absdot = oracle.gemv(ref, x)
    _close(y.cpu().numpy(), y_ref, absdot)


@pytest.mark.parametrize("fmt", [1, 3, 2])
def test_max_n(env, fmt):
    """N = 2^24 (the format's limit), K = 128, g = 64: 110 k rows per CTA, hundreds of accumulator
    passes, sections of hundreds of MB."""
    sg, torch = env
    n, k, g, tile = 1 << 24, 128, 64, 1024
    wt = synth.weights(tile, k, "max-n", fmt)
    x = synth.activations(1, k, "max-n", fmt)
    ref = oracle.pack(wt, fmt, g)
    yt_ref, absdot = oracle.gemv(ref, x)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    w_dev = torch.from_numpy(wt).cuda().repeat(n // tile, 1)
    layout, packed = sg.pack(w_dev, fmt, g, status=status)
    del w_dev
    y = sg.gemv(layout, packed, torch.from_numpy(x).cuda(), status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    # packed rows: row r of every section equals row r % tile of the tile's packing
    L = layout.as_dict()
    T = oracle.layout(fmt, tile, k, g)
    rng = np.random.default_rng(fmt)
    rows = np.unique(np.concatenate([[0, tile - 1, tile, n - 1], rng.integers(0, n, 64)]))
    sections = [("off_vals", "vals_pitch"), ("off_sz", "sz_pitch")] + ([("off_idx", "idx_pitch")] if fmt != 2 else [])
    for off, pitch in sections:
        p = int(L[pitch])
        for r in rows:
            got = packed[int(L[off]) + int(r) * p: int(L[off]) + (int(r) + 1) * p].cpu().numpy()
            want = ref[int(T[off]) + int(r % tile) * p: int(T[off]) + (int(r % tile) + 1) * p]
            assert np.array_equal(got, want), (off, int(r))
    if fmt != 2:  # row_ptr[r] = r * kept per row
        rp = packed[int(L["off_rowptr"]): int(L["off_rowptr"]) + 4 * (n + 1)].cpu().numpy().view(np.int32)
        kept = k // 2 if fmt == 1 else k // 4
        assert np.array_equal(rp[rows], (rows * kept).astype(np.int32))
        assert int(rp[n]) == n * kept
    # every output row against the tile's oracle output
    yg = y.cpu().numpy().reshape(n // tile, tile)
    _close(yg, np.broadcast_to(np.asarray(yt_ref).reshape(1, tile), yg.shape),
           np.broadcast_to(np.asarray(absdot).reshape(1, tile), yg.shape))
