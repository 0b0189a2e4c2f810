"""Out-of-bounds writes, checked with guard bands (the pool has no sanitizer): the packed buffer and y
are views into larger device buffers whose margins hold a sentinel pattern; after packing and after the
GEMV (single layers, split-K layers and a grouped stack) every margin byte must be unchanged and the
results must still match the oracle."""

import numpy as np
import pytest

import oracle
import synth

pytestmark = pytest.mark.gpu

GUARD = 4096  # bytes on each side (a multiple of 256: the views keep the buffers' alignment)
SENTINEL = 0xA5


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


def _guarded(torch, nbytes):
    """A device byte buffer of GUARD + nbytes + GUARD filled with the sentinel; returns (buffer, view)."""
    buf = torch.full((GUARD + nbytes + GUARD,), SENTINEL, dtype=torch.uint8, device="cuda")
    return buf, buf[GUARD:GUARD + nbytes]


def _margins_intact(buf, nbytes):
    b = buf.cpu().numpy()
    return bool(np.all(b[:GUARD] == SENTINEL) and np.all(b[GUARD + nbytes:] == SENTINEL))


def _close(y, y_ref, absdot):
    err = np.abs(y.astype(np.float64) - np.asarray(y_ref, dtype=np.float64))
    assert np.all(err <= 4e-3 * np.asarray(absdot, dtype=np.float64) + 2.0 ** -24)


CASES = [(1, 300, 1152, 128, 1), (1, 153, 2176, 64, 8), (2, 999, 9216, 256, 3), (3, 7, 640, 128, 2),
         (1, 19, 8192, 128, 1), (1, 19, 32768, 128, 1), (3, 5, 65536, 64, 8),
         (2, 3, 33792, 64, 4)]  # the last three split over K


@pytest.mark.parametrize("fmt,n,k,g,batch", CASES)
def test_pack_and_gemv_write_nothing_outside(env, fmt, n, k, g, batch):
    sg, torch = env
    w = synth.weights(n, k, "guard", fmt, n, k)
    x = synth.activations(batch, k, "guard", fmt, batch)
    layout = sg.sgemv_layout_query(fmt, n, k, g)
    pbuf, packed = _guarded(torch, layout.total_bytes)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    sg.sgemv_pack(layout, torch.from_numpy(w).cuda(), packed, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert _margins_intact(pbuf, layout.total_bytes), "packing wrote outside its buffer"
    ref = oracle.pack(w, fmt, g)
    assert np.array_equal(packed.cpu().numpy(), ref)
    ybuf, yv = _guarded(torch, 2 * batch * n)
    y = yv.view(torch.float16).view(batch, n)
    sg.gemv(layout, packed, torch.from_numpy(x).cuda(), out=y, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert _margins_intact(pbuf, layout.total_bytes), "the GEMV wrote into the packed buffer's margins"
    assert _margins_intact(ybuf, 2 * batch * n), "the GEMV wrote outside y"
    y_ref, absdot = oracle.gemv(ref, x)
    _close(y.cpu().numpy(), y_ref, absdot)


def test_stack_writes_nothing_outside(env):
    """A grouped stack (several layers in one launch) next to a split layer: every y stays in bounds."""
    sg, torch = env
    shapes = [(300, 1152, 128, 1), (4096, 1024, 64, 2), (19, 32768, 128, 1), (1000, 2048, 256, 3)]
    batch = 2
    layers, refs, guards = [], [], []
    for i, (n, k, g, fmt) in enumerate(shapes):
        w = synth.weights(n, k, "guard-stack", i)
        x = synth.activations(batch, k, "guard-stack", i)
        layout, packed = sg.pack(torch.from_numpy(w).cuda(), fmt, g)
        ybuf, yv = _guarded(torch, 2 * batch * n)
        layers.append((layout, packed, torch.from_numpy(x).cuda(), yv.view(torch.float16).view(batch, n)))
        guards.append((ybuf, 2 * batch * n))
        refs.append(oracle.gemv(oracle.pack(w, fmt, g), x))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    sg.sgemv_run_stack(layers, batch, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for (ybuf, nbytes), (layout, packed, xt, yt), (y_ref, absdot) in zip(guards, layers, refs):
        assert _margins_intact(ybuf, nbytes)
        _close(yt.cpu().numpy(), y_ref, absdot)
