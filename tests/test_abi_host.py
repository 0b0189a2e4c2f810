"""Host-side checks of the C ABI (no GPU needed): the library loads, exports every function declared in
include/sgemv.h, computes the same layout as the independently written oracle, parses headers the
oracle writes, and rejects bad arguments before touching the GPU."""

import ctypes
import os
import re

import numpy as np
import pytest

import oracle
import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def sg():
    import __graft_entry__
    __graft_entry__.build()
    import int4_weight_only_sgemv_gb300 as sg
    return sg


def _declared_functions():
    text = open(os.path.join(ROOT, "include", "sgemv.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(sgemv_[a-z_]+)\s*\(", text)))


def test_exports_every_declared_symbol(sg):
    names = _declared_functions()
    assert len(names) >= 9
    lib = ctypes.CDLL(sg.LIB_PATH)
    for name in names:
        assert hasattr(lib, name), name
    assert set(names) == set(sg.EXPORTED)
    assert sg.sgemv_abi_version() == 1


@pytest.mark.parametrize("fmt", [1, 2, 3])
@pytest.mark.parametrize("n,k,g", [(1, 128, 64), (1024, 1024, 128), (4096, 11008, 128), (32000, 4096, 256),
                                   (8192, 28672, 64), (37, 384, 128)])
def test_layout_matches_oracle(sg, fmt, n, k, g):
    L = sg.sgemv_layout_query(fmt, n, k, g).as_dict()
    O = oracle.layout(fmt, n, k, g)
    for key in ("vals_pitch", "idx_pitch", "sz_pitch", "off_vals", "off_idx", "off_sz", "off_rowptr",
                "total_bytes"):
        assert L[key] == O[key], key
    assert (L["format"], L["n"], L["k"], L["group"]) == (fmt, n, k, g)


def test_layout_rejects_bad_shapes(sg):
    for args, code in [((1, 0, 128, 128), sg.SGEMV_ERR_SHAPE), ((1, 4, 100, 64), sg.SGEMV_ERR_SHAPE),
                       ((1, 4, 384, 256), sg.SGEMV_ERR_SHAPE), ((1, 4, 128, 32), sg.SGEMV_ERR_SHAPE),
                       ((9, 4, 128, 128), sg.SGEMV_ERR_ARG), ((1, 1 << 25, 128, 128), sg.SGEMV_ERR_SHAPE)]:
        with pytest.raises(sg.SgemvError) as e:
            sg.sgemv_layout_query(*args)
        assert e.value.code == code


def test_layout_rejects_row_offsets_beyond_int32(sg):
    """row_ptr is int32 (packed format v1, section 7.4): a sparse layer whose N times kept elements per row
    passes 2^31 - 1 is rejected by both the library and the oracle; dense layers have no row_ptr."""
    for fmt, n, k in [(1, 1 << 24, 256), (3, 1 << 24, 512), (1, 131072, 32768)]:
        with pytest.raises(sg.SgemvError) as e:
            sg.sgemv_layout_query(fmt, n, k, 128)
        assert e.value.code == sg.SGEMV_ERR_SHAPE
        with pytest.raises(oracle.OracleError):
            oracle.layout(fmt, n, k, 128)
    # the largest admissible rows: N*K/2 = 2^30 and N*K/4 = 2^31 - 2^20 < 2^31
    for fmt, n, k in [(1, 1 << 24, 128), (3, (1 << 24) - 4096, 512), (2, 1 << 24, 256)]:
        L = sg.sgemv_layout_query(fmt, n, k, 128).as_dict()
        assert L["total_bytes"] == oracle.layout(fmt, n, k, 128)["total_bytes"]


def test_header_read_and_check_on_oracle_bytes(sg):
    w = synth.weights(9, 256, "hdr-abi")
    buf = oracle.pack(w, 1, 64)
    L = sg.sgemv_header_read(bytes(buf[:64]))
    assert L.as_dict() == sg.sgemv_layout_query(1, 9, 256, 64).as_dict()
    assert sg.sgemv_header_check(L, bytes(buf[:64])) == sg.SGEMV_OK
    other = sg.sgemv_layout_query(2, 9, 256, 64)
    assert sg.sgemv_header_check(other, bytes(buf[:64])) == sg.SGEMV_ERR_FORMAT
    buf14 = oracle.pack(w, 3, 64)
    L14 = sg.sgemv_header_read(bytes(buf14[:64]))
    assert L14.as_dict() == sg.sgemv_layout_query(3, 9, 256, 64).as_dict()
    assert sg.sgemv_header_check(L14, bytes(buf14[:64])) == sg.SGEMV_OK
    assert sg.sgemv_header_check(L, bytes(buf14[:64])) == sg.SGEMV_ERR_FORMAT
    bad = bytearray(buf[:64])
    bad[0] ^= 1
    with pytest.raises(sg.SgemvError) as e:
        sg.sgemv_header_read(bytes(bad))
    assert e.value.code == sg.SGEMV_ERR_FORMAT
    bad = bytearray(buf[:64])
    bad[24] ^= 0x10  # off_vals
    with pytest.raises(sg.SgemvError):
        sg.sgemv_header_read(bytes(bad))
    with pytest.raises(sg.SgemvError) as e:
        sg.sgemv_header_read(bytes(buf[:32]))
    assert e.value.code == sg.SGEMV_ERR_ARG


def test_run_argument_errors_before_any_launch(sg):
    """Raw C calls with invalid arguments return their status without touching CUDA (no GPU here)."""
    lib = ctypes.CDLL(sg.LIB_PATH)
    lib.sgemv_run.argtypes = sg._lib.sgemv_run.argtypes
    lib.sgemv_run_dense.argtypes = sg._lib.sgemv_run_dense.argtypes
    lib.sgemv_pack.argtypes = sg._lib.sgemv_pack.argtypes
    lib.sgemv_run_stack.argtypes = sg._lib.sgemv_run_stack.argtypes
    Ls = sg.sgemv_layout_query(1, 64, 256, 128)
    Ld = sg.sgemv_layout_query(2, 64, 256, 128)
    L14 = sg.sgemv_layout_query(3, 64, 256, 128)
    P, X, Y = 0x10000, 0x20000, 0x30000  # fake, never dereferenced on these paths
    ref = ctypes.byref
    assert lib.sgemv_run(None, P, X, 1, Y, None, None) == sg.SGEMV_ERR_ARG
    assert lib.sgemv_run(ref(Ls), None, X, 1, Y, None, None) == sg.SGEMV_ERR_ARG
    assert lib.sgemv_run(ref(Ls), P, X, 0, Y, None, None) == sg.SGEMV_ERR_ARG
    assert lib.sgemv_run(ref(Ls), P, X, 9, Y, None, None) == sg.SGEMV_ERR_ARG
    assert lib.sgemv_run(ref(Ls), P + 8, X, 1, Y, None, None) == sg.SGEMV_ERR_ALIGN
    assert lib.sgemv_run(ref(Ls), P + 16, X, 1, Y, None, None) == sg.SGEMV_ERR_ALIGN  # packed: 32 bytes
    assert lib.sgemv_run(ref(Ls), P, X + 2, 1, Y, None, None) == sg.SGEMV_ERR_ALIGN
    assert lib.sgemv_run(ref(Ld), P, X, 1, Y, None, None) == sg.SGEMV_ERR_FORMAT
    assert lib.sgemv_run_dense(ref(Ls), P, X, 1, Y, None, None) == sg.SGEMV_ERR_FORMAT
    assert lib.sgemv_run_dense(ref(L14), P, X, 1, Y, None, None) == sg.SGEMV_ERR_FORMAT
    broken = sg.Layout.from_buffer_copy(Ls)
    broken.off_sz += 256
    assert lib.sgemv_run(ref(broken), P, X, 1, Y, None, None) == sg.SGEMV_ERR_FORMAT
    broken = sg.Layout.from_buffer_copy(Ls)
    broken.k = 100
    assert lib.sgemv_run(ref(broken), P, X, 1, Y, None, None) == sg.SGEMV_ERR_SHAPE
    # y may overlap neither x nor the packed buffer; the status word must be 4-byte aligned
    assert lib.sgemv_run(ref(Ls), P, X, 1, X + 64, None, None) == sg.SGEMV_ERR_ARG
    assert lib.sgemv_run(ref(Ls), P, X, 2, X - 128, None, None) == sg.SGEMV_ERR_ARG  # y (256 B) runs into x
    assert lib.sgemv_run(ref(Ls), P, X, 1, P + 256, None, None) == sg.SGEMV_ERR_ARG
    assert lib.sgemv_run_dense(ref(Ld), P, X, 1, P + Ld.total_bytes - 16, None, None) == sg.SGEMV_ERR_ARG
    assert lib.sgemv_run(ref(Ls), P, X, 1, Y, Y + 4096 + 2, None) == sg.SGEMV_ERR_ALIGN
    assert lib.sgemv_pack(ref(Ls), None, P, None, None) == sg.SGEMV_ERR_ARG
    assert lib.sgemv_pack(ref(Ls), X + 4, P, None, None) == sg.SGEMV_ERR_ALIGN
    table = (sg.Layer * 2)()
    table[0].layout, table[0].packed_dev, table[0].x_dev, table[0].y_dev = Ls, P, X, Y
    table[1].layout, table[1].packed_dev, table[1].x_dev, table[1].y_dev = Ld, P, X, None
    assert lib.sgemv_run_stack(table, 2, 1, None, None) == sg.SGEMV_ERR_ARG  # row 1 has no y
    assert lib.sgemv_run_stack(table, 0, 1, None, None) == sg.SGEMV_ERR_ARG
    assert lib.sgemv_run_stack(None, 1, 1, None, None) == sg.SGEMV_ERR_ARG


def test_beam_decode_argument_errors_before_any_launch(sg):
    """sgemv_beam_decode rejects invalid arguments before touching CUDA (no GPU here)."""
    lib = ctypes.CDLL(sg.LIB_PATH)
    lib.sgemv_beam_decode.argtypes = sg._lib.sgemv_beam_decode.argtypes
    A = 0x10000  # fake device addresses, never dereferenced on these paths
    trie = sg.Trie(10, 9, A, A + 64, A + 128)
    logp = (ctypes.c_void_p * 4)(A + 256, A + 512, A + 768, A + 1024)
    outs = [A + 2048 + 64 * i for i in range(6)]

    def call(trie_p=ctypes.byref(trie), steps=4, vocab=100, beam_in=1, node=A, score=A + 32, lp=logp, stride=100,
             k=8, o=outs):
        return lib.sgemv_beam_decode(trie_p, steps, vocab, beam_in, node, score, lp, stride, k, *o, None, None)

    assert call(trie_p=None) == sg.SGEMV_ERR_ARG
    assert call(steps=0) == sg.SGEMV_ERR_ARG
    assert call(steps=33) == sg.SGEMV_ERR_ARG
    assert call(beam_in=0) == sg.SGEMV_ERR_ARG
    assert call(beam_in=65) == sg.SGEMV_ERR_ARG
    assert call(k=0) == sg.SGEMV_ERR_ARG
    assert call(k=65) == sg.SGEMV_ERR_ARG
    assert call(stride=7) == sg.SGEMV_ERR_ARG          # neither 0 nor vocab
    assert call(lp=None) == sg.SGEMV_ERR_ARG
    assert call(node=None) == sg.SGEMV_ERR_ARG
    assert call(o=outs[:5] + [None]) == sg.SGEMV_ERR_ARG  # seq
    holes = (ctypes.c_void_p * 4)(A + 256, None, A + 768, A + 1024)
    assert call(lp=holes) == sg.SGEMV_ERR_ARG
    assert call(node=A + 2) == sg.SGEMV_ERR_ALIGN
    odd = (ctypes.c_void_p * 4)(A + 256, A + 514, A + 768, A + 1024)
    assert call(lp=odd) == sg.SGEMV_ERR_ALIGN


def test_status_strings(sg):
    for code in range(-7, 1):
        assert sg.sgemv_status_str(code).startswith("SGEMV_")
    assert sg.sgemv_status_str(-99) == "SGEMV_ERR_UNKNOWN"


def test_algorithmic_bytes_closed_form(sg):
    L = sg.sgemv_layout_query(1, 4096, 11008, 128)
    assert sg.algorithmic_bytes(L, 1) == 4096 * (11008 // 4 + 11008 // 8 + 4 * 11008 // 128) + 2 * 11008 + 2 * 4096
    D = sg.sgemv_layout_query(2, 4096, 4096, 128)
    assert sg.algorithmic_bytes(D, 2) == 4096 * (4096 // 2 + 4 * 32) + 4 * 4096 + 4 * 4096
