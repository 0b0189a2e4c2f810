"""Thin Python binding of libsgemv.so, the GB300 INT4 + 2:4 "2bit-CSR" SparseGemv library.

The functions below carry the names of the C ABI (include/sgemv.h) and only marshal arguments: every
step of packing and of the GEMV runs in the library's CUDA kernels. PyTorch tensors serve as device
memory and streams. There is no fallback: if the compiled library is missing, importing this package
raises ImportError (build it with ``python int4_weight_only_sgemv_gb300/build.py`` or
``__graft_entry__.build()``).

Method: the paper "Efficient LLM-based Advertising via Model Compression and Parallel Verification",
§3.2 (group-wise INT4 weight-only quantisation, layer-adaptive 2:4 sparsity) and §3.3 (2bit-CSR index,
SparseGemv kernel). Byte layout: packed format v1.
"""

from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libsgemv.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is missing: build the CUDA library first "
        "(python int4_weight_only_sgemv_gb300/build.py, or __graft_entry__.build())")

_lib = ctypes.CDLL(LIB_PATH)

SGEMV_OK = 0
SGEMV_ERR_ARG = -1
SGEMV_ERR_SHAPE = -2
SGEMV_ERR_ALIGN = -3
SGEMV_ERR_FORMAT = -4
SGEMV_ERR_CUDA = -5
SGEMV_ERR_NONFINITE = -6
SGEMV_ERR_TIMEOUT = -7

SGEMV_FMT_SPARSE24 = 1
SGEMV_FMT_DENSE = 2
SGEMV_FMT_SPARSE14 = 3

EXPORTED = ("sgemv_layout_query", "sgemv_pack", "sgemv_run", "sgemv_run_dense", "sgemv_run_stack",
            "sgemv_beam_step", "sgemv_beam_traceback", "sgemv_beam_decode",
            "sgemv_header_read", "sgemv_header_check", "sgemv_status_str", "sgemv_abi_version")


class Layout(ctypes.Structure):
    """sgemv_layout (include/sgemv.h)."""

    _fields_ = [("format", ctypes.c_int32), ("n", ctypes.c_int32), ("k", ctypes.c_int32),
                ("group", ctypes.c_int32), ("vals_pitch", ctypes.c_uint64),
                ("idx_pitch", ctypes.c_uint64), ("sz_pitch", ctypes.c_uint64),
                ("off_vals", ctypes.c_uint64), ("off_idx", ctypes.c_uint64),
                ("off_sz", ctypes.c_uint64), ("off_rowptr", ctypes.c_uint64),
                ("total_bytes", ctypes.c_uint64)]

    def as_dict(self) -> dict:
        return {name: getattr(self, name) for name, _ in self._fields_}

    def __repr__(self) -> str:
        return f"Layout({self.as_dict()})"


class Layer(ctypes.Structure):
    """sgemv_layer: one row of the per-layer dispatch table."""

    _fields_ = [("layout", Layout), ("packed_dev", ctypes.c_void_p), ("x_dev", ctypes.c_void_p),
                ("y_dev", ctypes.c_void_p)]


class Trie(ctypes.Structure):
    """sgemv_trie: the prefix tree in CSR form (device arrays)."""

    _fields_ = [("n_nodes", ctypes.c_int32), ("n_edges", ctypes.c_int32), ("child_ptr_dev", ctypes.c_void_p),
                ("child_tok_dev", ctypes.c_void_p), ("child_node_dev", ctypes.c_void_p)]


_c = ctypes
_lib.sgemv_beam_step.argtypes = [_c.POINTER(Trie), _c.c_int, _c.c_int] + [_c.c_void_p] * 3 + [_c.c_int] + \
    [_c.c_void_p] * 7
_lib.sgemv_beam_traceback.argtypes = [_c.c_int, _c.c_int] + [_c.c_void_p] * 6
_lib.sgemv_beam_decode.argtypes = [_c.POINTER(Trie), _c.c_int, _c.c_int, _c.c_int, _c.c_void_p, _c.c_void_p,
                                   _c.POINTER(_c.c_void_p), _c.c_int, _c.c_int] + [_c.c_void_p] * 8
_lib.sgemv_layout_query.argtypes = [_c.c_int, _c.c_int, _c.c_int, _c.c_int, _c.POINTER(Layout)]
_lib.sgemv_pack.argtypes = [_c.POINTER(Layout), _c.c_void_p, _c.c_void_p, _c.c_void_p, _c.c_void_p]
_lib.sgemv_run.argtypes = [_c.POINTER(Layout), _c.c_void_p, _c.c_void_p, _c.c_int, _c.c_void_p,
                           _c.c_void_p, _c.c_void_p]
_lib.sgemv_run_dense.argtypes = _lib.sgemv_run.argtypes
_lib.sgemv_run_stack.argtypes = [_c.POINTER(Layer), _c.c_int, _c.c_int, _c.c_void_p, _c.c_void_p]
_lib.sgemv_header_read.argtypes = [_c.c_void_p, _c.c_uint64, _c.POINTER(Layout)]
_lib.sgemv_header_check.argtypes = [_c.POINTER(Layout), _c.c_void_p, _c.c_uint64]
_lib.sgemv_status_str.argtypes = [_c.c_int]
_lib.sgemv_status_str.restype = _c.c_char_p
_lib.sgemv_abi_version.argtypes = []
for _name in EXPORTED:
    if _name != "sgemv_status_str":
        getattr(_lib, _name).restype = _c.c_int


class SgemvError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {sgemv_status_str(code)} ({code})")
        self.code = code


def _check(code: int, what: str) -> None:
    if code != SGEMV_OK:
        raise SgemvError(code, what)


def _addr(t) -> int | None:
    """Device (or host) address of a tensor, an int address, or None."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream if torch.cuda.is_available() else None
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


# ---------------------------------------------------------------------------------------------- C ABI

def sgemv_abi_version() -> int:
    return _lib.sgemv_abi_version()


def sgemv_status_str(code: int) -> str:
    return _lib.sgemv_status_str(int(code)).decode()


def sgemv_layout_query(fmt: int, n: int, k: int, group: int) -> Layout:
    out = Layout()
    _check(_lib.sgemv_layout_query(fmt, n, k, group, ctypes.byref(out)), "sgemv_layout_query")
    return out


def _check_tensor(t, shape, dtype_name, what):
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{what}: expected a torch.Tensor")
    if not t.is_cuda or not t.is_contiguous() or str(t.dtype) != dtype_name:
        raise ValueError(f"{what}: expected a contiguous CUDA {dtype_name} tensor")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{what}: expected shape {tuple(shape)}, got {tuple(t.shape)}")


def _check_packed(layout: Layout, packed):
    import torch
    if not isinstance(packed, torch.Tensor) or not packed.is_cuda or packed.dtype != torch.uint8:
        raise ValueError("packed: expected a CUDA uint8 tensor")
    if packed.numel() < layout.total_bytes or not packed.is_contiguous():
        raise ValueError(f"packed: need {layout.total_bytes} contiguous bytes")


def sgemv_pack(layout: Layout, w, packed, status=None, stream=None) -> None:
    """Pack fp16 w[n][k] (CUDA tensor) into `packed` (CUDA uint8 tensor of layout.total_bytes)."""
    _check_tensor(w, (layout.n, layout.k), "torch.float16", "w")
    _check_packed(layout, packed)
    _check(_lib.sgemv_pack(ctypes.byref(layout), _addr(w), _addr(packed), _addr(status), _stream(stream)),
           "sgemv_pack")


def _run(fn, name, layout, packed, x, y, status, stream):
    _check_packed(layout, packed)
    if x.dim() != 2:
        raise ValueError("x: expected [batch, k]")
    batch = x.shape[0]
    _check_tensor(x, (batch, layout.k), "torch.float16", "x")
    _check_tensor(y, (batch, layout.n), "torch.float16", "y")
    _check(fn(ctypes.byref(layout), _addr(packed), _addr(x), batch, _addr(y), _addr(status), _stream(stream)),
           name)


def sgemv_run(layout: Layout, packed, x, y, status=None, stream=None) -> None:
    """y[b] = Ŵ x[b] for a SPARSE24 or SPARSE14 layer (x: fp16 [batch, k], y: fp16 [batch, n], batch 1..8)."""
    _run(_lib.sgemv_run, "sgemv_run", layout, packed, x, y, status, stream)


def sgemv_run_dense(layout: Layout, packed, x, y, status=None, stream=None) -> None:
    """y[b] = Ŵ x[b] for a DENSE INT4 layer."""
    _run(_lib.sgemv_run_dense, "sgemv_run_dense", layout, packed, x, y, status, stream)


def sgemv_run_stack(layers, batch: int, status=None, stream=None) -> None:
    """Run a dispatch table: layers = [(layout, packed, x, y), ...] in order, each with the kernel of
    its format. Tensor sizes are checked here; the table is marshalled into sgemv_layer rows."""
    Stack(layers, batch).run(status, stream)


class Stack:
    """A dispatch table marshalled once: the tensors of `layers` = [(layout, packed, x, y), ...] are
    checked and their addresses written into sgemv_layer rows here; each run() is one sgemv_run_stack
    call on the same buffers (the caller keeps the tensors alive and their contents current)."""

    def __init__(self, layers, batch: int):
        self.batch = int(batch)
        self.table = (Layer * len(layers))()
        self._keep = list(layers)  # the addresses in the table point into these tensors
        for i, (layout, packed, x, y) in enumerate(layers):
            _check_packed(layout, packed)
            _check_tensor(x, (batch, layout.k), "torch.float16", f"layers[{i}].x")
            _check_tensor(y, (batch, layout.n), "torch.float16", f"layers[{i}].y")
            self.table[i].layout = layout
            self.table[i].packed_dev = _addr(packed)
            self.table[i].x_dev = _addr(x)
            self.table[i].y_dev = _addr(y)

    def run(self, status=None, stream=None) -> None:
        _check(_lib.sgemv_run_stack(self.table, len(self.table), self.batch, _addr(status), _stream(stream)),
               "sgemv_run_stack")


def sgemv_header_read(header: bytes) -> Layout:
    out = Layout()
    buf = ctypes.create_string_buffer(bytes(header), len(header))
    _check(_lib.sgemv_header_read(buf, len(header), ctypes.byref(out)), "sgemv_header_read")
    return out


def sgemv_header_check(layout: Layout, header: bytes) -> int:
    buf = ctypes.create_string_buffer(bytes(header), len(header))
    return _lib.sgemv_header_check(ctypes.byref(layout), buf, len(header))


# ---------------------------------------------------------------------------------------------- helpers

def pack(w, fmt: int, group: int, status=None, stream=None):
    """Allocate a packed buffer (torch) and pack fp16 w[n][k] into it. Returns (layout, packed)."""
    import torch
    layout = sgemv_layout_query(fmt, w.shape[0], w.shape[1], group)
    packed = torch.empty(layout.total_bytes, dtype=torch.uint8, device=w.device)
    sgemv_pack(layout, w, packed, status, stream)
    return layout, packed


def gemv(layout: Layout, packed, x, out=None, status=None, stream=None):
    """y = Ŵ x for any format (x: fp16 [batch, k]); allocates y unless `out` is given."""
    import torch
    if out is None:
        out = torch.empty((x.shape[0], layout.n), dtype=torch.float16, device=x.device)
    fn = sgemv_run_dense if layout.format == SGEMV_FMT_DENSE else sgemv_run
    fn(layout, packed, x, out, status, stream)
    return out


def algorithmic_bytes(layout: Layout, batch: int) -> int:
    """Bytes a GEMV must move at minimum: the layer's vals, idx and scale entries (unpadded), plus x
    and y. Row offsets are not read by the kernels (every row keeps the same number of elements)."""
    n, k, g = layout.n, layout.k, layout.group
    weights = n * (layout.vals_pitch + layout.idx_pitch + 4 * (k // g))
    return int(weights + 2 * batch * k + 2 * batch * n)


# ---------------------------------------------------------------------------------------------- beam step

MAX_BEAM = 64


def make_trie(child_ptr, child_tok, child_node):
    """Device copy of a CSR prefix tree (int32 tensors); returns (Trie, tensors to keep alive)."""
    import torch
    t = [torch.as_tensor(a, dtype=torch.int32).cuda().contiguous() for a in (child_ptr, child_tok, child_node)]
    tr = Trie(int(t[0].numel()) - 1, int(t[1].numel()), t[0].data_ptr(), t[1].data_ptr(), t[2].data_ptr())
    return tr, t


def sgemv_beam_step(trie: Trie, node, score, logp, k: int, out, status=None, stream=None) -> None:
    """One trie-constrained beam-score step. node: int32 [beam_in], score: fp32 [beam_in], logp: fp32
    [beam_in, vocab] (device). out = (node, score, parent, tok, count) device tensors with >= k entries."""
    beam_in, vocab = int(logp.shape[0]), int(logp.shape[1])
    _check_tensor(node, (beam_in,), "torch.int32", "node")
    _check_tensor(score, (beam_in,), "torch.float32", "score")
    _check_tensor(logp, (beam_in, vocab), "torch.float32", "logp")
    o_node, o_score, o_parent, o_tok, o_count = out
    for t, dt, nm in ((o_node, "torch.int32", "out node"), (o_score, "torch.float32", "out score"),
                      (o_parent, "torch.int32", "out parent"), (o_tok, "torch.int32", "out tok")):
        if str(t.dtype) != dt or t.numel() < k or not t.is_contiguous():
            raise ValueError(f"{nm}: need a contiguous {dt} tensor of >= {k} entries")
    _check(_lib.sgemv_beam_step(ctypes.byref(trie), beam_in, vocab, _addr(node), _addr(score), _addr(logp), int(k),
                                _addr(o_node), _addr(o_score), _addr(o_parent), _addr(o_tok), _addr(o_count),
                                _addr(status), _stream(stream)), "sgemv_beam_step")


def sgemv_beam_decode(trie: Trie, node, score, logps, k: int, out, seq, shared_row: bool = False,
                      status=None, stream=None) -> None:
    """Every step of one decode plus the traceback, one launch. node: int32 [beam_in], score: fp32
    [beam_in] (the first step's beams); logps: a list of `steps` fp32 device tensors, step t's
    [rows, vocab] (rows >= k, or >= beam_in at step 0; one row when shared_row: the position's
    distribution for every beam). out = (node, score, parent, tok) int32/fp32 [steps, k] and count int32
    [steps]; seq: int32 [k, steps]."""
    steps = len(logps)
    beam_in = int(node.shape[0])
    vocab = int(logps[0].shape[-1])
    _check_tensor(node, (beam_in,), "torch.int32", "node")
    _check_tensor(score, (beam_in,), "torch.float32", "score")
    for t, lp in enumerate(logps):
        rows = 1 if shared_row else (beam_in if t == 0 else k)
        if lp.dim() != 2 or lp.shape[1] != vocab or lp.shape[0] < rows:
            raise ValueError(f"logps[{t}]: need [>= {rows}, {vocab}]")
        _check_tensor(lp, None, "torch.float32", f"logps[{t}]")
    o_node, o_score, o_parent, o_tok, o_count = out
    for t, dt, nm in ((o_node, "torch.int32", "out node"), (o_score, "torch.float32", "out score"),
                      (o_parent, "torch.int32", "out parent"), (o_tok, "torch.int32", "out tok")):
        _check_tensor(t, (steps, k), dt, nm)
    _check_tensor(o_count, (steps,), "torch.int32", "out count")
    _check_tensor(seq, (k, steps), "torch.int32", "seq")
    ptrs = (ctypes.c_void_p * steps)(*[lp.data_ptr() for lp in logps])
    _check(_lib.sgemv_beam_decode(ctypes.byref(trie), steps, vocab, beam_in, _addr(node), _addr(score), ptrs,
                                  0 if shared_row else vocab, int(k), _addr(o_node), _addr(o_score),
                                  _addr(o_parent), _addr(o_tok), _addr(o_count), _addr(seq), _addr(status),
                                  _stream(stream)), "sgemv_beam_decode")


def sgemv_beam_traceback(parent, tok, count, seq, status=None, stream=None) -> None:
    """parent, tok: int32 [steps, beam_max]; count: int32 [1]; seq: int32 [beam_max, steps] (output)."""
    steps, beam_max = int(parent.shape[0]), int(parent.shape[1])
    _check_tensor(tok, (steps, beam_max), "torch.int32", "tok")
    _check_tensor(seq, (beam_max, steps), "torch.int32", "seq")
    _check(_lib.sgemv_beam_traceback(steps, beam_max, _addr(parent), _addr(tok), _addr(count), _addr(seq),
                                     _addr(status), _stream(stream)), "sgemv_beam_traceback")
