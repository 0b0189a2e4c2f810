"""Seeded synthetic inputs shared by the tests, the bench and the oracle checks (a module of its own:
neither the GPU library nor the oracle imports it, and it holds no packing or GEMV arithmetic).

This module holds only random-number generation; none of the packing or GEMV arithmetic. Both the GPU
path and the CPU oracle receive the exact fp16 bits it produces.

Generator: splitmix64 on a counter (Steele, Lea and Flood, "Fast splittable pseudorandom number
generators", OOPSLA 2014), keyed per stream. Uniforms use the top 53 bits; normals use both branches
of the Box-Muller transform in binary64, one 64-bit output per pair; Student's t with nu degrees of
freedom is Z / sqrt(chi2_nu / nu) with chi2_nu a sum of nu squared normals from separate sub-streams.
Values are rounded to fp16 with numpy's round-to-nearest-even conversion.

Workload recipe (the paper's ERNIE 1.5B layers and datasets are not available; LLM-shaped synthetic
layers stand in for them):
  * weights  W ~ N(0, 0.02^2) (standard deviation 0.02), or 0.02 * StudentT(3) for heavy-tailed rows;
  * activations x ~ N(0, 1), rows independent for batch > 1.
"""

from __future__ import annotations

import os
import zlib

import numpy as np

_M64 = np.uint64(0xFFFFFFFFFFFFFFFF)
_GOLDEN = np.uint64(0x9E3779B97F4A7C15)


def _splitmix64(counter: np.ndarray) -> np.ndarray:
    with np.errstate(over="ignore"):
        z = counter * _GOLDEN  # the stream state after `counter` steps (state_0 = key)
        z = (z ^ (z >> np.uint64(30))) * np.uint64(0xBF58476D1CE4E5B9)
        z = (z ^ (z >> np.uint64(27))) * np.uint64(0x94D049BB133111EB)
        return z ^ (z >> np.uint64(31))


def stream_key(*parts) -> int:
    """A 64-bit key from any labels (config name, layer index, role, seed ...)."""
    text = "/".join(str(p) for p in parts).encode()
    lo = zlib.crc32(text)
    hi = zlib.crc32(text[::-1] + b"#")
    return (hi << 32) | lo


def _bits(key: int, start: int, count: int) -> np.ndarray:
    """splitmix64 outputs for counters start .. start+count-1 of stream `key`."""
    with np.errstate(over="ignore"):
        ctr = np.arange(start, start + count, dtype=np.uint64) + np.uint64(1)
        ctr += np.uint64(key & 0xFFFFFFFFFFFFFFFF) * np.uint64(0xD1B54A32D192ED03)
    return _splitmix64(ctr)


def uniform53(key: int, count: int, offset: int = 0) -> np.ndarray:
    """count uniforms in (0, 1] from stream `key`, starting at counter `offset`."""
    bits = _bits(key, offset, count)
    return ((bits >> np.uint64(11)).astype(np.float64) + 1.0) * (1.0 / 9007199254740992.0)


_CHUNK = 1 << 20


def _chunked(total: int, fill) -> None:
    """Run fill(start, count) over [0, total) in chunks of _CHUNK, on a few threads when there are many
    chunks (numpy releases the GIL inside these array operations; every chunk is independent because
    the generator is counter-based, so the values do not depend on the threading)."""
    starts = list(range(0, total, _CHUNK))
    if len(starts) < 4:
        for p0 in starts:
            fill(p0, min(_CHUNK, total - p0))
        return
    from concurrent.futures import ThreadPoolExecutor
    with ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 1)) as ex:
        list(ex.map(lambda p0: fill(p0, min(_CHUNK, total - p0)), starts))


def normal(key: int, count: int) -> np.ndarray:
    """count standard normals (binary64) from stream `key`.

    Pair i uses one splitmix64 output: u1 = (high 32 bits + 1) / 2^32 in (0, 1], u2 = low 32 bits / 2^32;
    Box-Muller gives element 2i = r cos(2 pi u2) and element 2i+1 = r sin(2 pi u2), r = sqrt(-2 ln u1).
    """
    out = np.empty(count + 1, dtype=np.float64)
    npairs = (count + 1) // 2

    def fill(p0, m):
        bits = _bits(key, p0, m)
        u1 = ((bits >> np.uint64(32)).astype(np.float64) + 1.0) * (1.0 / 4294967296.0)
        u2 = (bits & np.uint64(0xFFFFFFFF)).astype(np.float64) * (2.0 * np.pi / 4294967296.0)
        r = np.sqrt(-2.0 * np.log(u1))
        out[2 * p0:2 * (p0 + m):2] = r * np.cos(u2)
        out[2 * p0 + 1:2 * (p0 + m):2] = r * np.sin(u2)

    _chunked(npairs, fill)
    return out[:count]


def student_t(key: int, count: int, nu: int = 3) -> np.ndarray:
    z = normal(key, count)
    chi2 = np.zeros(count)
    for i in range(nu):
        c = normal(stream_key(key, "chi", i), count)
        np.multiply(c, c, out=c)
        chi2 += c
    np.divide(chi2, nu, out=chi2)
    np.sqrt(chi2, out=chi2)
    np.divide(z, chi2, out=z)
    return z


def weights(n: int, k: int, *key_parts, dist: str = "normal", std: float = 0.02) -> np.ndarray:
    """fp16 W[n][k] ~ std * N(0,1) (dist="normal") or std * StudentT(3) (dist="t3")."""
    key = stream_key("W", *key_parts)
    if dist == "normal":
        v = normal(key, n * k)
    elif dist == "t3":
        v = student_t(key, n * k, 3)
    else:
        raise ValueError(dist)
    v *= std
    return v.astype(np.float16).reshape(n, k)


def activations(batch: int, k: int, *key_parts) -> np.ndarray:
    """fp16 x[batch][k] ~ N(0, 1), rows independent."""
    key = stream_key("x", *key_parts)
    return normal(key, batch * k).astype(np.float16).reshape(batch, k)


def integer_exact_case(n: int, k: int, g: int, batch: int, *key_parts, kept: int = 2):
    """A 2:4-sparse (kept=2) or 1:4-sparse (kept=1) W whose quantisation is exact and an integer x, so
    every product and partial sum is an exactly representable small integer.

    Every group of every row holds, at kept positions, integers in [-8, 7] including both -8 and 7, so
    the group range is 15 and the scale is exactly 1 with zero point 8; the kept positions of each
    4-block carry distinct non-zero magnitudes larger than the dropped ones (which are 0). x holds
    integers in [-2, 2]. Returns (W fp16 [n][k], x fp16 [batch][k]).
    """
    key = stream_key("exact", *key_parts)
    u = uniform53(key, n * k * 3).reshape(3, n, k)
    w = np.zeros((n, k), dtype=np.float64)
    pairs = [(0, 1), (0, 2), (0, 3), (1, 2), (1, 3), (2, 3)]
    for r in range(n):
        for t in range(k // 4):
            p0, p1 = pairs[int(u[0, r, 4 * t] * 6) % 6]
            a = int(u[1, r, 4 * t] * 7) + 1      # 1..7
            b = int(u[2, r, 4 * t] * 7) + 1
            if a == b:
                b = b % 7 + 1
            sa = -1 if u[0, r, 4 * t + 1] < 0.5 else 1
            sb = -1 if u[0, r, 4 * t + 2] < 0.5 else 1
            w[r, 4 * t + p0] = sa * a
            if kept == 2:
                w[r, 4 * t + p1] = sb * b
        for G in range(k // g):
            # force the group range to exactly [-8, 7]: first block gets -8, second block gets 7
            t0 = G * g // 4
            if kept == 2:
                w[r, 4 * t0:4 * t0 + 4] = [-8, 7, 0, 0]
                w[r, 4 * t0 + 4:4 * t0 + 8] = [0, 0, 7, -8]
            else:
                w[r, 4 * t0:4 * t0 + 4] = [-8, 0, 0, 0]
                w[r, 4 * t0 + 4:4 * t0 + 8] = [0, 0, 7, 0]
    xu = uniform53(stream_key(key, "x"), batch * k)
    x = (np.floor(xu * 5) - 2).reshape(batch, k)
    return w.astype(np.float16), x.astype(np.float16)


# 7B-class decoder block: (role, N, K) of its seven linear layers.
DECODER_LINEARS = (("q", 4096, 4096), ("k", 4096, 4096), ("v", 4096, 4096), ("o", 4096, 4096),
                   ("gate", 11008, 4096), ("up", 11008, 4096), ("down", 4096, 11008))


def stack_table(n_blocks: int = 32, seed: int = 0, scale: int = 1, formats=(1, 2)):
    """Layer-adaptive stack: for every linear of every block a seeded choice of format among `formats`
    (equal probability; default 1 = 2:4 sparse INT4 and 2 = dense INT4; 3 = 1:4 sparse INT4 for the
    mixed-density stack) and of group size (64, 128 or 256, 1/3 each).

    Returns [(name, N, K, format, group)]. scale > 1 shrinks N and K (rounded up to multiples of 256)
    for quick tests.
    """
    u = uniform53(stream_key("stack-policy", seed), n_blocks * len(DECODER_LINEARS) * 2)
    out = []
    for blk in range(n_blocks):
        for j, (role, n, k) in enumerate(DECODER_LINEARS):
            i = blk * len(DECODER_LINEARS) + j
            fmt = formats[min(len(formats) - 1, int(u[2 * i] * len(formats)))]
            g = (64, 128, 256)[min(2, int(u[2 * i + 1] * 3))]
            if scale > 1:
                n = -(-(n // scale) // 256) * 256
                k = -(-(k // scale) // 256) * 256
            out.append((f"block{blk}.{role}", n, k, fmt, g))
    return out


def trie(branching, vocab: int, *key_parts):
    """A synthetic prefix tree of token ids in CSR form, built level by level the way hierarchical
    clustering builds one (broad at the top, narrower below): every node at depth d has branching[d]
    children with distinct token ids drawn from [0, vocab), stored in ascending token order; all leaves
    sit at depth len(branching). Node 0 is the root; nodes are numbered level by level.

    Returns (child_ptr int32 [n_nodes+1], child_tok int32 [n_edges], child_node int32 [n_edges]).
    """
    key = stream_key("trie", *key_parts)
    level = [0]
    next_id = 1
    children = {}
    draw = 0
    for d, b in enumerate(branching):
        nxt = []
        for u in level:
            # b distinct tokens: sample b * 4 candidates, keep the first b distinct ones
            cand = (uniform53(stream_key(key, "tok", draw), 4 * b + 16) * vocab).astype(np.int64)
            draw += 1
            toks = []
            seen = set()
            for t in cand:
                if int(t) not in seen:
                    seen.add(int(t))
                    toks.append(int(t))
                if len(toks) == b:
                    break
            assert len(toks) == b
            toks.sort()
            kids = list(range(next_id, next_id + b))
            next_id += b
            children[u] = list(zip(toks, kids))
            nxt.extend(kids)
        level = nxt
    n_nodes = next_id
    ptr = np.zeros(n_nodes + 1, dtype=np.int32)
    tok, node = [], []
    for u in range(n_nodes):
        kids = children.get(u, [])
        ptr[u + 1] = ptr[u] + len(kids)
        for t, v in kids:
            tok.append(t)
            node.append(v)
    return ptr, np.array(tok, dtype=np.int32), np.array(node, dtype=np.int32)


def log_probs(rows: int, vocab: int, *key_parts, spread: float = 2.0):
    """Decoder output rows as log-probabilities: logits ~ N(0, spread^2), log-softmax in fp64, fp32."""
    z = normal(stream_key("logp", *key_parts), rows * vocab).reshape(rows, vocab) * spread
    z = z - z.max(axis=1, keepdims=True)
    lp = z - np.log(np.exp(z).sum(axis=1, keepdims=True))
    return lp.astype(np.float32)
