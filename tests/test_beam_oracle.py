"""Pins for the beam-step oracle (oracle/beam.py), each against something other than the oracle.

Source: the paper "Efficient LLM-based Advertising via Model Compression and Parallel Verification",
§3.4 "Tree-Based Parallel Verification". Pins:
  * a hand-worked two-step example with ties (golden file);
  * exhaustive enumeration: when every step keeps every candidate, beam search over a small trie must
    return every root-to-leaf path, with its score summed along the path by plain iteration, best first;
  * the first step equals a direct sort of the root's children by log-probability;
  * invariants on random tries: outputs are children of their parents' nodes, scores are non-increasing,
    count = min(K, candidates), NaN scores are dropped and counted, -inf scores rank last.
"""

import os

import numpy as np
import pytest

import synth
from oracle import beam

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _fixture():
    fx = {}
    with open(os.path.join(GOLDEN, "beam_step_worked_example.txt")) as f:
        for ln in f:
            if ln.startswith("#") or not ln.strip():
                continue
            key, *rest = ln.split()
            fx[key] = rest
    return fx


def test_worked_example():
    fx = _fixture()
    ptr = np.array(fx["trie_ptr"], dtype=np.int32)
    tok = np.array(fx["trie_tok"], dtype=np.int32)
    nod = np.array(fx["trie_node"], dtype=np.int32)
    V = 8
    lp1 = np.full((1, V), -10.0, dtype=np.float32)
    lp1[0, 2], lp1[0, 5], lp1[0, 7] = -1.0, -0.5, -0.5
    r1 = beam.beam_step(ptr, tok, nod, [0], [0.0], lp1, 2)
    assert list(r1["node"]) == [int(v) for v in fx["step1_node"]]
    assert list(r1["score"]) == [float(v) for v in fx["step1_score"]]
    assert list(r1["parent"]) == [int(v) for v in fx["step1_parent"]]
    assert list(r1["tok"]) == [int(v) for v in fx["step1_tok"]]
    lp2 = np.full((2, V), -10.0, dtype=np.float32)
    lp2[0, 1], lp2[0, 3], lp2[1, 1] = -0.25, -2.0, -0.25
    r2 = beam.beam_step(ptr, tok, nod, r1["node"], r1["score"], lp2, 2)
    assert list(r2["node"]) == [int(v) for v in fx["step2_node"]]
    assert list(r2["score"]) == [float(v) for v in fx["step2_score"]]
    assert list(r2["parent"]) == [int(v) for v in fx["step2_parent"]]
    assert list(r2["tok"]) == [int(v) for v in fx["step2_tok"]]
    seqs = beam.traceback([r1["parent"], r2["parent"]], [r1["tok"], r2["tok"]], r2["count"])
    assert seqs.tolist() == [[int(v) for v in fx["seq0"]], [int(v) for v in fx["seq1"]]]


def _logp_for_node(u, vocab):
    # the decoder's output for a prefix is a function of the prefix (= the trie node), drawn per node
    return synth.log_probs(1, vocab, "beam-pin", int(u))[0]


@pytest.mark.parametrize("branching", [[3, 2, 2], [5, 1, 3], [2, 2, 2, 2]])
def test_exhaustive_paths_when_nothing_is_pruned(branching):
    vocab = 64
    ptr, tok, nod = synth.trie(branching, vocab, "exhaustive", *branching)
    n_leaves = int(np.prod(branching))
    # brute force: every root-to-leaf path and its score, summed step by step in binary32
    paths = []

    def walk(u, seq, s):
        if ptr[u] == ptr[u + 1]:
            paths.append((tuple(seq), s))
            return
        lp = _logp_for_node(u, vocab)
        for e in range(ptr[u], ptr[u + 1]):
            walk(int(nod[e]), seq + [int(tok[e])], np.float32(s + lp[tok[e]]))

    walk(0, [], np.float32(0.0))
    assert len(paths) == n_leaves
    # beam search keeping everything
    nodes, scores = np.array([0]), np.array([0.0], dtype=np.float32)
    parents, toks = [], []
    for _ in branching:
        lp = np.stack([_logp_for_node(u, vocab) for u in nodes])
        r = beam.beam_step(ptr, tok, nod, nodes, scores, lp, k=10 ** 6)
        parents.append(r["parent"])
        toks.append(r["tok"])
        nodes, scores = r["node"], r["score"]
    seqs = beam.traceback(parents, toks, len(nodes))
    got = sorted((tuple(int(v) for v in sq), float(s)) for sq, s in zip(seqs, scores))
    want = sorted((sq, float(s)) for sq, s in paths)
    assert got == want
    assert np.all(np.diff(scores.astype(np.float64)) <= 0)          # best first


def test_first_step_is_a_sort_of_the_root_children():
    vocab = 1000
    ptr, tok, nod = synth.trie([200, 3], vocab, "root-sort")
    lp = synth.log_probs(1, vocab, "root-sort")
    r = beam.beam_step(ptr, tok, nod, [0], [0.0], lp, k=20)
    ch = [(float(lp[0, tok[e]]), int(tok[e]), int(nod[e])) for e in range(ptr[0], ptr[1])]
    ch.sort(key=lambda c: (-c[0], c[1]))
    assert [(float(s), int(t), int(n)) for s, t, n in zip(r["score"], r["tok"], r["node"])] == ch[:20]


@pytest.mark.parametrize("beam_in,k", [(1, 1), (4, 8), (20, 20), (32, 32)])
def test_invariants_random(beam_in, k):
    vocab = 5000
    ptr, tok, nod = synth.trie([40, 12, 6], vocab, "inv", beam_in, k)
    rng = np.random.default_rng(beam_in * 100 + k)
    level1 = np.arange(1, 41)
    nodes = rng.choice(level1, beam_in, replace=beam_in > 40)
    scores = (-rng.random(beam_in) * 5).astype(np.float32)
    lp = synth.log_probs(beam_in, vocab, "inv", beam_in, k)
    lp[0, tok[ptr[nodes[0]]]] = np.nan                               # one NaN candidate
    lp[-1, tok[ptr[nodes[-1] + 1] - 1]] = -np.inf                     # one impossible token
    r = beam.beam_step(ptr, tok, nod, nodes, scores, lp, k)
    n_cand = sum(int(ptr[u + 1] - ptr[u]) for u in nodes) - 1
    assert r["nan"] == 1 and r["count"] == min(k, n_cand)
    for i in range(r["count"]):
        b = r["parent"][i]
        u = nodes[b]
        edges = range(ptr[u], ptr[u + 1])
        e = [e for e in edges if tok[e] == r["tok"][i]]
        assert len(e) == 1 and nod[e[0]] == r["node"][i]
        assert r["score"][i] == np.float32(scores[b] + lp[b, r["tok"][i]])
    assert np.all(np.diff(r["score"].astype(np.float64)) <= 0)
    if r["count"] == n_cand:
        assert r["score"][-1] == -np.inf
