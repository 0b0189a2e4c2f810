"""GPU parity of the trie-constrained beam-score step (sgemv_beam_step / sgemv_beam_traceback) against
the CPU oracle (oracle/beam.py). Source: the paper "Efficient LLM-based Advertising via Model
Compression and Parallel Verification", §3.4 "Tree-Based Parallel Verification".

The bar is bit-exact: every kept node, token, parent and score must equal the oracle's (scores are
single binary32 additions, and the ranking and its ties are fixed), step after step, and the traced-back
sequences must be identical.
"""

import numpy as np
import pytest

import synth
from oracle import beam as obeam

pytestmark = pytest.mark.gpu


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


def _out(torch, k):
    return (torch.empty(k, dtype=torch.int32, device="cuda"), torch.empty(k, dtype=torch.float32, device="cuda"),
            torch.empty(k, dtype=torch.int32, device="cuda"), torch.empty(k, dtype=torch.int32, device="cuda"),
            torch.empty(1, dtype=torch.int32, device="cuda"))


def _gpu_step(env, trie, node, score, logp, k, status):
    sg, torch = env
    out = _out(torch, k)
    sg.sgemv_beam_step(trie, torch.from_numpy(np.asarray(node, dtype=np.int32)).cuda(),
                       torch.from_numpy(np.asarray(score, dtype=np.float32)).cuda(),
                       torch.from_numpy(np.ascontiguousarray(logp, dtype=np.float32)).cuda(), k, out, status=status)
    torch.cuda.synchronize()
    cnt = int(out[4].item())
    return {"node": out[0][:cnt].cpu().numpy(), "score": out[1][:cnt].cpu().numpy(),
            "parent": out[2][:cnt].cpu().numpy(), "tok": out[3][:cnt].cpu().numpy(), "count": cnt}, out


def _same(g, o):
    assert g["count"] == o["count"]
    for key in ("node", "parent", "tok"):
        assert np.array_equal(g[key], o[key]), key
    assert np.array_equal(g["score"].view(np.uint32), o["score"].astype(np.float32).view(np.uint32))


@pytest.mark.parametrize("branching,vocab,k", [([64, 16, 8, 4], 32000, 20), ([300, 20, 5], 50000, 8),
                                                ([4, 4, 4, 4, 4], 1000, 64), ([2, 3], 16, 1)])
def test_decode_matches_oracle(env, branching, vocab, k):
    sg, torch = env
    ptr, tok, nod = synth.trie(branching, vocab, "gpu-beam", *branching)
    trie, keep = sg.make_trie(ptr, tok, nod)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    nodes, scores = np.array([0], dtype=np.int32), np.array([0.0], dtype=np.float32)
    parents_dev, toks_dev, parents, toks = [], [], [], []
    for step in range(len(branching)):
        logp = synth.log_probs(len(nodes), vocab, "gpu-beam", step, *branching)
        o = obeam.beam_step(ptr, tok, nod, nodes, scores, logp, k)
        g, out = _gpu_step(env, trie, nodes, scores, logp, k, status)
        _same(g, o)
        assert int(status.item()) == 0
        pad = np.full(k, -1, dtype=np.int32)
        pd, td = pad.copy(), pad.copy()
        pd[:g["count"]], td[:g["count"]] = g["parent"], g["tok"]
        parents_dev.append(pd)
        toks_dev.append(td)
        parents.append(o["parent"])
        toks.append(o["tok"])
        nodes, scores = o["node"], o["score"].astype(np.float32)
        last_count = out[4]
    seq = torch.empty((k, len(branching)), dtype=torch.int32, device="cuda")
    sg.sgemv_beam_traceback(torch.from_numpy(np.stack(parents_dev)).cuda(), torch.from_numpy(np.stack(toks_dev)).cuda(),
                            last_count, seq, status=status)
    torch.cuda.synchronize()
    want = obeam.traceback(parents, toks, len(nodes))
    got = seq.cpu().numpy()
    assert np.array_equal(got[:len(nodes)], want)
    assert np.all(got[len(nodes):] == -1)
    assert int(status.item()) == 0


def test_ties_nan_and_minus_inf(env):
    sg, torch = env
    vocab = 512
    ptr, tok, nod = synth.trie([32, 16], vocab, "gpu-ties")
    trie, keep = sg.make_trie(ptr, tok, nod)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    nodes = np.arange(1, 33, dtype=np.int32)
    scores = np.repeat(np.array([-1.0, -0.5], dtype=np.float32), 16)
    logp = np.round(synth.log_probs(32, vocab, "gpu-ties") * 2) / 2      # many equal scores
    logp = logp.astype(np.float32)
    logp[3, tok[ptr[nodes[3]]]] = np.nan
    logp[5, tok[ptr[nodes[5]] + 1]] = -np.inf
    logp[7, tok[ptr[nodes[7]]]] = -0.0
    for k in (1, 17, 64):
        status.zero_()
        o = obeam.beam_step(ptr, tok, nod, nodes, scores, logp, k)
        g, _ = _gpu_step(env, trie, nodes, scores, logp, k, status)
        _same(g, o)
        assert int(status.item()) == sg.SGEMV_ERR_NONFINITE     # the NaN was dropped and reported


@pytest.mark.parametrize("beam_in,children", [(64, 40), (33, 250), (3, 5)])
def test_wide_steps_match_oracle(env, beam_in, children):
    """Candidate counts on both sides of the 1024-key register sort (2560, 8250 and 15 keys)."""
    sg, torch = env
    vocab = 40000
    ptr, tok, nod = synth.trie([64, children], vocab, "gpu-wide", beam_in, children)
    trie, keep = sg.make_trie(ptr, tok, nod)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    nodes = np.arange(1, 1 + beam_in, dtype=np.int32)
    scores = (-np.arange(beam_in) * 0.125).astype(np.float32)
    logp = synth.log_probs(beam_in, vocab, "gpu-wide", beam_in, children)
    for k in (1, 20, 64):
        o = obeam.beam_step(ptr, tok, nod, nodes, scores, logp, k)
        g, _ = _gpu_step(env, trie, nodes, scores, logp, k, status)
        _same(g, o)
    assert int(status.item()) == 0


def test_everything_kept_ends_with_minus_inf(env):
    sg, torch = env
    vocab = 64
    ptr, tok, nod = synth.trie([8, 4], vocab, "gpu-all")
    trie, keep = sg.make_trie(ptr, tok, nod)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    nodes = np.arange(1, 9, dtype=np.int32)
    scores = np.zeros(8, dtype=np.float32)
    logp = synth.log_probs(8, vocab, "gpu-all")
    logp[2, tok[ptr[nodes[2]]]] = -np.inf
    o = obeam.beam_step(ptr, tok, nod, nodes, scores, logp, 64)
    g, _ = _gpu_step(env, trie, nodes, scores, logp, 64, status)
    _same(g, o)
    assert g["count"] == 32 and g["score"][-1] == -np.inf


def test_bad_node_and_too_many_candidates_reported(env):
    sg, torch = env
    vocab = 20000
    ptr, tok, nod = synth.trie([64, 300], vocab, "gpu-big")
    trie, keep = sg.make_trie(ptr, tok, nod)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    # 64 beams x 300 children = 19200 candidates > 16384: reported, nothing kept
    nodes = np.arange(1, 65, dtype=np.int32)
    logp = synth.log_probs(64, vocab, "gpu-big")
    g, _ = _gpu_step(env, trie, nodes, np.zeros(64, np.float32), logp, 8, status)
    assert g["count"] == 0 and int(status.item()) == sg.SGEMV_ERR_SHAPE
    # an out-of-range node id contributes nothing and is reported; the others are ranked as usual
    status.zero_()
    nodes2 = np.array([1, len(ptr) + 5, 2], dtype=np.int32)
    o = obeam.beam_step(ptr, tok, nod, [1, 2], [0.0, 0.0], logp[[0, 2]], 10)
    g, _ = _gpu_step(env, trie, nodes2, np.zeros(3, np.float32), logp[:3], 10, status)
    assert int(status.item()) == sg.SGEMV_ERR_ARG
    o["parent"] = np.where(o["parent"] == 1, 2, o["parent"])          # input beam 1 of the oracle is beam 2 here
    _same(g, o)


def test_argument_errors(env):
    sg, torch = env
    ptr, tok, nod = synth.trie([4], 16, "gpu-args")
    trie, keep = sg.make_trie(ptr, tok, nod)
    node = torch.zeros(1, dtype=torch.int32, device="cuda")
    score = torch.zeros(1, dtype=torch.float32, device="cuda")
    logp = torch.zeros((1, 16), dtype=torch.float32, device="cuda")
    with pytest.raises(sg.SgemvError) as e:
        sg.sgemv_beam_step(trie, node, score, logp, 0, _out(torch, 1))
    assert e.value.code == sg.SGEMV_ERR_ARG
    with pytest.raises(sg.SgemvError) as e:
        sg.sgemv_beam_step(trie, node, score, logp, 65, _out(torch, 65))
    assert e.value.code == sg.SGEMV_ERR_ARG


def _oracle_decode(ptr, tok, nod, logps, k, shared):
    """The oracle's steps one after the other; step t reads row b of logps[t] (row 0 when shared)."""
    nodes, scores = np.array([0], dtype=np.int32), np.array([0.0], dtype=np.float32)
    steps, parents, toks = [], [], []
    for lp in logps:
        rows = np.broadcast_to(lp[0], (len(nodes), lp.shape[1])) if shared else lp[:len(nodes)]
        o = obeam.beam_step(ptr, tok, nod, nodes, scores, rows, k)
        steps.append(o)
        parents.append(o["parent"])
        toks.append(o["tok"])
        nodes, scores = o["node"], o["score"].astype(np.float32)
    return steps, obeam.traceback(parents, toks, steps[-1]["count"])


@pytest.mark.parametrize("branching,vocab,k,shared,extra", [
    ([64, 16, 8, 4], 32000, 20, False, 0), ([64, 16, 8, 4], 32000, 20, True, 0),
    ([4, 4, 4, 4, 4], 1000, 64, False, 0), ([2, 3], 16, 1, True, 0),
    ([8, 4], 500, 16, False, 2),  # two steps past the leaves: no candidates, empty beams from there on
])
def test_fused_decode_matches_oracle(env, branching, vocab, k, shared, extra):
    """sgemv_beam_decode (all steps and the traceback in one launch) equals the oracle's steps one by one,
    bit for bit, with per-beam rows or one shared row per position."""
    sg, torch = env
    ptr, tok, nod = synth.trie(branching, vocab, "fused", *branching)
    trie, keep = sg.make_trie(ptr, tok, nod)
    steps = len(branching) + extra
    logps = [synth.log_probs(1 if (shared or t == 0) else k, vocab, "fused", t, *branching) for t in range(steps)]
    want, want_seq = _oracle_decode(ptr, tok, nod, logps, k, shared)
    dev = lambda a, dt: torch.from_numpy(np.ascontiguousarray(a, dtype=dt)).cuda()
    out = (torch.full((steps, k), -7, dtype=torch.int32, device="cuda"),
           torch.zeros((steps, k), dtype=torch.float32, device="cuda"),
           torch.full((steps, k), -7, dtype=torch.int32, device="cuda"),
           torch.full((steps, k), -7, dtype=torch.int32, device="cuda"),
           torch.full((steps,), -7, dtype=torch.int32, device="cuda"))
    seq = torch.full((k, steps), -7, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    sg.sgemv_beam_decode(trie, dev([0], np.int32), dev([0.0], np.float32), [dev(lp, np.float32) for lp in logps], k,
                         out, seq, shared_row=shared, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    counts = out[4].cpu().numpy()
    for t, o in enumerate(want):
        c = int(counts[t])
        g = {"count": c, "node": out[0][t, :c].cpu().numpy(), "score": out[1][t, :c].cpu().numpy(),
             "parent": out[2][t, :c].cpu().numpy(), "tok": out[3][t, :c].cpu().numpy()}
        _same(g, o)
    final = int(counts[-1])
    s = seq.cpu().numpy()
    assert np.array_equal(s[:final], want_seq)
    assert np.all(s[final:] == -1)
    if extra:
        assert final == 0
