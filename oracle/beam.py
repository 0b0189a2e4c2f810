"""CPU oracle for the trie-constrained beam-score step -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may use this module;
the product never imports it and shares no code with it.

Source: the paper "Efficient LLM-based Advertising via Model Compression and Parallel Verification",
§3.4 "Tree-Based Parallel Verification": the decoder's per-position distribution T_score is filtered by
the prefix tree to the valid next tokens, each valid token's score is added to its parent node's score
in log space to give B_score, beam search keeps the best B_score nodes, and at the last position the
best nodes are traced back into sequences.

Readings (where the page leaves a step open):
  * T_score arrives as log-probabilities, so the "logarithmic summation" is one binary32 addition
    B = parent + T[token] (round to nearest even); the ranking therefore depends on nothing but IEEE
    additions and is reproducible on any device;
  * candidates are ranked by B descending, then by input beam ascending, then by token ascending (the
    children of a node are stored in ascending token order);
  * a NaN score is not a candidate (it is counted and reported); -inf (probability 0) is a candidate;
  * a beam whose node is a leaf contributes no candidate; if fewer than K candidates exist, fewer than
    K beams come out.
Every function works on one step at a time with numpy primitives (an fp32 add, a stable lexicographic
sort), so it can be checked against the page by eye. Pinned by tests/test_beam_oracle.py (exhaustive
path enumeration on small tries, a hand-worked example, invariants).
"""

from __future__ import annotations

import numpy as np


def beam_step(child_ptr, child_tok, child_node, node, score, logp, k: int):
    """One step. node/score: the input beams' trie nodes and scores (len beam_in); logp: fp32
    [beam_in][vocab]. Returns dict(node, score, parent, tok, count, nan) for the first
    count = min(k, candidates) candidates in rank order."""
    child_ptr = np.asarray(child_ptr, dtype=np.int64)
    node = np.asarray(node, dtype=np.int64)
    score = np.asarray(score, dtype=np.float32)
    logp = np.asarray(logp, dtype=np.float32)
    c_beam, c_edge = [], []
    for b in range(len(node)):
        for e in range(child_ptr[node[b]], child_ptr[node[b] + 1]):  # children, ascending token
            c_beam.append(b)
            c_edge.append(e)
    c_beam = np.array(c_beam, dtype=np.int64)
    c_edge = np.array(c_edge, dtype=np.int64)
    toks = np.asarray(child_tok, dtype=np.int64)[c_edge] if len(c_edge) else np.zeros(0, np.int64)
    s = (score[c_beam] + logp[c_beam, toks]).astype(np.float32)  # binary32 add
    nan = int(np.isnan(s).sum())
    keep = ~np.isnan(s)
    order = np.arange(len(s))[keep]
    # rank: B descending; ties by candidate index (input beam, then token) ascending
    order = order[np.lexsort((order, -s[keep].astype(np.float64)))]
    order = order[:k]
    return {
        "node": np.asarray(child_node, dtype=np.int32)[c_edge[order]] if len(order) else np.zeros(0, np.int32),
        "score": s[order],
        "parent": c_beam[order].astype(np.int32),
        "tok": toks[order].astype(np.int32),
        "count": int(len(order)),
        "nan": nan,
    }


def traceback(parents, toks, final_count: int):
    """Sequences of the final beams: parents[t][i] / toks[t][i] are the parent index (into step t-1's
    beams) and token of beam i after step t. Returns int32 [final_count][steps]."""
    steps = len(parents)
    out = np.zeros((final_count, steps), dtype=np.int32)
    for f in range(final_count):
        i = f
        for t in range(steps - 1, -1, -1):
            out[f, t] = toks[t][i]
            i = parents[t][i]
    return out
