"""Dynamic top-k draft tree (expand, frontier select, final rerank).

Sources: "EAGLE-3: Engineering Implementation of LLM Inference Acceleration",
sections IV.3 and XI.6 (EAGLE-2's dynamic tree: acceptance is estimated from
draft confidence, the tree is expanded and pruned at the end of drafting; the
official engine defaults to 60 nodes, depth 7 and top-k 10),
"EAGLE-3: Training-Time Test for Speculative Decoding", section "Dynamic Draft
Trees Spend Verification Where It Can Pay Off", and "Advanced speculative
decoding: tree drafts and EAGLE" (``build_draft_tree``: each node's children
are the draft's top-k tokens; node 0 is the root).

The pages give the selection rule only in prose, so this is the plainest
reading of "expand to depth D with top-k per node, rerank by cumulative
log-probability down to N nodes":
* depth 1: the root row's top-k tokens; score = logq (the DSM log-normaliser
  at T = 1, :mod:`oracle.dsm`); ties in top-k go to the lower token id.
* depth t = 2..D: the frontier is the k best depth-(t-1) candidates by
  (score desc, creation index asc); each frontier node runs one draft row and
  contributes its top-k children with score = fp32(parent score + logq);
  creation index = frontier rank * k + child rank.
* final: the N-1 best of all candidates by (score desc, depth asc, creation
  asc) - ancestor-closed because logq <= 0 and ties favour the shallower
  node - emitted after the root in (depth asc, score desc, creation asc)
  order, so parents precede children and siblings are in score order.

Draft rows (positions per "EAGLE-3: Engineering Implementation of LLM
Inference Acceleration", section XI.2): the root's row is the last catch-up
row at position L-1; a frontier node at depth t-1 runs the row
(x = a of its parent's row, e = its token) at position L-1+(t-1), attending
to the draft cache, to its tree ancestors' rows and to itself.

Reduced draft vocabulary ("EAGLE-3: Engineering Implementation of LLM
Inference Acceleration", sections VIII.5-VIII.6): the draft's LM head covers a
sorted subset of target tokens and ``d2t[i]`` is the target id of draft id i.
Top-k and logq then run over the draft logits (ties to the lower draft id) and
a candidate's token is the mapped target id; this equals expanding over the
target vocabulary with -inf outside the subset (pinned in the tests).

parity unpinned beyond invariants: the EAGLE-2 source is not on the pages.
The invariants tested are the node count, depth bound, ancestor closure,
frontier = top-k at each depth, every candidate's score recomputed as the fp32
running sum of the log-softmax of its ancestors' expansion rows at their
tokens, final set = top N-1 over all candidates by brute-force sort, that
top_k = 1 gives the chain drafting of section XI.2, and that at depth 2 with a
budget keeping every candidate (N = 1 + k + k^2) the tree is the fixed-branching
expansion [k, k] of "Advanced speculative decoding: tree drafts and EAGLE"
(``build_draft_tree``) for a path-dependent draft.
"""
import numpy as np

from . import dsm
from .accept import order_key
from .tree import anc_bits


def topk_tokens(row, k):
    """k largest entries of an fp32 row, ties to the lower index."""
    key = order_key(row)
    idx = np.lexsort((np.arange(len(row)), -key))
    return [int(i) for i in idx[:k]]


def select_tree(expand, depth, top_k, n_nodes, cands=None, d2t=None):
    """Run the dynamic tree selection.

    expand(t, frontier) returns fp32 logits [len(frontier), V]; for t = 1 the
    frontier is [None] (the root row), otherwise a list of candidate ids at
    depth t-1 in frontier-rank order; with ``d2t`` the logits are over the
    draft vocabulary and tokens are mapped to target ids.  ``cands`` (a list the caller may read
    from inside expand) receives the candidate table: dicts with token, score,
    depth, creation, parent (candidate id, -1 for the root).  Returns tokens,
    parents, depth, score per emitted node (node 0 = root, token -1 here), the
    candidate table, the frontier of every depth and the chosen candidates."""
    cands = [] if cands is None else cands
    frontiers = []
    front = [None]
    for t in range(1, depth + 1):
        logits = np.asarray(expand(t, front), dtype=np.float32)
        for r, f in enumerate(front):
            lq = dsm.logq(logits[r])
            for c, tok in enumerate(topk_tokens(logits[r], top_k)):
                score = lq[tok] if f is None else np.float32(cands[f]["score"] + lq[tok])
                tgt = tok if d2t is None else int(d2t[tok])
                cands.append({"token": tgt, "score": np.float32(score), "depth": t,
                              "creation": r * top_k + c, "parent": -1 if f is None else f})
        frontiers.append(front)
        if t < depth:
            at_t = [i for i, c in enumerate(cands) if c["depth"] == t]
            at_t.sort(key=lambda i: (-float(cands[i]["score"]), cands[i]["creation"]))
            front = at_t[:top_k]
    order = sorted(range(len(cands)),
                   key=lambda i: (-float(cands[i]["score"]), cands[i]["depth"], cands[i]["creation"]))
    chosen = order[: n_nodes - 1]
    chosen.sort(key=lambda i: (cands[i]["depth"], -float(cands[i]["score"]), cands[i]["creation"]))
    node_of = {cid: n + 1 for n, cid in enumerate(chosen)}
    tokens, parents, depths_, scores = [-1], [-1], [0], [np.float32(0.0)]
    for cid in chosen:
        c = cands[cid]
        par = 0 if c["parent"] == -1 else node_of[c["parent"]]      # KeyError = not ancestor-closed
        tokens.append(c["token"])
        parents.append(par)
        depths_.append(c["depth"])
        scores.append(c["score"])
    return {"tokens": np.asarray(tokens, np.int64), "parents": np.asarray(parents, np.int64),
            "depth": np.asarray(depths_, np.int64), "score": np.asarray(scores, np.float32),
            "cands": cands, "frontiers": frontiers, "chosen": chosen,
            "anc": anc_bits(parents)}


def draft_tree_for_sequence(draft, d_cache, a_root, root_token, L, depth, top_k, n_nodes,
                            logits_log=None, select_logits=None, d2t=None):
    """Build the tree for one sequence with the oracle draft model.

    d_cache holds draft K/V for positions 0..L-1; a_root is the last catch-up
    row's output.  ``logits_log`` (a list) receives each depth's fp32 logits.
    ``select_logits(t, frontier)``, when given, supplies the logits the selection
    uses (replay of another implementation's logits); the oracle still runs and
    logs its own rows for that tree, so the two can be compared row by row."""
    cands, rows_a, rows_k, rows_v, row_of = [], [], [], [], {}

    def expand(t, front):
        if t == 1:
            out = draft.logits(np.asarray(a_root, dtype=np.float64)[None])
        else:
            toks, xs, vis = [], [], []
            for f in front:
                c = cands[f]
                toks.append(c["token"])
                xs.append(a_root if c["parent"] == -1 else rows_a[row_of[c["parent"]]])
                anc, j = [], c["parent"]
                while j != -1:
                    anc.append(row_of[j])
                    j = cands[j]["parent"]
                # indexes into [pool rows; new rows]: ancestors' rows, then this row
                vis.append(anc[::-1] + [len(rows_a) + len(vis)])
            pool_k = np.stack(rows_k, 0) if rows_k else None
            pool_v = np.stack(rows_v, 0) if rows_v else None
            a, k, v = draft.layer(toks, np.stack(xs, 0), np.full(len(toks), L - 1 + (t - 1)),
                                  d_cache, vis, pool_k, pool_v)
            for r, f in enumerate(front):
                row_of[f] = len(rows_a)
                rows_a.append(a[r])
                rows_k.append(k[r])
                rows_v.append(v[r])
            out = draft.logits(a)
        out = out.astype(np.float32)
        if logits_log is not None:
            logits_log.append(out)
        return out if select_logits is None else np.asarray(select_logits(t, front), dtype=np.float32)

    res = select_tree(expand, depth, top_k, n_nodes, cands, d2t)
    res["tokens"][0] = root_token
    return res
