"""GPU parity of eagle3_accept_lazy: acceptance with a lazy target LM head (logits only for the
nodes the walk visits, level by level; "Speculative Decoding (EAGLE3) in the vLLM Neuron
Framework", section "Rejection Sampling", with the walk of eagle3_accept).

The oracle replays each sequence with the logits rows the GPU computed for the nodes it visited
(every other row is NaN, so a walk that strays from the GPU's path fails) and must reproduce the
path, the emitted tokens and the next root bit for bit; the lazily computed rows themselves are
checked against the fp64 product of the same bf16 operands.  Planted trees (children whose tokens
are the parent's greedy prediction, with sharpened logits for TOPK) make the walks several levels
deep.
"""
import numpy as np
import pytest
import torch

import synth
from oracle import accept as oacc
from oracle import tree as otree
from tests._util import close, require_gpu

pytestmark = pytest.mark.gpu


def _setup(seed, B, N, d, V, scale):
    r = np.random.default_rng(seed)
    hs_t, hs = synth.to_bf16(scale * r.standard_normal((B, N, d), dtype=np.float32))
    lm_t, lm = synth.to_bf16(0.02 * r.standard_normal((V, d), dtype=np.float32))
    parents = np.stack([synth.random_tree(r, N) for _ in range(B)]).astype(np.int32)
    tokens = r.integers(0, V, (B, N)).astype(np.int32)
    return hs_t, hs, lm_t, lm, parents, tokens


def _plant(hs, lm, parents, tokens):
    """Children along the path to each tree's deepest node carry the parent's greedy token
    (argmax of the fp64 logits of the parent's hidden state)."""
    for b in range(parents.shape[0]):
        dep = otree.depths(parents[b].tolist())
        path = otree.path_to(parents[b], int(np.argmax(dep)))
        for u, c in zip(path[:-1], path[1:]):
            tokens[b, c] = int(np.argmax(lm.astype(np.float64) @ hs[b, u].astype(np.float64)))


def _run(mode, hs_t, lm_t, parents, tokens, W, T=1.0, seed=3, step=0):
    from eagle_tree_speculative_spec_gb300 import eagle3_accept_lazy
    dev = require_gpu()
    B, N, _ = hs_t.shape
    V = lm_t.shape[0]
    i32 = dict(dtype=torch.int32, device=dev)
    out = dict(alen=torch.full((B,), -7, **i32), path=torch.full((B, W), -7, **i32),
               emitted=torch.full((B, W), -7, **i32), root=torch.full((B,), -7, **i32),
               st=torch.zeros(1, **i32))
    dbg = torch.full((W, B, V), float("nan"), dtype=torch.float32, device=dev)
    eagle3_accept_lazy(mode, hs_t.to(dev), lm_t.to(dev), torch.as_tensor(tokens, **i32),
                       torch.as_tensor(parents, **i32), out["alen"], out["path"], out["emitted"], out["root"],
                       temperature=T, seed=seed, step=step, dev_status=out["st"], dbg_level_logits=dbg)
    torch.cuda.synchronize()
    res = {k: v.cpu().numpy() for k, v in out.items()}
    res["dbg"] = dbg.cpu().numpy()
    return res


def _check(mode, g, hs, lm, parents, tokens, W, T=1.0, seed=3, step=0, rows_checked=4):
    B, N, d = hs.shape
    V = lm.shape[0]
    assert g["st"][0] == 0
    checked = 0
    for b in range(B):
        n = int(g["alen"][b])
        path = [int(x) for x in g["path"][b, : n + 1]]
        z = np.full((N, V), np.nan, dtype=np.float32)
        for lvl, node in enumerate(path):
            z[node] = g["dbg"][lvl, b]
            if checked < rows_checked:      # the lazily computed row against the fp64 product
                ok, err = close(z[node], lm.astype(np.float64) @ hs[b, node].astype(np.float64), 1e-3, 1e-3)
                assert ok, (b, node, err)
                checked += 1
        res = oacc.accept(mode, tokens[b], parents[b], z, temperature=T, seed=seed, step=step, b=b)
        want_path, want_emit = oacc.pad(res, W)
        assert res["accept_len"] == n, (b, res, n)
        assert (g["path"][b] == want_path).all(), b
        assert (g["emitted"][b] == want_emit).all(), b
        assert g["root"][b] == res["next_root"], b


@pytest.mark.parametrize("mode_name,scale", [("greedy", 1.0), ("topk", 40.0)])
def test_lazy_accept_planted_walks(mode_name, scale):
    from eagle_tree_speculative_spec_gb300 import GREEDY, TOPK
    mode = {"greedy": GREEDY, "topk": TOPK}[mode_name]
    B, N, d, V, W = 6, 16, 256, 1000, 7
    hs_t, hs, lm_t, lm, parents, tokens = _setup(11, B, N, d, V, scale)
    _plant(hs, lm, parents, tokens)
    g = _run(mode, hs_t, lm_t, parents, tokens, W)
    _check(mode, g, hs, lm, parents, tokens, W, rows_checked=40)
    assert (g["alen"] >= 2).sum() >= B // 2                # the planted paths are walked several levels


@pytest.mark.parametrize("mode_name", ["greedy", "topk"])
def test_lazy_accept_full_vocabulary(mode_name):
    """Llama-3.1-8B head shapes: B = 64, 60-node trees, d = 4096, V = 128256."""
    from eagle_tree_speculative_spec_gb300 import GREEDY, TOPK
    mode = {"greedy": GREEDY, "topk": TOPK}[mode_name]
    B, N, d, V, W = 64, 60, 4096, 128256, 7
    hs_t, hs, lm_t, lm, parents, tokens = _setup(12, B, N, d, V, 1.0)
    # plant greedy children for a quarter of the sequences (the rest stop at the root)
    sub = slice(0, 16)
    t16 = tokens[sub].copy()
    _plant(hs[sub], lm, parents[sub], t16)
    tokens[sub] = t16
    g = _run(mode, hs_t, lm_t, parents, tokens, W, step=5)
    _check(mode, g, hs, lm, parents, tokens, W, step=5)


def test_lazy_accept_equals_full_head_acceptance():
    """The same decisions as eagle3_accept on the full head's logits (the products of both paths
    agree to fp32 rounding; with these inputs no decision sits on a tie)."""
    from eagle_tree_speculative_spec_gb300 import EPI_F32, GREEDY, eagle3_accept, eagle3_linear
    dev = require_gpu()
    B, N, d, V, W = 8, 12, 512, 3000, 7
    hs_t, hs, lm_t, lm, parents, tokens = _setup(13, B, N, d, V, 1.0)
    _plant(hs, lm, parents, tokens)
    g = _run(GREEDY, hs_t, lm_t, parents, tokens, W)
    logits = torch.empty(B * N, V, dtype=torch.float32, device=dev)
    eagle3_linear(hs_t.to(dev).view(B * N, d), lm_t.to(dev), logits, epilogue=EPI_F32)
    i32 = dict(dtype=torch.int32, device=dev)
    alen, path = torch.empty(B, **i32), torch.empty(B, W, **i32)
    emitted, root = torch.empty(B, W, **i32), torch.empty(B, **i32)
    eagle3_accept(GREEDY, logits.view(B, N, V), torch.as_tensor(tokens, **i32), torch.as_tensor(parents, **i32),
                  alen, path, emitted, root)
    torch.cuda.synchronize()
    assert (alen.cpu().numpy() == g["alen"]).all()
    assert (path.cpu().numpy() == g["path"]).all()
    assert (root.cpu().numpy() == g["root"]).all()
