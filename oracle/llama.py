"""Tiny Llama target, EAGLE-3 draft head, vanilla and speculative greedy decoding.

Sources:
* "EAGLE-3: Engineering Implementation of LLM Inference Acceleration":
  appendix C (RMSNorm, rotate-half RoPE, grouped-query attention), section
  VIII.1 (the draft decoder layer with two input streams: input_norm(e) and
  hidden_norm(x) concatenated to 2k, Q/K/V read the 2k vector, the residual
  stream is x only, SwiGLU MLP), sections VIII.4-VIII.5 (frozen copy of the
  target embedding; logits = lm_head(norm(a)), the recurrent state is the
  pre-norm a), sections IX.1-IX.5 (aux taps are the hidden states *entering*
  the tapped decoder layers, concatenated per position, fused by a bias-free
  Linear(3k, k)), section XI (catch-up, drafting, verify, commit and rollback
  of both caches).
* "Advanced speculative decoding: tree drafts and EAGLE": the target verifies
  a whole tree in one pass with the tree mask at positions prefix + depth,
  walks the longest greedy-matching path and appends that path's K/V.
* "Speculative Decoding (EAGLE3) in the vLLM Neuron Framework", section
  "Auxiliary Hidden State Extraction" (capture before the layer runs).

Readings taken: the decoder layer is the standard Llama layer (pre-norm
attention and SwiGLU MLP, each with a residual); all norm weights are 1 unless
given; the draft's LM head may be the target's (tiny config) or its own.

Every row is computed on its own (matrix-vector products, attention over an
explicit key list in position order), so a row's values do not depend on which
other rows share the call.  That makes greedy speculative decoding produce
exactly the vanilla greedy tokens, the losslessness check that "EAGLE-3:
Engineering Implementation of LLM Inference Acceleration" section XI.6 and the
tree-drafts page run.  Pinned by that equality, and RMSNorm and SiLU by
torch.nn.functional.rms_norm and silu (tests/test_oracle_model.py).
"""
import math

import numpy as np

from .accept import accept_greedy, argmax
from .attention import ROPE_THETA, rope_apply
from .tree import anc_bits, depths


def rmsnorm(x, w, eps):
    x = np.asarray(x, dtype=np.float64)
    return np.asarray(w, dtype=np.float64) * (x / np.sqrt(np.mean(x * x, -1, keepdims=True) + eps))


def silu(x):
    return x / (1.0 + np.exp(-x))


def _rows(W, X):
    """Row-by-row X @ W.T (each output row is one matrix-vector product)."""
    W = np.asarray(W, dtype=np.float64)
    return np.stack([W @ np.asarray(x, dtype=np.float64) for x in X], 0)


class KV:
    """Per-layer K/V cache: lists of [Hkv, D] rows in position order."""

    def __init__(self, n_layers):
        self.k = [[] for _ in range(n_layers)]
        self.v = [[] for _ in range(n_layers)]

    def __len__(self):
        return len(self.k[0])

    def crop(self, n):
        for lst in self.k + self.v:
            del lst[n:]

    def append(self, layer, k_rows, v_rows):
        self.k[layer].extend(list(k_rows))
        self.v[layer].extend(list(v_rows))


def _attend_rows(q, k_new, v_new, cache_k, cache_v, visible, n_kv, scale, pool_k=None, pool_v=None):
    """q [T, Hq, D]; k_new/v_new [T, Hkv, D].  Row i attends to the whole cache, then
    to the rows listed in visible[i], which index the concatenation [pool rows; new rows]."""
    T, Hq, D = q.shape
    rep = Hq // n_kv
    out = np.zeros((T, Hq, D))
    ck = np.stack(cache_k, 0) if cache_k else np.zeros((0, n_kv, D))
    cv = np.stack(cache_v, 0) if cache_v else np.zeros((0, n_kv, D))
    if pool_k is not None and len(pool_k):
        k_new = np.concatenate([np.asarray(pool_k, dtype=np.float64), k_new], 0)
        v_new = np.concatenate([np.asarray(pool_v, dtype=np.float64), v_new], 0)
    for i in range(T):
        keys = np.concatenate([ck, k_new[visible[i]]], 0)             # [S, Hkv, D]
        vals = np.concatenate([cv, v_new[visible[i]]], 0)
        for h in range(Hq):
            g = h // rep
            s = keys[:, g, :] @ q[i, h] * scale
            e = np.exp(s - s.max())
            out[i, h] = (e @ vals[:, g, :]) / e.sum()
    return out


def chain_visible(T):
    return [list(range(i + 1)) for i in range(T)]


def tree_visible(parents):
    bits = anc_bits(parents)
    return [[j for j in range(len(parents)) if (int(bits[i]) >> j) & 1] for i in range(len(parents))]


class Llama:
    """Llama-style decoder: x = Emb[t]; per layer h = x + Attn(norm(x)); x = h + MLP(norm(h))."""

    def __init__(self, w, n_layers, n_heads, n_kv_heads, head_dim, eps=1e-5, theta=ROPE_THETA,
                 aux_layers=()):
        self.w, self.L, self.H, self.KVH, self.D = w, n_layers, n_heads, n_kv_heads, head_dim
        self.eps, self.theta, self.aux_layers = eps, theta, tuple(aux_layers)

    def new_cache(self):
        return KV(self.L)

    def forward(self, tokens, positions, cache, visible):
        """Run rows (tokens at positions) over ``cache`` (not modified).

        Returns (logits [T, V], aux [T, 3d] or None, new_k/new_v per layer [T, Hkv, D])."""
        w, T = self.w, len(tokens)
        x = np.asarray(w["embed"], dtype=np.float64)[np.asarray(tokens)]
        scale = 1.0 / math.sqrt(self.D)
        aux, new_k, new_v = [], [], []
        for l in range(self.L):
            if l in self.aux_layers:
                aux.append(x.copy())
            p = f"layers.{l}."
            h = rmsnorm(x, w[p + "attn_norm"], self.eps)
            q = _rows(w[p + "wq"], h).reshape(T, self.H, self.D)
            k = _rows(w[p + "wk"], h).reshape(T, self.KVH, self.D)
            v = _rows(w[p + "wv"], h).reshape(T, self.KVH, self.D)
            q, k = rope_apply(q, positions, self.theta), rope_apply(k, positions, self.theta)
            new_k.append(k)
            new_v.append(v)
            o = _attend_rows(q, k, v, cache.k[l], cache.v[l], visible, self.KVH, scale)
            x = x + _rows(w[p + "wo"], o.reshape(T, -1))
            h = rmsnorm(x, w[p + "mlp_norm"], self.eps)
            x = x + _rows(w[p + "w_down"], silu(_rows(w[p + "w_gate"], h)) * _rows(w[p + "w_up"], h))
        logits = _rows(w["lm_head"], rmsnorm(x, w["final_norm"], self.eps))
        return logits, (np.concatenate(aux, -1) if aux else None), new_k, new_v

    def commit(self, cache, new_k, new_v, rows):
        for l in range(self.L):
            cache.append(l, new_k[l][rows], new_v[l][rows])


class Eagle3Draft:
    """EAGLE-3 draft head: fc(3k->k), one two-stream decoder layer, norm, LM head."""

    def __init__(self, w, n_heads, n_kv_heads, head_dim, eps=1e-5, theta=ROPE_THETA):
        self.w, self.H, self.KVH, self.D = w, n_heads, n_kv_heads, head_dim
        self.eps, self.theta = eps, theta

    def fuse(self, aux):
        return _rows(self.w["fc"], aux)

    def layer(self, tokens, x, positions, cache, visible, pool_k=None, pool_v=None):
        """Two-stream decoder layer.  Returns (a [T, d], new_k, new_v).

        Rows see the whole draft cache plus the rows ``visible`` lists, indexing
        [pool rows (earlier draft-tree rows); these rows]."""
        w, T = self.w, len(tokens)
        e = np.asarray(w["embed"], dtype=np.float64)[np.asarray(tokens)]
        x = np.asarray(x, dtype=np.float64)
        a2k = np.concatenate([rmsnorm(e, w["input_norm"], self.eps),
                              rmsnorm(x, w["hidden_norm"], self.eps)], -1)
        q = _rows(w["wq"], a2k).reshape(T, self.H, self.D)
        k = _rows(w["wk"], a2k).reshape(T, self.KVH, self.D)
        v = _rows(w["wv"], a2k).reshape(T, self.KVH, self.D)
        q, k = rope_apply(q, positions, self.theta), rope_apply(k, positions, self.theta)
        o = _attend_rows(q, k, v, cache.k[0], cache.v[0], visible, self.KVH, 1.0 / math.sqrt(self.D),
                         pool_k, pool_v)
        x = x + _rows(w["wo"], o.reshape(T, -1))
        h = rmsnorm(x, w["post_norm"], self.eps)
        x = x + _rows(w["w_down"], silu(_rows(w["w_gate"], h)) * _rows(w["w_up"], h))
        return x, k, v

    def logits(self, a):
        return _rows(self.w["lm_head"], rmsnorm(a, self.w["final_norm"], self.eps))


def vanilla_greedy(target, prompt, max_new):
    """Plain greedy decoding, one target row per token."""
    cache = target.new_cache()
    logits, _, nk, nv = target.forward(prompt, np.arange(len(prompt)), cache, chain_visible(len(prompt)))
    target.commit(cache, nk, nv, list(range(len(prompt))))
    out = [argmax(logits[-1].astype(np.float32))]
    while len(out) < max_new:
        pos = len(prompt) + len(out) - 1
        logits, _, nk, nv = target.forward([out[-1]], np.array([pos]), cache, [[0]])
        target.commit(cache, nk, nv, [0])
        out.append(argmax(logits[-1].astype(np.float32)))
    return out


def speculative_greedy(target, draft, prompt, max_new, build_tree):
    """EAGLE-3 greedy speculative decoding for one sequence.

    ``build_tree(draft_step, a_last, root, L)`` returns (tokens, parents) of the
    draft tree with the root token (the target's last output) as node 0; ``draft_step(rows)`` runs draft
    rows for tree nodes (see :func:`oracle.draft_tree.draft_tree_for_sequence`).
    Returns (generated tokens, accepted drafts per cycle)."""
    P = len(prompt)
    t_cache, d_cache = target.new_cache(), KV(1)
    logits, aux, nk, nv = target.forward(prompt, np.arange(P), t_cache, chain_visible(P))
    target.commit(t_cache, nk, nv, list(range(P)))
    committed = list(prompt)
    root = argmax(logits[-1].astype(np.float32))
    fresh_g = draft.fuse(aux)
    drafted, per_cycle = 0, []
    while len(committed) - P < max_new:
        n = len(committed)
        # 1) catch-up: each committed position the draft cache lacks (drafted .. n-1) runs once,
        #    with its fused target feature and the embedding of the token after it (root last)
        cu_tokens = committed[drafted + 1:] + [root]
        a, dk, dv = draft.layer(cu_tokens, fresh_g, np.arange(drafted, n), d_cache, chain_visible(len(cu_tokens)))
        d_cache.append(0, dk, dv)
        drafted = n
        # 2) the draft tree under the root token
        tokens, parents = build_tree(draft, d_cache, a[-1], root, n)
        # 3) verify: one target pass over the tree at positions n + depth
        pos = n + depths(parents)
        logits, aux, nk, nv = target.forward(tokens, pos, t_cache, tree_visible(parents))
        res = accept_greedy(tokens, parents, logits.astype(np.float32))
        path = res["path"]
        # 4) commit the accepted path's target K/V and keep its features for the next catch-up;
        #    the draft cache already ends at the last committed position
        target.commit(t_cache, nk, nv, path)
        committed += [int(tokens[c]) for c in path]
        root = res["next_root"]
        fresh_g = draft.fuse(aux[path])
        per_cycle.append(res["accept_len"])
    out = (committed + [root])[P:P + max_new]
    return out, per_cycle
