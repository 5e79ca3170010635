"""The tiny lossless configuration on the GPU: a small fp32 Llama-style target and its EAGLE-3 head,
composed from the library's fp32 blocks (eagle3_f32_*), greedy acceptance (eagle3_accept) and
compaction (eagle3_compact_kv).  Every computation runs in the library's kernels; this module only
sequences the calls and moves token ids between steps.

Sources: "EAGLE-3: Engineering Implementation of LLM Inference Acceleration", appendix C (the
Llama layer), section VIII (the draft head: fc over the aux states, a two-stream decoder layer,
norm, LM head), sections IX and XI (aux taps entering layers; catch-up, draft, verify, accept,
commit); "Advanced speculative decoding: tree drafts and EAGLE", section "Implementation" (one
verification pass over the draft at positions prefix + depth, the longest greedy-matching path,
its K/V appended without recomputation).

Greedy speculative decoding reproduces vanilla greedy decoding token for token because the fp32
blocks compute every row on its own in a fixed order (see include/eagle3_f32.h).
"""
import numpy as np
import torch

from . import _lib as L

ROPE_THETA = 500000.0


def _t(a, dev, dtype=torch.float32):
    return torch.as_tensor(np.ascontiguousarray(a), dtype=dtype, device=dev)


def _bits(rows):
    """int64 tensor of bitmasks from lists of visible new-row indices."""
    out = []
    for r in rows:
        v = 0
        for j in r:
            v |= 1 << j
        out.append(v - (1 << 64) if v >= (1 << 63) else v)
    return out


def chain_visible(T):
    return [list(range(i + 1)) for i in range(T)]


class _Cache:
    """K/V cache [layers][1, Hkv, s_max, D] fp32 plus its device length, filled by compaction."""

    def __init__(self, n_layers, n_kv_heads, head_dim, s_max, dev):
        self.k = torch.zeros(n_layers, 1, n_kv_heads, s_max, head_dim, device=dev)
        self.v = torch.zeros_like(self.k)
        self.length = torch.zeros(1, dtype=torch.int32, device=dev)
        self.n_layers, self.Hkv, self.D, self.S = n_layers, n_kv_heads, head_dim, s_max

    def commit(self, tree_k, tree_v, path, n_rows, aux=None):
        """Append rows `path` (host list) of this pass's tree_k / tree_v [layers, T, Hkv*D] at the
        current length; returns the gathered aux rows [len(path), A] when aux [T, A] is given."""
        dev = self.k.device
        W = len(path)
        path_d = _t(path, dev, torch.int32)
        alen = _t([W - 1], dev, torch.int32)
        slot_map = torch.empty(W, dtype=torch.int32, device=dev)
        aux_out = torch.empty(W, aux.shape[1], device=dev) if aux is not None else None
        L.eagle3_compact_kv(self.k, self.v, tree_k.view(self.n_layers, 1, n_rows, self.Hkv, self.D),
                            tree_v.view(self.n_layers, 1, n_rows, self.Hkv, self.D), path_d.view(1, W),
                            alen, self.length, slot_map.view(1, W),
                            aux_tree=None if aux is None else aux.view(1, n_rows, -1),
                            aux_out=None if aux_out is None else aux_out.view(1, W, -1))
        return aux_out


class TinyTarget:
    def __init__(self, w, n_layers, n_heads, n_kv_heads, head_dim, aux_layers, s_max, dev, eps=1e-5):
        self.w = {k: _t(v, dev) for k, v in w.items()}
        self.Lyr, self.H, self.KVH, self.D, self.eps = n_layers, n_heads, n_kv_heads, head_dim, eps
        self.aux_layers = tuple(aux_layers)
        self.d = self.w["embed"].shape[1]
        self.dev = dev
        self.cache = _Cache(n_layers, n_kv_heads, head_dim, s_max, dev)

    def forward(self, tokens, positions, visible, cache_len):
        """Rows for `tokens` at `positions` over the first cache_len cache positions; row i also sees
        the new rows listed in visible[i].  Returns logits [T, V], aux [T, 3d] (or None) and the
        rows' rotated keys / values [layers, T, Hkv*D]."""
        w, dev, T, d = self.w, self.dev, len(tokens), self.d
        H, KVH, D = self.H, self.KVH, self.D
        tok, pos = _t(tokens, dev, torch.int32), _t(positions, dev, torch.int32)
        vis = _t(_bits(visible), dev, torch.int64)
        x = torch.empty(T, d, device=dev)
        L.eagle3_f32_gather(w["embed"], tok, x)
        aux = torch.empty(T, len(self.aux_layers) * d, device=dev) if self.aux_layers else None
        ident = torch.arange(T, dtype=torch.int32, device=dev)
        tree_k = torch.empty(self.Lyr, T, KVH * D, device=dev)
        tree_v = torch.empty_like(tree_k)
        h = torch.empty(T, d, device=dev)
        q = torch.empty(T, H * D, device=dev)
        o = torch.empty(T, H * D, device=dev)
        act = torch.empty(T, w["layers.0.w_gate"].shape[0], device=dev)
        for l in range(self.Lyr):
            if l in self.aux_layers:
                s = self.aux_layers.index(l)
                L.eagle3_f32_gather(x, ident, aux[:, s * d:(s + 1) * d])
            p = f"layers.{l}."
            L.eagle3_f32_rmsnorm(x, w[p + "attn_norm"], h, eps=self.eps)
            L.eagle3_f32_linear(h, w[p + "wq"], q)
            L.eagle3_f32_linear(h, w[p + "wk"], tree_k[l])
            L.eagle3_f32_linear(h, w[p + "wv"], tree_v[l])
            L.eagle3_f32_rope(q, H, D, pos, theta=ROPE_THETA)
            L.eagle3_f32_rope(tree_k[l], KVH, D, pos, theta=ROPE_THETA)
            L.eagle3_f32_attn(q, tree_k[l], tree_v[l], self.cache.k[l, 0], self.cache.v[l, 0], vis, o,
                              n_heads=H, n_kv_heads=KVH, head_dim=D, cache_len=cache_len)
            L.eagle3_f32_linear(o, w[p + "wo"], x, epilogue=L.F32_EPI_RESIDUAL, residual=x)
            L.eagle3_f32_rmsnorm(x, w[p + "mlp_norm"], h, eps=self.eps)
            L.eagle3_f32_linear(h, w[p + "w_gate"], act, epilogue=L.F32_EPI_SWIGLU, w2=w[p + "w_up"])
            L.eagle3_f32_linear(act, w[p + "w_down"], x, epilogue=L.F32_EPI_RESIDUAL, residual=x)
        L.eagle3_f32_rmsnorm(x, w["final_norm"], h, eps=self.eps)
        logits = torch.empty(T, w["lm_head"].shape[0], device=dev)
        L.eagle3_f32_linear(h, w["lm_head"], logits)
        return logits, aux, tree_k, tree_v


class TinyDraft:
    """EAGLE-3 head: fc(3d -> d), one two-stream decoder layer, final norm, LM head."""

    def __init__(self, w, n_heads, n_kv_heads, head_dim, s_max, dev, eps=1e-5):
        self.w = {k: _t(v, dev) for k, v in w.items()}
        self.H, self.KVH, self.D, self.eps, self.dev = n_heads, n_kv_heads, head_dim, eps, dev
        self.d = self.w["fc"].shape[0]
        self.cache = _Cache(1, n_kv_heads, head_dim, s_max, dev)

    def fuse(self, aux):
        g = torch.empty(aux.shape[0], self.d, device=self.dev)
        L.eagle3_f32_linear(aux, self.w["fc"], g)
        return g

    def layer(self, tokens, x, positions, visible, cache_len):
        """Returns a [T, d] (pre-norm output) and the rows' rotated keys / values [1, T, Hkv*D]."""
        w, dev, T, d = self.w, self.dev, len(tokens), self.d
        H, KVH, D = self.H, self.KVH, self.D
        tok, pos = _t(tokens, dev, torch.int32), _t(positions, dev, torch.int32)
        vis = _t(_bits(visible), dev, torch.int64)
        e = torch.empty(T, d, device=dev)
        L.eagle3_f32_gather(w["embed"], tok, e)
        a2k = torch.empty(T, 2 * d, device=dev)
        L.eagle3_f32_rmsnorm(e, w["input_norm"], a2k[:, :d], eps=self.eps)
        L.eagle3_f32_rmsnorm(x, w["hidden_norm"], a2k[:, d:], eps=self.eps)
        q = torch.empty(T, H * D, device=dev)
        k = torch.empty(1, T, KVH * D, device=dev)
        v = torch.empty_like(k)
        L.eagle3_f32_linear(a2k, w["wq"], q)
        L.eagle3_f32_linear(a2k, w["wk"], k[0])
        L.eagle3_f32_linear(a2k, w["wv"], v[0])
        L.eagle3_f32_rope(q, H, D, pos, theta=ROPE_THETA)
        L.eagle3_f32_rope(k[0], KVH, D, pos, theta=ROPE_THETA)
        o = torch.empty(T, H * D, device=dev)
        L.eagle3_f32_attn(q, k[0], v[0], self.cache.k[0, 0], self.cache.v[0, 0], vis, o,
                          n_heads=H, n_kv_heads=KVH, head_dim=D, cache_len=cache_len)
        a = torch.empty(T, d, device=dev)
        L.eagle3_f32_linear(o, w["wo"], a, epilogue=L.F32_EPI_RESIDUAL, residual=x)
        h = torch.empty(T, d, device=dev)
        L.eagle3_f32_rmsnorm(a, w["post_norm"], h, eps=self.eps)
        act = torch.empty(T, w["w_gate"].shape[0], device=dev)
        L.eagle3_f32_linear(h, w["w_gate"], act, epilogue=L.F32_EPI_SWIGLU, w2=w["w_up"])
        L.eagle3_f32_linear(act, w["w_down"], a, epilogue=L.F32_EPI_RESIDUAL, residual=a)
        return a, k, v

    def logits(self, a):
        h = torch.empty_like(a)
        L.eagle3_f32_rmsnorm(a, self.w["final_norm"], h, eps=self.eps)
        out = torch.empty(a.shape[0], self.w["lm_head"].shape[0], device=self.dev)
        L.eagle3_f32_linear(h, self.w["lm_head"], out)
        return out


def _argmax(logits_row):
    out = torch.empty(1, dtype=torch.int32, device=logits_row.device)
    L.eagle3_f32_argmax(logits_row.view(1, -1), out)
    return int(out.item())


def vanilla_greedy(target, prompt, max_new):
    """Plain greedy decoding: the prompt in one pass, then one target row per token."""
    P = len(prompt)
    logits, _, tk, tv = target.forward(prompt, list(range(P)), chain_visible(P), 0)
    target.cache.commit(tk, tv, list(range(P)), P)
    out = [_argmax(logits[P - 1])]
    while len(out) < max_new:
        pos = P + len(out) - 1
        logits, _, tk, tv = target.forward([out[-1]], [pos], [[0]], pos)
        target.cache.commit(tk, tv, [0], 1)
        out.append(_argmax(logits[0]))
    return out


def speculative_greedy(target, draft, prompt, max_new, k_draft=4, propose=None):
    """EAGLE-3 greedy speculative decoding with a chain draft of k_draft tokens.  Returns the
    generated tokens and the accepted drafts per cycle.

    propose(n, root, k), when given, returns the k chain tokens to verify in place of the draft's
    own argmax choices (n = committed positions, root = the token at position n).  The draft head
    still runs its catch-up and its chain rows on those tokens, so a proposer that agrees with the
    target exercises accepted drafts, multi-row commits and catch-ups of several rows, which a
    random-init draft never reaches."""
    dev = target.dev
    P = len(prompt)
    logits, aux, tk, tv = target.forward(prompt, list(range(P)), chain_visible(P), 0)
    target.cache.commit(tk, tv, list(range(P)), P)
    committed = list(prompt)
    root = _argmax(logits[P - 1])
    fresh_g = draft.fuse(aux)
    drafted, per_cycle = 0, []
    N = k_draft + 1
    parents = _t([-1] + list(range(k_draft)), dev, torch.int32).view(1, N)
    while len(committed) - P < max_new:
        n = len(committed)
        # catch-up: each committed position the draft cache lacks (drafted .. n-1) runs once, with
        # its fused target feature and the embedding of the token after it (the root for the last)
        cu_tokens = committed[drafted + 1:] + [root]
        a, dk, dv = draft.layer(cu_tokens, fresh_g, list(range(drafted, n)), chain_visible(len(cu_tokens)), drafted)
        draft.cache.commit(dk, dv, list(range(len(cu_tokens))), len(cu_tokens))
        drafted = n
        # chain draft: depth 1 from the last catch-up row; each later depth one row at position
        # n + depth - 2 over the draft cache and the chain rows before it (kept in the cache slots
        # after n, which the next catch-up overwrites)
        a_prev = a[-1:].clone()
        forced = None if propose is None else [int(t) for t in propose(n, root, k_draft)]
        chain = [_argmax(draft.logits(a_prev)[0]) if forced is None else forced[0]]
        for t in range(2, k_draft + 1):
            row_a, rk, rv = draft.layer([chain[-1]], a_prev, [n + t - 2], [[0]], n + t - 2)
            draft.cache.commit(rk, rv, [0], 1)
            chain.append(_argmax(draft.logits(row_a)[0]) if forced is None else forced[t - 1])
            a_prev = row_a
        draft.cache.length.copy_(torch.tensor([drafted], dtype=torch.int32))   # drop the chain rows
        # verify [root] + chain at positions n + depth
        tokens = [root] + chain
        logits, aux, tk, tv = target.forward(tokens, list(range(n, n + N)), chain_visible(N), n)
        tok_d = _t(tokens, dev, torch.int32).view(1, N)
        alen = torch.empty(1, dtype=torch.int32, device=dev)
        path = torch.empty(1, N, dtype=torch.int32, device=dev)
        emitted = torch.empty(1, N, dtype=torch.int32, device=dev)
        nroot = torch.empty(1, dtype=torch.int32, device=dev)
        L.eagle3_accept(L.GREEDY, logits.view(1, N, -1), tok_d, parents, alen, path, emitted, nroot)
        n_acc = int(alen.item())
        path_h = [int(v) for v in path[0, :n_acc + 1].tolist()]
        aux_rows = target.cache.commit(tk, tv, path_h, N, aux=aux)
        committed += [tokens[c] for c in path_h]
        root = int(nroot.item())
        fresh_g = draft.fuse(aux_rows)
        per_cycle.append(n_acc)
    return committed[P:P + max_new], per_cycle
