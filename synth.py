"""Seeded synthetic inputs shared by the oracle tests, the GPU parity tests and bench.py.

This module only draws random numbers and lays them out; it holds none of the
method's arithmetic (no softmax, no attention, no acceptance rule).  Every
array is a pure function of (seed, shape), drawn with numpy's PCG64 so that a
test can regenerate one sequence of a batch without drawing the others
(``per_row`` generators seed each batch row as (seed, b)).

bf16 data is produced as fp32 values rounded to bf16 (round-to-nearest-even)
and returned as torch bf16 tensors on the CPU together with the fp32 copy of
the same (already rounded) values for the oracle.

Workloads (all synthetic, random-init; no dataset is read):
* tiny Llama target + EAGLE-3 head: d=64, 4 layers, 4 heads of 16, FFN 172,
  vocab 256, N(0, 0.02) weights, norm weights 1, 32-token uniform prompt.
* acceptance: target logits N(0, 3^2), draft logits = target + N(0, 1),
  random parent arrays with depth <= 6 and <= 10 children per node.
* verify attention: Q, tree K/V and cache K/V N(0, 1) in bf16.
* draft head at Llama-3.1-8B shapes: aux states N(0, 1), weights N(0, 0.02).
"""
import numpy as np
import torch


def rng(*seed):
    return np.random.Generator(np.random.PCG64(list(seed)))


def to_bf16(x):
    """fp32 array -> (torch bf16 tensor, fp32 numpy copy of the rounded values)."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t, t.float().numpy()


# ----------------------------------------------------------------------------- trees
def random_tree(r, n_nodes=60, max_depth=6, max_children=10):
    """Random parent array: node 0 root, parents[i] < i, depth <= max_depth,
    at most max_children children per node, nodes ordered by depth."""
    if n_nodes == 1:
        return np.array([-1], dtype=np.int32)
    # nodes per depth: at least one per depth up to a random depth, the rest spread
    # smallest depth whose capacity (max_children + max_children**2 + ...) holds n_nodes - 1
    d_min, cap = 1, max_children
    while cap < n_nodes - 1:
        d_min += 1
        cap += max_children ** d_min
    hi = min(max_depth, n_nodes - 1)
    if d_min > hi:
        raise ValueError("no tree with these limits has that many nodes")
    depth = int(r.integers(d_min, hi + 1))
    counts = np.ones(depth, dtype=np.int64)
    for _ in range(n_nodes - 1 - depth):
        while True:
            d = int(r.integers(0, depth))
            cap = max_children if d == 0 else counts[d - 1] * max_children
            if counts[d] < cap:
                counts[d] += 1
                break
    parents, level_prev, nxt = [-1], [0], 1
    for d in range(depth):
        level = list(range(nxt, nxt + int(counts[d])))
        kids = {p: 0 for p in level_prev}
        chosen = []
        for _ in level:
            free = [p for p in level_prev if kids[p] < max_children]
            p = free[int(r.integers(0, len(free)))]
            kids[p] += 1
            chosen.append(p)
        chosen.sort()
        parents.extend(chosen)
        level_prev, nxt = level, nxt + len(level)
    return np.asarray(parents, dtype=np.int32)


def chain_tree(n_nodes):
    return np.arange(-1, n_nodes - 1, dtype=np.int32)


# ----------------------------------------------------------------------------- acceptance
def accept_row(seed, b, N, V):
    """Per-sequence logits and tree: (z_target [N, V] f32, z_draft [N, V] f32, parents [N])."""
    r = rng(seed, b)
    parents = random_tree(r, N)
    z_t = (3.0 * r.standard_normal((N, V), dtype=np.float32)).astype(np.float32)
    z_d = (z_t + r.standard_normal((N, V), dtype=np.float32)).astype(np.float32)
    return z_t, z_d, parents


def tokens_top_draft(z_draft, parents):
    """Children of node u take the draft's highest-logit tokens at u, in node order."""
    N = len(parents)
    tokens = np.zeros(N, dtype=np.int32)
    tokens[0] = 0
    for u in range(N):
        kids = [c for c in range(N) if parents[c] == u]
        if not kids:
            continue
        top = np.argpartition(-z_draft[u], len(kids))[: len(kids)]
        top = top[np.argsort(-z_draft[u][top], kind="stable")]
        for c, t in zip(kids, top):
            tokens[c] = t
    return tokens


def tokens_sampled_draft(z_draft, parents, seed, b):
    """Children of node u are distinct tokens drawn without replacement from
    softmax(z_draft[u]) (Gumbel top-k with numpy's own generator)."""
    r = rng(seed, b, 7)
    N = len(parents)
    tokens = np.zeros(N, dtype=np.int32)
    for u in range(N):
        kids = [c for c in range(N) if parents[c] == u]
        if not kids:
            continue
        g = z_draft[u].astype(np.float64) - np.log(-np.log(r.random(z_draft.shape[1])))
        top = np.argpartition(-g, len(kids))[: len(kids)]
        top = top[np.argsort(-g[top], kind="stable")]
        for c, t in zip(kids, top):
            tokens[c] = t
    return tokens


def accept_batch(seed, B, N, V, sampled=False):
    """Whole batch for the acceptance stage (numpy, fp32 logits)."""
    zt = np.empty((B, N, V), np.float32)
    zd = np.empty((B, N, V), np.float32)
    parents = np.empty((B, N), np.int32)
    tokens = np.empty((B, N), np.int32)
    for b in range(B):
        zt[b], zd[b], parents[b] = accept_row(seed, b, N, V)
        tokens[b] = (tokens_sampled_draft(zd[b], parents[b], seed, b) if sampled
                     else tokens_top_draft(zd[b], parents[b]))
    return zt, zd, parents, tokens


# ----------------------------------------------------------------------------- verify attention
def verify_attn_row(seed, b, N, Hq, Hkv, D, L, S_max):
    """Per-sequence fp32 values (already bf16-representable after to_bf16)."""
    r = rng(seed, b)
    parents = random_tree(r, N)
    q = r.standard_normal((N, Hq, D), dtype=np.float32)
    tk = r.standard_normal((N, Hkv, D), dtype=np.float32)
    tv = r.standard_normal((N, Hkv, D), dtype=np.float32)
    kc = np.zeros((Hkv, S_max, D), np.float32)
    vc = np.zeros((Hkv, S_max, D), np.float32)
    kc[:, :L] = r.standard_normal((Hkv, L, D), dtype=np.float32)
    vc[:, :L] = r.standard_normal((Hkv, L, D), dtype=np.float32)
    return q, tk, tv, kc, vc, parents


def verify_attn_batch(seed, B, N, Hq, Hkv, D, prefix_lens, S_max):
    """bf16 torch tensors (CPU) + fp32 numpy copies for the whole batch."""
    q = np.empty((B, N, Hq, D), np.float32)
    tk = np.empty((B, N, Hkv, D), np.float32)
    tv = np.empty((B, N, Hkv, D), np.float32)
    kc = np.empty((B, Hkv, S_max, D), np.float32)
    vc = np.empty((B, Hkv, S_max, D), np.float32)
    parents = np.empty((B, N), np.int32)
    for b in range(B):
        q[b], tk[b], tv[b], kc[b], vc[b], parents[b] = verify_attn_row(
            seed, b, N, Hq, Hkv, D, int(prefix_lens[b]), S_max)
    out = {}
    for name, arr in (("q", q), ("tree_k", tk), ("tree_v", tv), ("k_cache", kc), ("v_cache", vc)):
        out[name], out[name + "_f32"] = to_bf16(arr)
    out["parents"] = parents
    out["prefix_len"] = np.asarray(prefix_lens, np.int32)
    return out


# ----------------------------------------------------------------------------- models
def normal(seed, tag, shape, std):
    return (std * rng(seed, tag).standard_normal(shape, dtype=np.float32)).astype(np.float32)


def llama_weights(seed, d, n_layers, n_heads, n_kv_heads, head_dim, ffn, vocab, std=0.02):
    """Target weights as fp32 numpy arrays; matrices are [out, in] (nn.Linear layout)."""
    w, tag = {}, 0

    def nxt(shape):
        nonlocal tag
        tag += 1
        return normal(seed, tag, shape, std)

    w["embed"] = nxt((vocab, d))
    for l in range(n_layers):
        p = f"layers.{l}."
        w[p + "attn_norm"] = np.ones(d, np.float32)
        w[p + "wq"] = nxt((n_heads * head_dim, d))
        w[p + "wk"] = nxt((n_kv_heads * head_dim, d))
        w[p + "wv"] = nxt((n_kv_heads * head_dim, d))
        w[p + "wo"] = nxt((d, n_heads * head_dim))
        w[p + "mlp_norm"] = np.ones(d, np.float32)
        w[p + "w_gate"] = nxt((ffn, d))
        w[p + "w_up"] = nxt((ffn, d))
        w[p + "w_down"] = nxt((d, ffn))
    w["final_norm"] = np.ones(d, np.float32)
    w["lm_head"] = nxt((vocab, d))
    return w


def eagle3_weights(seed, d, n_heads, n_kv_heads, head_dim, ffn, vocab, embed, lm_head=None,
                   std=0.02):
    """EAGLE-3 head weights; ``embed`` is the target's table, ``lm_head`` the
    target head to share (tiny config) or None for an own random head."""
    w, tag = {}, 1000

    def nxt(shape):
        nonlocal tag
        tag += 1
        return normal(seed, tag, shape, std)

    w["fc"] = nxt((d, 3 * d))
    w["embed"] = embed
    w["input_norm"] = np.ones(d, np.float32)
    w["hidden_norm"] = np.ones(d, np.float32)
    w["wq"] = nxt((n_heads * head_dim, 2 * d))
    w["wk"] = nxt((n_kv_heads * head_dim, 2 * d))
    w["wv"] = nxt((n_kv_heads * head_dim, 2 * d))
    w["wo"] = nxt((d, n_heads * head_dim))
    w["post_norm"] = np.ones(d, np.float32)
    w["w_gate"] = nxt((ffn, d))
    w["w_up"] = nxt((ffn, d))
    w["w_down"] = nxt((d, ffn))
    w["final_norm"] = np.ones(d, np.float32)
    w["lm_head"] = lm_head if lm_head is not None else nxt((vocab, d))
    return w


TINY = dict(d=64, n_layers=4, n_heads=4, n_kv_heads=4, head_dim=16, ffn=172, vocab=256)
TINY_AUX_LAYERS = (1, 2, 3)


def tiny_prompt(seed=0, length=32, vocab=256):
    return [int(t) for t in rng(seed, 99).integers(0, vocab, length)]


# ----------------------------------------------------------------------------- ragged chains
def chain_batch(seed, R, K, V, greedy_every=3):
    """A ragged verify batch of R requests: draft counts in 0..K, target logits N(0, 3^2) for each
    request's d + 1 rows (its verification rows, then its bonus row), draft tokens that are the
    argmax of the row's logits plus N(0, 1) noise (a draft that often, not always, agrees), and
    every greedy_every-th request greedy.  Returns numpy arrays: num_draft [R], logits [rows, V]
    fp32, drafts [sum d] int32, greedy [R] int32."""
    r = rng(seed, 31)
    d = r.integers(0, K + 1, R).astype(np.int32)
    rows = int(d.sum()) + R
    logits = (3.0 * r.standard_normal((rows, V), dtype=np.float32)).astype(np.float32)
    drafts, row = [], 0
    for i in range(R):
        for j in range(int(d[i])):
            noisy = logits[row + j] + r.standard_normal(V, dtype=np.float32)
            drafts.append(int(np.argmax(noisy)))
        row += int(d[i]) + 1
    greedy = (np.arange(R) % greedy_every == 0).astype(np.int32)
    return d, logits, np.asarray(drafts, np.int32), greedy


# ----------------------------------------------------------------------------- training-time test
def ttt_batch(seed, Bt, T, Hq, Hkv, D, S):
    """q [Bt, T, Hq, D] and k / v [S, Bt, T, Hkv, D] (step 0 native, then S - 1 simulated steps),
    N(0, 1) rounded to bf16: (torch bf16 tensors, fp32 numpy copies)."""
    r = rng(seed, 41)
    q = r.standard_normal((Bt, T, Hq, D), dtype=np.float32)
    k = r.standard_normal((S, Bt, T, Hkv, D), dtype=np.float32)
    v = r.standard_normal((S, Bt, T, Hkv, D), dtype=np.float32)
    out = {}
    for name, arr in (("q", q), ("k", k), ("v", v)):
        out[name], out[name + "_f32"] = to_bf16(arr)
    return out
