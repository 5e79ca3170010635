"""Pins of the oracle's attention, tiny Llama / EAGLE-3 head and draft-tree builder (CPU only)."""
import math

import numpy as np
import pytest

import synth
from oracle import attention as att
from oracle import draft_tree, llama, tree
from oracle.accept import order_key
from tests._util import agreeing_proposer


# ----------------------------------------------------------------------------- RoPE / attention
def test_rope_preserves_norm_and_is_relative():
    r = np.random.default_rng(0)
    D = 128
    q = r.standard_normal((1, 1, D))
    k = r.standard_normal((1, 1, D))
    for m, n in ((3, 1), (300, 298), (700, 698)):
        qm, kn = att.rope_apply(q, [m]), att.rope_apply(k, [n])
        assert abs(np.linalg.norm(qm) - np.linalg.norm(q)) < 1e-9
        if m < 400:
            # relative-position property: <R_m q, R_n k> depends only on m - n
            ref = float((att.rope_apply(q, [2]) * att.rope_apply(k, [0])).sum())
            assert abs(float((qm * kn).sum()) - ref) < 2e-3
    assert np.allclose(att.rope_apply(q, [0]), q)


def test_rope_is_the_complex_rotation_of_half_split_pairs():
    """Rotate-half RoPE is the complex rotation z_j * exp(i * pos * inv_j) of z_j = x_j + i x_{j+D/2},
    with inv_j = theta^(-2j/D): the pairing and the frequencies, which the invariants above do not
    fix (an interleaved pairing or another frequency law keeps norms and relative positions)."""
    assert att.rope_inv(4, 10000.0).tolist() == [1.0, np.float32(0.01)]
    r = np.random.default_rng(3)
    D, T = 128, 5
    x = r.standard_normal((T, 2, D))
    pos = np.array([0, 1, 17, 2048, 131071])
    got = att.rope_apply(x, pos)
    ang = pos[:, None].astype(np.float32) * att.rope_inv(D)[None, :]          # fp32 angles
    z = (x[..., : D // 2] + 1j * x[..., D // 2:]) * np.exp(1j * ang.astype(np.float64))[:, None, :]
    ref = np.concatenate([z.real, z.imag], -1)
    assert np.abs(got - ref).max() < 1e-12


def test_rmsnorm_and_silu_match_torch():
    torch = pytest.importorskip("torch")
    r = np.random.default_rng(4)
    x, w = r.standard_normal((7, 96)), r.standard_normal(96)
    ref = torch.nn.functional.rms_norm(torch.from_numpy(x), (96,), torch.from_numpy(w), 1e-5).numpy()
    assert np.abs(llama.rmsnorm(x, w, 1e-5) - ref).max() < 1e-12
    y = 6.0 * r.standard_normal(1000)
    assert np.abs(llama.silu(y) - torch.nn.functional.silu(torch.from_numpy(y)).numpy()).max() < 1e-12


def _inputs(seed, N, L, Hq=4, Hkv=2, D=16, parents=None):
    r = np.random.default_rng(seed)
    q = r.standard_normal((1, N, Hq, D))
    tk = r.standard_normal((1, N, Hkv, D))
    tv = r.standard_normal((1, N, Hkv, D))
    kc = r.standard_normal((1, Hkv, L + 5, D))
    vc = r.standard_normal((1, Hkv, L + 5, D))
    if parents is None:
        parents = synth.random_tree(r, N, max_depth=4, max_children=3)
    return q, tk, tv, kc, vc, np.asarray(parents)[None]


def test_chain_tree_is_causal_attention():
    N, L, Hq, Hkv, D = 6, 9, 4, 2, 16
    q, tk, tv, kc, vc, parents = _inputs(1, N, L, parents=synth.chain_tree(N))
    o, lse, kr = att.verify_attention(q, tk, tv, kc, vc, parents, [L])
    pos = L + np.arange(N)
    qr = att.rope_apply(q[0], pos)
    for h in range(Hq):
        g = h // (Hq // Hkv)
        keys = np.concatenate([kc[0, g, :L], kr[0, :, g]], 0)
        vals = np.concatenate([vc[0, g, :L], tv[0, :, g]], 0)
        qs = np.concatenate([np.zeros((L, D)), qr[:, h]], 0)          # prefix rows unused
        ref = att.causal_attention(qs, keys, vals, 1 / math.sqrt(D))[L:]
        assert np.abs(o[0, :, h] - ref).max() < 1e-12


def test_each_node_equals_its_path_as_a_sequence():
    N, L, Hq, Hkv, D = 12, 7, 4, 2, 16
    q, tk, tv, kc, vc, parents = _inputs(2, N, L)
    o, lse, kr = att.verify_attention(q, tk, tv, kc, vc, parents, [L])
    par = parents[0].tolist()
    for i in range(N):
        path = tree.path_to(par, i)
        pos = L + np.arange(len(path))
        qr = att.rope_apply(q[0, path], pos)
        krp = att.rope_apply(tk[0, path], pos)
        for h in range(Hq):
            g = h // (Hq // Hkv)
            keys = np.concatenate([kc[0, g, :L], krp[:, g]], 0)
            vals = np.concatenate([vc[0, g, :L], tv[0, path, g]], 0)
            qs = np.concatenate([np.zeros((L, D)), qr[:, h]], 0)
            ref = att.causal_attention(qs, keys, vals, 1 / math.sqrt(D))[-1]
            assert np.abs(o[0, i, h] - ref).max() < 1e-12
            s = keys @ qr[-1, h] / math.sqrt(D)
            assert abs(lse[0, i, h] - math.log(np.exp(s).sum())) < 1e-9


def test_empty_prefix():
    q, tk, tv, kc, vc, parents = _inputs(3, 5, 0)
    o, lse, kr = att.verify_attention(q, tk, tv, kc, vc, parents, [0])
    # the root sees only itself: output = its own value row
    for h in range(4):
        assert np.abs(o[0, 0, h] - tv[0, 0, h // 2]).max() < 1e-12


# ----------------------------------------------------------------------------- tiny Llama / EAGLE-3
def _tiny():
    cfg = synth.TINY
    tw = synth.llama_weights(0, **cfg)
    target = llama.Llama(tw, cfg["n_layers"], cfg["n_heads"], cfg["n_kv_heads"], cfg["head_dim"],
                         aux_layers=synth.TINY_AUX_LAYERS)
    dw = synth.eagle3_weights(0, cfg["d"], cfg["n_heads"], cfg["n_kv_heads"], cfg["head_dim"],
                              cfg["ffn"], cfg["vocab"], embed=tw["embed"], lm_head=tw["lm_head"])
    draft = llama.Eagle3Draft(dw, cfg["n_heads"], cfg["n_kv_heads"], cfg["head_dim"])
    return target, draft


def _builder(depth, top_k, n_nodes):
    def build(draft, d_cache, a_last, pending, L):
        res = draft_tree.draft_tree_for_sequence(draft, d_cache, a_last, pending, L, depth, top_k, n_nodes)
        return res["tokens"].tolist(), res["parents"].tolist()
    return build


def test_greedy_speculative_equals_vanilla_chain():
    """Tiny lossless check: K = 4 chain, 64 new tokens, output == vanilla greedy."""
    target, draft = _tiny()
    prompt = synth.tiny_prompt(0)
    ref = llama.vanilla_greedy(target, prompt, 64)
    out, accepted = llama.speculative_greedy(target, draft, prompt, 64, _builder(4, 1, 5))
    assert out == ref
    assert len(out) == 64
    assert all(0 <= a <= 4 for a in accepted)


def test_greedy_speculative_equals_vanilla_tree():
    target, draft = _tiny()
    prompt = synth.tiny_prompt(1)
    ref = llama.vanilla_greedy(target, prompt, 24)
    out, _ = llama.speculative_greedy(target, draft, prompt, 24, _builder(3, 3, 10))
    assert out == ref


def _proposal_builder(propose, k, siblings=False):
    """build_tree for the oracle loop from a proposer: the proposal as a chain under the root and,
    with siblings, one extra child per level carrying another token (a tree whose accepted path is
    one of several branches)."""
    def build(draft, d_cache, a_last, root, L):
        chain = propose(L, root, k)
        tokens, parents = [root] + chain, [-1] + list(range(k))
        if siblings:
            for j in range(1, k + 1):
                tokens.append((chain[j - 1] + 17) % draft.w["lm_head"].shape[0])
                parents.append(j - 1)
        return tokens, parents
    return build


@pytest.mark.parametrize("siblings", [False, True])
def test_greedy_speculative_equals_vanilla_with_accepted_drafts(siblings):
    """Losslessness with drafts that are accepted: a proposer that follows vanilla greedy (with
    planted mismatches) drives accept lengths of 4 and of 1-3, multi-row commits and catch-ups of
    several rows ("EAGLE-3: Engineering Implementation of LLM Inference Acceleration", section XI.6:
    the kept positions are caught up by the draft, the rest of the draft is rolled back); the
    output still equals vanilla greedy token for token."""
    target, draft = _tiny()
    prompt = synth.tiny_prompt(0)
    ref = llama.vanilla_greedy(target, prompt, 64)
    V = synth.TINY["vocab"]
    propose = agreeing_proposer(ref, len(prompt), 4, V)
    out, accepted = llama.speculative_greedy(target, draft, prompt, 64, _proposal_builder(propose, 4, siblings))
    assert out == ref
    assert 4 in accepted and any(1 <= a <= 3 for a in accepted), accepted
    assert sum(accepted) + len(accepted) >= 64 - 1


def _tree_vs_paths(target, prompt, parents, tokens, visible):
    cache = target.new_cache()
    P = len(prompt)
    _, _, nk, nv = target.forward(prompt, np.arange(P), cache, llama.chain_visible(P))
    target.commit(cache, nk, nv, list(range(P)))
    logits, _, _, _ = target.forward(tokens, P + tree.depths(parents), cache, visible)
    worst = 0.0
    for i in range(len(parents)):
        path = tree.path_to(parents, i)
        c2 = target.new_cache()
        seq = prompt + [tokens[j] for j in path]
        ref, _, _, _ = target.forward(seq, np.arange(len(seq)), c2, llama.chain_visible(len(seq)))
        worst = max(worst, float(np.abs(logits[i] - ref[-1]).max()))
    return worst


def test_tree_verify_logits_equal_path_logits():
    """Each node's logits equal prefix + its path run as an ordinary sequence; the
    comparison is sharp: a mask that lets every node see every node is caught."""
    target, _ = _tiny()
    prompt = synth.tiny_prompt(2)[:10]
    parents = [-1, 0, 0, 1, 1, 2, 3, 5]
    tokens = [7, 100, 200, 30, 31, 45, 12, 9]
    assert _tree_vs_paths(target, prompt, parents, tokens, llama.tree_visible(parents)) < 1e-12
    everything = [list(range(len(parents)))] * len(parents)
    assert _tree_vs_paths(target, prompt, parents, tokens, everything) > 1e-6


def _torch_stream(w, cfg, tokens, theta=att.ROPE_THETA, eps=1e-5):
    """The tiny Llama's residual stream written with torch ops in fp64, independently of the
    oracle: torch rms_norm, scaled_dot_product_attention with a causal mask, SiLU, and RoPE as the
    complex rotation of half-split pairs at the fp32 angles fp32(pos) * fp32(theta^(-2j/D)).
    Returns [x entering layer 0, x entering layer 1, ..., x after the last layer] and the logits."""
    torch = pytest.importorskip("torch")
    F = torch.nn.functional
    d, H, KVH, D, nl = cfg["d"], cfg["n_heads"], cfg["n_kv_heads"], cfg["head_dim"], cfg["n_layers"]
    t = lambda a: torch.from_numpy(np.asarray(a, dtype=np.float64))
    T = len(tokens)
    inv = torch.tensor((float(theta) ** (-2.0 * np.arange(D // 2) / D)).astype(np.float32))
    ang = (torch.arange(T, dtype=torch.float32)[:, None] * inv[None, :]).double()       # [T, D/2]
    rot = torch.polar(torch.ones_like(ang), ang)

    def rope(x):                                   # [T, heads, D]
        z = torch.complex(x[..., : D // 2], x[..., D // 2:]) * rot[:, None, :]
        return torch.cat([z.real, z.imag], -1)

    x = t(w["embed"])[torch.tensor(tokens)]
    streams = [x]
    for l in range(nl):
        p = f"layers.{l}."
        h = F.rms_norm(x, (d,), t(w[p + "attn_norm"]), eps)
        q = rope((h @ t(w[p + "wq"]).T).view(T, H, D))
        k = rope((h @ t(w[p + "wk"]).T).view(T, KVH, D)).repeat_interleave(H // KVH, 1)
        v = (h @ t(w[p + "wv"]).T).view(T, KVH, D).repeat_interleave(H // KVH, 1)
        o = F.scaled_dot_product_attention(q.transpose(0, 1), k.transpose(0, 1), v.transpose(0, 1),
                                           is_causal=True).transpose(0, 1).reshape(T, H * D)
        x = x + o @ t(w[p + "wo"]).T
        h = F.rms_norm(x, (d,), t(w[p + "mlp_norm"]), eps)
        x = x + (F.silu(h @ t(w[p + "w_gate"]).T) * (h @ t(w[p + "w_up"]).T)) @ t(w[p + "w_down"]).T
        streams.append(x)
    logits = F.rms_norm(x, (d,), t(w["final_norm"]), eps) @ t(w["lm_head"]).T
    return [s.numpy() for s in streams], logits.numpy()


def test_aux_taps_enter_layers():
    """Aux tap of layer i = the residual stream entering decoder layer i, i.e. after layers
    0..i-1 and before any norm ("EAGLE-3: Engineering Implementation of LLM Inference
    Acceleration", sections IX.1-IX.3; "Speculative Decoding (EAGLE3) in the vLLM Neuron
    Framework", "Auxiliary Hidden State Extraction": captured before the layer runs).  Checked
    against the stream of an independent torch fp64 model; a tap of layer i's output (the planted
    off-by-one) differs from it, and the oracle's logits match the torch model's."""
    target, _ = _tiny()
    cfg = synth.TINY
    d = cfg["d"]
    prompt = synth.tiny_prompt(0)[:9]
    cache = target.new_cache()
    logits, aux, _, _ = target.forward(prompt, np.arange(9), cache, llama.chain_visible(9))
    streams, ref_logits = _torch_stream(target.w, cfg, prompt)
    assert aux.shape == (9, 3 * d)
    assert np.abs(logits - ref_logits).max() < 1e-10
    for k, layer in enumerate(synth.TINY_AUX_LAYERS):
        tap = aux[:, k * d:(k + 1) * d]
        assert np.abs(tap - streams[layer]).max() < 1e-12
        assert np.abs(tap - streams[layer + 1]).max() > 1e-4       # not the layer's output


# ----------------------------------------------------------------------------- dynamic tree
def _random_expand(seed, V):
    r = np.random.default_rng(seed)

    def expand(t, front):
        return (2.0 * r.standard_normal((len(front), V))).astype(np.float32)
    return expand


@pytest.mark.parametrize("depth,top_k,n_nodes", [(6, 10, 60), (4, 3, 16), (3, 5, 9), (5, 1, 6)])
def test_dynamic_tree_invariants(depth, top_k, n_nodes):
    logs = []
    base = _random_expand(depth * 100 + top_k, 300)

    def expand(t, front):
        out = base(t, front)
        logs.append(out)
        return out

    res = draft_tree.select_tree(expand, depth, top_k, n_nodes)
    parents, dep, cands = res["parents"], res["depth"], res["cands"]
    tree.validate(parents)
    assert len(parents) == n_nodes
    assert dep.max() <= depth and (dep == tree.depths(parents)).all()
    # final set = the top N-1 by (score desc, depth asc, creation asc), brute force
    keys = sorted(((-float(c["score"]), c["depth"], c["creation"]) for c in cands))
    chosen = sorted((-float(cands[i]["score"]), cands[i]["depth"], cands[i]["creation"]) for i in res["chosen"])
    assert chosen == keys[: n_nodes - 1]
    # ancestor-closed; siblings in descending score, parents precede children
    for i in range(1, n_nodes):
        assert res["score"][i] <= res["score"][parents[i]] or parents[i] == 0
    # frontier at each depth = the top_k candidates of the previous depth
    for t in range(2, depth + 1):
        prev = [i for i, c in enumerate(cands) if c["depth"] == t - 1]
        prev.sort(key=lambda i: (-float(cands[i]["score"]), cands[i]["creation"]))
        assert res["frontiers"][t - 1] == prev[:top_k]
    # scores are cumulative log-probabilities: a candidate made from frontier rank r of depth t
    # scores its parent's score plus the log-softmax of that expansion row at its token, summed in
    # fp32 from the root down (the log-softmax itself is pinned in test_oracle_basics)
    from oracle import dsm
    for c in cands:
        path, j = [], c
        while True:
            path.append(j)
            if j["parent"] == -1:
                break
            j = cands[j["parent"]]
        acc = None
        for node in reversed(path):
            row = logs[node["depth"] - 1][node["creation"] // top_k]
            lq = dsm.logq(row)[node["token"]]
            acc = lq if acc is None else np.float32(acc + lq)
        assert np.float32(acc).view(np.uint32) == np.float32(c["score"]).view(np.uint32)
        assert c["token"] in draft_tree.topk_tokens(logs[c["depth"] - 1][c["creation"] // top_k], top_k)
    # each expansion contributes the row's top-k tokens (ties to the lower id)
    first = [c for c in cands if c["depth"] == 1]
    row = logs[0][0]
    assert [c["token"] for c in first] == list(np.lexsort((np.arange(300), -order_key(row)))[:top_k])


@pytest.mark.parametrize("top_k,V", [(3, 50), (7, 300)])   # 1 + k + k^2 <= 64 nodes
def test_full_budget_depth2_is_the_static_expansion(top_k, V):
    """With depth 2 and a node budget that keeps every candidate (N = 1 + k + k^2), the dynamic tree
    is the fixed-branching expansion of "Advanced speculative decoding: tree drafts and EAGLE"
    ("Implementation", build_draft_tree with branching [k, k]): the root's k likeliest draft tokens,
    and under each of them that node's own k likeliest.  The draft here is path-dependent (each
    node's logits are drawn from a seed made of the tokens on its path), so a wrong parent link or
    a child taken from another node's row changes the set of paths."""
    def logits_for(path):
        seed = 7
        for tok in path:
            seed = (seed * 1000003 + tok + 1) % (2 ** 31)
        return (2.0 * np.random.default_rng(seed).standard_normal(V)).astype(np.float32)

    def best(row, k):
        return sorted(range(V), key=lambda i: (-float(row[i]), i))[:k]

    cands = []

    def path_of(cid):
        toks = []
        while cid != -1:
            toks.append(cands[cid]["token"])
            cid = cands[cid]["parent"]
        return tuple(reversed(toks))

    def expand(t, front):
        return np.stack([logits_for(() if f is None else path_of(f)) for f in front])

    res = draft_tree.select_tree(expand, 2, top_k, 1 + top_k + top_k * top_k, cands=cands)
    tokens, parents = res["tokens"], res["parents"]
    got = set()
    for i in range(1, len(tokens)):
        path, j = [], i
        while j != 0:
            path.append(int(tokens[j]))
            j = int(parents[j])
        got.add(tuple(reversed(path)))
    # the static expansion, level by level
    want = set()
    for a in best(logits_for(()), top_k):
        want.add((a,))
        for b in best(logits_for((a,)), top_k):
            want.add((a, b))
    assert len(got) == top_k + top_k * top_k
    assert got == want


def test_top1_tree_is_a_chain():
    res = draft_tree.select_tree(_random_expand(5, 100), 4, 1, 5)
    assert res["parents"].tolist() == [-1, 0, 1, 2, 3]


@pytest.mark.parametrize("depth,top_k,n_nodes", [(6, 10, 60), (4, 3, 16)])
def test_reduced_vocab_equals_target_vocab_with_masked_tokens(depth, top_k, n_nodes):
    """A reduced draft vocabulary (sorted target ids d2t, "EAGLE-3: Engineering Implementation of
    LLM Inference Acceleration", sections VIII.5-VIII.6) is the same tree as the target-vocabulary
    draft whose logits are -inf outside the subset: the scattered draft distribution."""
    V, Vd = 300, 80
    d2t = np.sort(np.random.default_rng(9).choice(V, Vd, replace=False))
    reduced = draft_tree.select_tree(_random_expand(21, Vd), depth, top_k, n_nodes, d2t=d2t)
    draft_rows = _random_expand(21, Vd)

    def expand_full(t, front):
        z = np.full((len(front), V), -np.inf, np.float32)
        z[:, d2t] = draft_rows(t, front)
        return z

    full = draft_tree.select_tree(expand_full, depth, top_k, n_nodes)
    for key in ("tokens", "parents", "depth"):
        assert (reduced[key] == full[key]).all(), key
    assert np.array_equal(reduced["score"].view(np.uint32), full["score"].view(np.uint32))
    assert set(reduced["tokens"][1:].tolist()) <= set(d2t.tolist())


def test_identity_map_is_the_plain_tree():
    V = 200
    plain = draft_tree.select_tree(_random_expand(22, V), 4, 4, 12)
    mapped = draft_tree.select_tree(_random_expand(22, V), 4, 4, 12, d2t=np.arange(V))
    for key in ("tokens", "parents", "depth", "score"):
        assert np.array_equal(plain[key], mapped[key]), key


def test_ttt_attention_without_simulated_steps_is_causal():
    r = np.random.default_rng(6)
    T, Hq, Hkv, D = 9, 4, 2, 16
    q, k, v = r.standard_normal((T, Hq, D)), r.standard_normal((T, Hkv, D)), r.standard_normal((T, Hkv, D))
    got = att.ttt_attention(q, [k], [v], 0.25)
    for h in range(Hq):
        ref = att.causal_attention(q[:, h], k[:, h // 2], v[:, h // 2], 0.25)
        assert np.abs(got[:, h] - ref).max() < 1e-12


def test_ttt_attention_equals_the_diagonal_dot_product_form():
    """The page's check of its forward_ttt ("EAGLE-3: Engineering Implementation of LLM Inference
    Acceleration", section VIII): causal scores against the native keys plus one dot product per
    simulated step at the query's own position, softmax over both."""
    r = np.random.default_rng(7)
    T, Hq, Hkv, D, S = 11, 4, 2, 16, 4
    q = r.standard_normal((T, Hq, D))
    ks = [r.standard_normal((T, Hkv, D)) for _ in range(S)]
    vs = [r.standard_normal((T, Hkv, D)) for _ in range(S)]
    scale = 1 / math.sqrt(D)
    got = att.ttt_attention(q, ks, vs, scale)
    for h in range(Hq):
        g = h // (Hq // Hkv)
        for i in range(T):
            s0 = [float(q[i, h] @ ks[0][j, g]) * scale for j in range(i + 1)]
            sd = [float(q[i, h] @ ks[t][i, g]) * scale for t in range(1, S)]
            w = np.exp(np.array(s0 + sd) - max(s0 + sd))
            w /= w.sum()
            ref = sum(w[j] * vs[0][j, g] for j in range(i + 1))
            ref = ref + sum(w[i + t] * vs[t][i, g] for t in range(1, S))
            assert np.abs(got[i, h] - ref).max() < 1e-12
