"""Pins of the chain rejection sampler with Gumbel-max recovered tokens (CPU only)."""
import numpy as np
import pytest

import synth
from oracle import accept, chain_sampler as cs


def _probs(r, K, V, sharp=2.0):
    z = sharp * r.standard_normal((K + 1, V))
    e = np.exp(z - z.max(-1, keepdims=True))
    return e / e.sum(-1, keepdims=True)


def test_greedy_equals_the_tree_walk_on_a_chain():
    r = np.random.default_rng(1)
    K, V = 5, 40
    for trial in range(200):
        p = _probs(r, K, V)
        best = p.argmax(-1)
        drafts = [int(best[i]) if r.random() < 0.7 else int(r.integers(V)) for i in range(K)]
        out, n = cs.chain_verify(p, drafts, greedy=True)
        tokens = np.array([0] + drafts)
        res = accept.accept_greedy(tokens, synth.chain_tree(K + 1), np.log(p).astype(np.float32))
        assert n == res["accept_len"]
        assert out[:n] == drafts[:n] and out[n] == res["next_root"]
        assert all(t == -1 for t in out[n + 1:])


def test_first_token_is_exactly_p0():
    """Draft d is kept with probability p0(d); otherwise the token comes from p0 with d removed,
    renormalised: P(x) = p0(d) [x = d] + (1 - p0(d)) p0(x) / (1 - p0(d)) [x != d] = p0(x)."""
    r = np.random.default_rng(2)
    V = 12
    p = _probs(r, 1, V)
    for d in range(V):
        total = np.zeros(V)
        total[d] += p[0, d]
        adj = p[0].copy()
        adj[d] = 0.0
        total += (1.0 - p[0, d]) * adj / adj.sum()
        assert np.abs(total - p[0]).max() < 1e-15


def _chi2_ok(counts, probs, n):
    exp = n * probs
    keep = exp > 5
    stat = float((((counts - exp) ** 2) / np.where(keep, exp, 1.0))[keep].sum())
    dof = int(keep.sum()) - 1
    return stat < dof + 6.0 * np.sqrt(2.0 * dof)       # about 4 sigma above the mean


def test_gumbel_max_draws_from_the_renormalised_weights():
    r = np.random.default_rng(3)
    w = np.array([0.0, 0.05, 0.3, 0.15, 0.0, 0.5])
    n = 40000
    counts = np.zeros(len(w))
    for _ in range(n):
        counts[cs.gumbel_max(w, r.exponential(size=len(w)))] += 1
    assert counts[0] == 0 and counts[4] == 0
    assert _chi2_ok(counts, w / w.sum(), n)


def test_first_emitted_token_follows_p0_under_sampling():
    r = np.random.default_rng(4)
    K, V, n = 3, 8, 30000
    p = _probs(r, K, V, sharp=1.0)
    drafts = [3, 1, 5]
    counts = np.zeros(V)
    lengths = np.zeros(K + 1)
    for _ in range(n):
        out, acc = cs.chain_verify(p, drafts, greedy=False, uniforms=r.random(K),
                                   exp_noise=r.exponential(size=(K + 1, V)))
        counts[out[0]] += 1
        lengths[acc] += 1
    assert _chi2_ok(counts, p[0], n)
    # acceptance lengths: P(n = j) = prod_{i<j} p_i(d_i) * (1 - p_j(d_j)), P(n = K) = prod_i p_i(d_i)
    keep = np.array([p[i, drafts[i]] for i in range(K)])
    want = np.array([np.prod(keep[:j]) * (1 - keep[j]) for j in range(K)] + [np.prod(keep)])
    assert _chi2_ok(lengths, want, n)


def test_output_layout():
    p = np.full((3, 4), 0.25)
    out, n = cs.chain_verify(p, [0, 1], greedy=False, uniforms=[0.1, 0.9], exp_noise=np.ones((3, 4)))
    assert n == 1 and out[0] == 0 and out[1] != 1 and out[2] == -1
    with pytest.raises(IndexError):
        cs.chain_verify(p, [0, 1], greedy=False, uniforms=[0.1], exp_noise=np.ones((3, 4)))
