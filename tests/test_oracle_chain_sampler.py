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


# ----------------------------------------------------------------------------- the specified sampler
def _noise_excess(fn, w):
    """max |fn(w) - (-ln u)| / bound with u = (2 (w >> 9) + 1) / 2^24; the bound: the atanh series
    and its fp32 steps are within a few ulp of ln m, and the final fp32 subtraction rounds by half
    an ulp of E, so 4 * 2^-24 relative (plus 2^-30 absolute for E near 0) covers them."""
    u = (2 * (np.asarray(w, np.uint64) >> np.uint64(9)) + 1).astype(np.float64) / 2.0**24
    ref = -np.log(u)
    return float((np.abs(fn(w).astype(np.float64) - ref) / (4 * 2.0**-24 * ref + 2.0**-30)).max())


def test_exp_noise_is_minus_log_u():
    r = np.random.default_rng(7)
    w = np.concatenate([r.integers(0, 2**32, 200000, dtype=np.uint64),
                        np.array([0, 1, 511, 512, 2**31 - 1, 2**31, 2**32 - 513, 2**32 - 512, 2**32 - 1],
                                 dtype=np.uint64)])
    E = cs.exp_noise(w)
    assert (E > 0).all()
    assert _noise_excess(cs.exp_noise, w) <= 1.0
    # planted mistakes: the exponent off by one, the fold skipped, the sign of the series flipped
    planted = [lambda x: (cs.exp_noise(x) + np.float32(np.log(2.0))).astype(np.float32),
               lambda x: np.abs((-np.log1p(-(2 * (np.asarray(x, np.uint64) >> np.uint64(9)) + 1)
                                           .astype(np.float64) / 2.0**24)).astype(np.float32)),
               lambda x: (2 * cs.exp_noise(x)).astype(np.float32)]
    for bad in planted:
        assert _noise_excess(bad, w) > 1.0


def test_exp_noise_is_exponential():
    r = np.random.default_rng(8)
    E = cs.exp_noise(r.integers(0, 2**32, 400000, dtype=np.uint64)).astype(np.float64)
    n = len(E)
    assert abs(E.mean() - 1.0) < 5 / np.sqrt(n)
    edges = np.array([0.0, 0.1, 0.25, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, np.inf])
    counts = np.histogram(E, edges)[0]
    probs = np.exp(-edges[:-1]) - np.exp(-edges[1:])
    assert _chi2_ok(counts, probs, n)


def test_specified_gumbel_max_draws_from_the_weights():
    """argmax fp32(W)/E over Philox-driven noise draws x with probability W_x / S."""
    W = np.array([0, 3 * 2**28, 2**31, 0, 2**29, 7 * 2**27, 1, 2**30], dtype=np.int64)
    n = 20000
    counts = np.zeros(len(W))
    for s in range(n):
        counts[cs.gumbel_argmax_f32(W, cs.exp_noise(cs._row_words(s, 0, 0, 0, len(W))))] += 1
    assert counts[0] == 0 and counts[3] == 0
    assert _chi2_ok(counts, W / W.sum(), n)


def test_specified_greedy_equals_the_tree_walk_on_a_chain():
    r = np.random.default_rng(9)
    K, V = 5, 40
    for _ in range(100):
        z = (3.0 * r.standard_normal((K + 1, V))).astype(np.float32)
        best = z.argmax(-1)
        drafts = [int(best[i]) if r.random() < 0.7 else int(r.integers(V)) for i in range(K)]
        out, n = cs.chain_verify_specified(z, drafts, True, 1.0, 0, 0, 0)
        res = accept.accept_greedy(np.array([0] + drafts), synth.chain_tree(K + 1), z)
        assert n == res["accept_len"] and out[:n] == drafts[:n] and out[n] == res["next_root"]
        assert all(t == -1 for t in out[n + 1:])


def test_specified_sampler_emits_p0_and_accepts_with_p():
    """Random requests: the first emitted token follows p0 = DSM(z0 / T) exactly in law, and the
    acceptance lengths follow the product of p_i(d_i) (chi-square over Philox seeds)."""
    from oracle import dsm
    r = np.random.default_rng(10)
    K, V, n, T = 3, 8, 6000, 0.8
    z = (1.5 * r.standard_normal((K + 1, V))).astype(np.float32)
    drafts = [int(np.argsort(-z[i])[1]) for i in range(K)]       # plausible but not the argmax
    p = np.stack([dsm.probabilities(z[i], dsm.inv_temperature(T)) for i in range(K + 1)])
    counts, lengths = np.zeros(V), np.zeros(K + 1)
    for s in range(n):
        out, acc = cs.chain_verify_specified(z, drafts, False, T, seed=1000 + s, step=s, r=s % 5)
        counts[out[0]] += 1
        lengths[acc] += 1
    assert _chi2_ok(counts, p[0], n)
    keep = np.array([p[i, drafts[i]] for i in range(K)])
    want = np.array([np.prod(keep[:j]) * (1 - keep[j]) for j in range(K)] + [np.prod(keep)])
    assert _chi2_ok(lengths, want, n)
