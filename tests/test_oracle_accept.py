"""Pins of the oracle's acceptance stage (CPU only).

* Exact enumeration: the probability of every branch of the integer procedure
  is computed in rational arithmetic (the share of the 2**32 U32 values or
  2**64 R64 values that take it); the first emitted token must follow the
  target distribution p = W/S at every node, up to the 2**-32 granularity of
  the uniform draws.  For children drawn from the draft, the enumeration also
  runs over every ordered draw without replacement.
* Chi-square: the oracle functions themselves, fed Philox draws over many
  seeds, emit tokens distributed as p (first and second emission).
* Closed form: a chain whose drafted tokens all have p = a gives
  (1 - a**(k+1)) / (1 - a) emitted tokens per step on average (3.36 at a = 0.8,
  k = 4, the figure printed on the tree-drafts page).
* Worked example of the acceptance probability min(1, p/q): 0.6 / 0.8 = 0.75,
  and an under-confident draft (0.4 vs 0.6) is always accepted.
"""
import math
from fractions import Fraction

import numpy as np
import pytest
from scipy import stats

import synth
from oracle import accept as acc
from oracle import dsm, tree

TWO32, TWO64 = 2**32, 2**64


def _count_u32(a, b):
    """#{U in [0, 2**32): U * a < b}."""
    if b <= 0:
        return 0
    if a == 0:
        return TWO32
    return min(TWO32, -(-b // a))


def _inverse_cdf_probs(W, S):
    """P(token k) of the R64 inverse-CDF draw over integer weights W with sum S."""
    out, run, prev = {}, 0, 0
    for k, w in enumerate(W):
        run += int(w)
        cnt = min(TWO64, -(-(run * TWO64) // S))
        if cnt > prev:
            out[k] = Fraction(cnt - prev, TWO64)
        prev = cnt
    return out


def _node_first_emission_topk(W, S, child_tokens):
    """Exact P(first emitted token) at one node, children fixed (TOPK)."""
    dist, reach, s_cur, Wm = {}, Fraction(1), S, [int(w) for w in W]
    for x in child_tokens:
        pa = Fraction(_count_u32(s_cur, Wm[x] << 32), TWO32)
        dist[x] = dist.get(x, 0) + reach * pa
        reach *= 1 - pa
        s_cur -= Wm[x]
        Wm[x] = 0
    for k, pk in _inverse_cdf_probs(Wm, s_cur).items():
        dist[k] = dist.get(k, 0) + reach * pk
    return dist


def _node_first_emission_sampled(Wp, Sp, Wq, Sq, child_tokens):
    """Exact P(first emitted token) at one node for a given ordered draw of children."""
    dist, reach = {}, Fraction(1)
    Wp, Wq = [int(w) for w in Wp], [int(w) for w in Wq]
    for x in child_tokens:
        pa = Fraction(_count_u32(Wq[x] * Sp, (Wp[x] * Sq) << 32), TWO32) if Sq > 0 else Fraction(0)
        dist[x] = dist.get(x, 0) + reach * pa
        reach *= 1 - pa
        if Sq > 0:
            r = [max(0, a * Sq - b * Sp) for a, b in zip(Wp, Wq)]
            mr = max(r)
            if mr > 0:
                sh = max(0, mr.bit_length() - dsm.FIX_BITS)
                Wp = [v >> sh for v in r]
                Sp = sum(Wp)
        Sq -= Wq[x]
        Wq[x] = 0
    for k, pk in _inverse_cdf_probs(Wp, Sp).items():
        dist[k] = dist.get(k, 0) + reach * pk
    return dist


def _ordered_draws(Wq, Sq, m):
    """All ordered draws of m distinct tokens by repeated inverse-CDF sampling, with probabilities."""
    out = []

    def rec(prefix, W, S, prob):
        if len(prefix) == m or S == 0:
            out.append((tuple(prefix), prob))
            return
        for k, pk in _inverse_cdf_probs(W, S).items():
            W2 = list(W)
            W2[k] = 0
            rec(prefix + [k], W2, S - W[k], prob * pk)

    rec([], [int(w) for w in Wq], Sq, Fraction(1))
    return out


def _rand_logits(r, V, scale=1.5):
    return (scale * r.standard_normal(V)).astype(np.float32)


@pytest.mark.parametrize("seed", range(6))
def test_exact_enumeration_topk(seed):
    r = np.random.default_rng(100 + seed)
    V = 8
    z = _rand_logits(r, V)
    W, S = dsm.weights(z, dsm.inv_temperature(1.0))
    p = [Fraction(int(w), S) for w in W]
    for m in range(0, V):
        kids = [int(x) for x in r.permutation(V)[:m]]
        dist = _node_first_emission_topk(W, S, kids)
        assert sum(dist.values()) == 1
        for y in range(V):
            assert abs(dist.get(y, 0) - p[y]) <= Fraction(m + 1, TWO32)


@pytest.mark.parametrize("seed", range(4))
@pytest.mark.parametrize("temperature", [1.0, 0.6])
def test_exact_enumeration_sampled(seed, temperature):
    r = np.random.default_rng(200 + seed)
    V = 6
    zt = _rand_logits(r, V)
    zd = (zt + r.standard_normal(V)).astype(np.float32) if seed % 2 else _rand_logits(r, V)
    inv_t = dsm.inv_temperature(temperature)
    Wp, Sp = dsm.weights(zt, inv_t)
    Wq, Sq = dsm.weights(zd, inv_t)
    p = [Fraction(int(w), Sp) for w in Wp]
    for m in (1, 2, 3):
        total = {}
        for kids, pk in _ordered_draws(Wq, Sq, m):
            for y, py in _node_first_emission_sampled(Wp, Sp, Wq, Sq, list(kids)).items():
                total[y] = total.get(y, 0) + pk * py
        assert abs(sum(total.values()) - 1) < Fraction(1, 2**50)
        # each accept test is within 2**-32 of its ideal probability; each
        # re-quantised residual moves p by at most V * 2**-31
        bound = Fraction(m + 1, TWO32) + Fraction(m * V, 2**31)
        for y in range(V):
            assert abs(total.get(y, 0) - p[y]) <= bound, (m, y)


def test_exact_enumeration_detects_a_wrong_residual():
    """The enumeration is sharp: a residual that forgets to subtract q is caught."""
    r = np.random.default_rng(7)
    zt, zd = _rand_logits(r, 6), _rand_logits(r, 6)
    Wp, Sp = dsm.weights(zt, dsm.inv_temperature(1.0))
    Wq, Sq = dsm.weights(zd, dsm.inv_temperature(1.0))
    total = {}
    for kids, pk in _ordered_draws(Wq, Sq, 1):
        # planted mistake: resample from p itself instead of norm(max(0, p - q))
        x = kids[0]
        pa = Fraction(_count_u32(int(Wq[x]) * Sp, (int(Wp[x]) * Sq) << 32), TWO32)
        total[x] = total.get(x, 0) + pk * pa
        for k, pr in _inverse_cdf_probs(Wp, Sp).items():
            total[k] = total.get(k, 0) + pk * (1 - pa) * pr
    err = max(abs(total.get(y, 0) - Fraction(int(Wp[y]), Sp)) for y in range(6))
    assert err > 1e-3


def _chi2_ok(counts, probs, n):
    keep = probs * n >= 5
    obs = np.append(counts[keep], counts[~keep].sum())
    exp = np.append(probs[keep] * n, probs[~keep].sum() * n)
    if exp[-1] == 0:
        obs, exp = obs[:-1], exp[:-1]
    return stats.chisquare(obs, exp * obs.sum() / exp.sum()).pvalue


def test_chi_square_first_and_second_emission_topk():
    r = np.random.default_rng(11)
    V, n = 8, 20000
    parents = [-1, 0, 0, 0, 1, 1, 2]
    zt = np.stack([_rand_logits(r, V) for _ in parents])
    tokens = [0, 2, 5, 7, 1, 3, 4]
    first = np.zeros(V)
    second = {c: np.zeros(V) for c in (1, 2)}
    for s in range(n):
        res = acc.accept_topk(tokens, parents, zt, 1.0, seed=12345, step=s, b=3)
        first[res["emitted"][0]] += 1
        if res["accept_len"] >= 1 and res["path"][1] in second:
            second[res["path"][1]][res["emitted"][1]] += 1
    p0 = dsm.probabilities(zt[0], dsm.inv_temperature(1.0))
    assert _chi2_ok(first, p0, n) > 1e-3
    assert 0.5 * np.abs(first / n - p0).sum() < 0.02
    for c, h in second.items():
        pc = dsm.probabilities(zt[c], dsm.inv_temperature(1.0))
        assert _chi2_ok(h, pc, h.sum()) > 1e-3


def test_chi_square_sampled_children():
    r = np.random.default_rng(12)
    V, n = 8, 12000
    parents = [-1, 0, 0, 0]
    zt = np.stack([_rand_logits(r, V) for _ in parents])
    zd = np.stack([(zt[i] + r.standard_normal(V)).astype(np.float32) for i in range(4)])
    first = np.zeros(V)
    for s in range(n):
        kids = acc.draw_children(zd[0], 1.0, 3, seed=77, step=s, b=0, node=0)
        tokens = [0] + kids
        res = acc.accept_sampled(tokens, parents, zt, zd, 1.0, seed=77, step=s, b=0)
        first[res["emitted"][0]] += 1
    p0 = dsm.probabilities(zt[0], dsm.inv_temperature(1.0))
    assert _chi2_ok(first, p0, n) > 1e-3
    assert 0.5 * np.abs(first / n - p0).sum() < 0.025


def test_closed_form_chain_expected_tokens():
    V, k, alpha = 8, 4, 0.8
    z = np.full(V, math.log((1 - alpha) / (V - 1)), np.float32)
    z[5] = math.log(alpha)
    zt = np.stack([z] * (k + 1))
    parents = synth.chain_tree(k + 1).tolist()
    tokens = [0] + [5] * k
    W, S = dsm.weights(z, dsm.inv_temperature(1.0))
    a = Fraction(_count_u32(S, int(W[5]) << 32), TWO32)
    exact = sum(a**j for j in range(k + 1))
    assert abs(float(exact) - (1 - alpha ** (k + 1)) / (1 - alpha)) < 1e-6
    assert abs((1 - alpha ** (k + 1)) / (1 - alpha) - 3.36) < 0.005
    n = 20000
    emitted = [len(acc.accept_topk(tokens, parents, zt, 1.0, 9, s, 0)["emitted"]) for s in range(n)]
    mean, sd = np.mean(emitted), np.std(emitted)
    assert abs(mean - float(exact)) < 4 * sd / math.sqrt(n)


def test_worked_example_acceptance_probability():
    zt = np.log(np.array([0.6, 0.4])).astype(np.float32)
    for q0, want in ((0.8, 0.75), (0.4, 1.0)):
        zd = np.log(np.array([q0, 1 - q0])).astype(np.float32)
        Wp, Sp = dsm.weights(zt, dsm.inv_temperature(1.0))
        Wq, Sq = dsm.weights(zd, dsm.inv_temperature(1.0))
        pa = _count_u32(int(Wq[0]) * Sp, (int(Wp[0]) * Sq) << 32) / TWO32
        assert abs(pa - want) < 1e-6


def test_greedy_chain_is_first_mismatch():
    r = np.random.default_rng(13)
    V, K = 50, 5
    for _ in range(50):
        z = (3 * r.standard_normal((K + 1, V))).astype(np.float32)
        pred = [acc.argmax(z[i]) for i in range(K + 1)]
        drafts = [pred[i] if r.random() < 0.7 else int((pred[i] + 1) % V) for i in range(K)]
        tokens = [0] + drafts
        res = acc.accept_greedy(tokens, synth.chain_tree(K + 1), z)
        match = [drafts[i] == pred[i] for i in range(K)]
        n = match.index(False) if False in match else K
        assert res["accept_len"] == n
        assert res["emitted"] == drafts[:n] + [pred[n]]
        path, emitted = acc.pad(res, K + 1)
        assert (emitted[n + 1:] == -1).all() and (path[n + 1:] == -1).all()


def test_greedy_tree_walk_and_ties():
    parents = [-1, 0, 0, 1, 2, 2]
    tokens = [9, 3, 4, 1, 2, 2]
    V = 6
    z = np.zeros((6, V), np.float32)
    z[0, 4] = 1.0         # root predicts 4 -> node 2
    z[2, 2] = 1.0         # node 2 predicts 2 -> nodes 4 and 5 both match: lowest index 4
    z[4, :] = 0.5         # tie across the row: lowest token id 0
    res = acc.accept_greedy(tokens, parents, z)
    assert res["path"] == [0, 2, 4] and res["emitted"] == [4, 2, 0] and res["next_root"] == 0
    assert acc.argmax(np.float32([-0.0, 0.0])) == 1      # +0 orders above -0
    assert acc.argmax(np.float32([1.0, np.inf, np.inf])) == 1


def test_topk_leaf_root_is_bonus_from_p():
    # a root with no children emits a bonus token drawn from p
    r = np.random.default_rng(14)
    z = _rand_logits(r, 8)[None]
    W, S = dsm.weights(z[0], dsm.inv_temperature(1.0))
    dist = _node_first_emission_topk(W, S, [])
    for y in range(8):
        assert abs(dist.get(y, 0) - Fraction(int(W[y]), S)) <= Fraction(1, TWO32)
    res = acc.accept_topk([0], [-1], z, 1.0, 1, 0, 0)
    assert res["accept_len"] == 0 and len(res["emitted"]) == 1


def test_c2_shapes_run():
    """The oracle walks one full-size (V = 128256, N = 60) sequence in all three modes."""
    zt, zd, parents = synth.accept_row(1, 0, 60, 128256)
    tokens = synth.tokens_top_draft(zd, parents)
    g = acc.accept_greedy(tokens, parents, zt)
    t = acc.accept_topk(tokens, parents, zt, 1.0, 1, 0, 0)
    tree.validate(parents)
    for res in (g, t):
        assert 1 <= len(res["emitted"]) <= 7
        assert all(parents[res["path"][i + 1]] == res["path"][i] for i in range(res["accept_len"]))
