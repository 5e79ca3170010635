"""Lossless acceptance of a verified draft tree.

Sources:
* "EAGLE-3: Engineering Implementation of LLM Inference Acceleration",
  section III.5 and sections X.3-X.6: drafts are tested in order, each kept
  when a uniform draw falls below p(x) / q(x) (capped at 1); the first
  rejection ends the walk with a replacement drawn from max(0, p - q)
  renormalised; when all drafts are kept, one more token is drawn from the
  last target distribution.  At temperature 0 the rule
  reduces to "accept iff the draft equals the target argmax" (section I).
* "Advanced speculative decoding: tree drafts and EAGLE", section
  "Implementation" (greedy tree walk: from the root, follow the child whose
  token equals the target's argmax) and exercise 2 (trees under sampling:
  try the children of a node in turn, on each rejection replace p by
  norm(max(0, p - q)) with q adjusted to how the candidates were drawn; when
  all are rejected sample from the final residual).
* "Speculative Decoding (EAGLE3) in the vLLM Neuron Framework", section
  "Rejection Sampling": the output row is [accepted drafts..., correction or
  bonus] padded with -1; with a deterministic (greedy) draft q = 1 at the
  drafted token, so the residual is p with that token zeroed.

Readings taken (the pages state the multi-candidate rule only in prose):
* Children of a node are tried in ascending node index.
* argmax uses a total order on fp32 bit patterns (``order_key``) and the
  lowest token id on ties.
* TOPK mode: children were chosen deterministically (top-k of the draft), so
  q is the point mass on each child: accept child x iff U32 * S_cur < 2**32 W_x,
  on rejection S_cur -= W_x and W_x := 0.  P(emit x) = W_x / S.
* SAMPLED mode: children were drawn without replacement from the draft's DSM
  distribution q; accept iff U32 * Wq_x * S_p < 2**32 * Wp_x * S_q, on rejection
  r = max(0, Wp * S_q - Wq * S_p), Wp := r >> max(0, bitlen(max r) - 31),
  S_p := sum Wp, then remove x from q.  If S_q is 0 or max r is 0 the target
  weights are left unchanged.
* Residual / bonus draw: target = (R64 * S) >> 64, the token is the smallest k
  whose running sum of W exceeds target.

Pinned by: exact enumeration of the emitted distribution over all branches
in rational arithmetic on a tiny vocabulary, a chi-square test over many
Philox seeds, the closed form (1 - a**(k+1)) / (1 - a) of the expected
tokens per step for a chain, and the section III.5 worked example
(tests/test_oracle_accept.py).  The greedy walk is pinned by greedy
speculative decoding matching vanilla greedy decoding (tests/test_oracle_model.py).
"""
import numpy as np

from . import dsm
from .philox import SLOT_DRAW, SLOT_RESIDUAL, draw
from .tree import children, validate

GREEDY, TOPK, SAMPLED = 0, 1, 2


def order_key(z):
    """Monotone int64 key of fp32 values: a > b as floats <=> key(a) > key(b)."""
    i = np.asarray(z, dtype=np.float32).view(np.int32).astype(np.int64)
    return np.where(i < 0, i ^ 0x7FFFFFFF, i)


def argmax(z):
    """Index of the largest value; lowest index on ties."""
    return int(np.argmax(order_key(z)))


def _inverse_cdf(W, S, R64):
    """Smallest k with W[0] + ... + W[k] > (R64 * S) >> 64."""
    target = (int(R64) * int(S)) >> 64
    run = 0
    for k, w in enumerate(W):
        run += int(w)
        if run > target:
            return k
    raise AssertionError("inverse CDF ran off the end (S does not match W)")


def _result(path, tokens, next_root):
    return {
        "path": list(path),
        "accept_len": len(path) - 1,
        "emitted": [int(tokens[c]) for c in path[1:]] + [int(next_root)],
        "next_root": int(next_root),
    }


def accept_greedy(tokens, parents, z_target):
    """Greedy longest matching path.  z_target[node] is that node's fp32 logit row."""
    validate(parents)
    node, path = 0, [0]
    while True:
        pred = argmax(z_target[node])
        match = [c for c in children(parents, node) if int(tokens[c]) == pred]
        if not match:
            return _result(path, tokens, pred)
        node = match[0]
        path.append(node)


def accept_topk(tokens, parents, z_target, temperature, seed, step, b):
    """Multi-candidate rejection sampling with deterministically chosen children."""
    validate(parents)
    inv_t = dsm.inv_temperature(temperature)
    node, path = 0, [0]
    while True:
        W, S = dsm.weights(z_target[node], inv_t)
        W = [int(w) for w in W]
        s_cur, moved = S, False
        for s, c in enumerate(children(parents, node)):
            x = int(tokens[c])
            wx = W[x]
            u32, _ = draw(seed, step, b, node, s)
            if u32 * s_cur < (wx << 32):
                node, moved = c, True
                path.append(c)
                break
            s_cur -= wx
            W[x] = 0
        if not moved:
            _, r64 = draw(seed, step, b, node, SLOT_RESIDUAL)
            return _result(path, tokens, _inverse_cdf(W, s_cur, r64))


def accept_sampled(tokens, parents, z_target, z_draft, temperature, seed, step, b):
    """Recursive rejection sampling for children drawn without replacement from q."""
    validate(parents)
    inv_t = dsm.inv_temperature(temperature)
    node, path = 0, [0]
    while True:
        Wp, Sp = dsm.weights(z_target[node], inv_t)
        Wq, Sq = dsm.weights(z_draft[node], inv_t)
        Wp = [int(w) for w in Wp]
        Wq = [int(w) for w in Wq]
        moved = False
        for s, c in enumerate(children(parents, node)):
            x = int(tokens[c])
            u32, _ = draw(seed, step, b, node, s)
            if Sq > 0 and u32 * Wq[x] * Sp < ((Wp[x] * Sq) << 32):
                node, moved = c, True
                path.append(c)
                break
            if Sq > 0:
                r = [max(0, wp * Sq - wq * Sp) for wp, wq in zip(Wp, Wq)]
                mr = max(r)
                if mr > 0:
                    sh = max(0, mr.bit_length() - dsm.FIX_BITS)
                    Wp = [v >> sh for v in r]
                    Sp = sum(Wp)
            Sq -= Wq[x]
            Wq[x] = 0
        if not moved:
            _, r64 = draw(seed, step, b, node, SLOT_RESIDUAL)
            return _result(path, tokens, _inverse_cdf(Wp, Sp, r64))


def draw_children(z_draft_row, temperature, m, seed, step, b, node):
    """Draw m distinct tokens from the draft's DSM distribution (slots 128 + s)."""
    Wq, Sq = dsm.weights(z_draft_row, dsm.inv_temperature(temperature))
    Wq = [int(w) for w in Wq]
    out = []
    for s in range(m):
        if Sq == 0:
            break
        _, r64 = draw(seed, step, b, node, SLOT_DRAW + s)
        k = _inverse_cdf(Wq, Sq, r64)
        out.append(k)
        Sq -= Wq[k]
        Wq[k] = 0
    return out


def accept(mode, tokens, parents, z_target, z_draft=None, temperature=1.0, seed=0, step=0, b=0):
    if mode == GREEDY:
        return accept_greedy(tokens, parents, z_target)
    if mode == TOPK:
        return accept_topk(tokens, parents, z_target, temperature, seed, step, b)
    if mode == SAMPLED:
        return accept_sampled(tokens, parents, z_target, z_draft, temperature, seed, step, b)
    raise ValueError(f"unknown mode {mode}")


def pad(result, width):
    """path / emitted rows padded with -1 to ``width`` (the -1 fill of the Neuron sampler)."""
    path = result["path"] + [-1] * (width - len(result["path"]))
    emitted = result["emitted"] + [-1] * (width - len(result["emitted"]))
    return np.asarray(path[:width], np.int32), np.asarray(emitted[:width], np.int32)
