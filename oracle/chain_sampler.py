"""Chain rejection sampler with Gumbel-max recovered tokens (NEXT-4; no device side yet).

Source: "Speculative Decoding (EAGLE3) in the vLLM Neuron Framework", section "Rejection
Sampling", the CPU sampler.  A request verifies K chained draft tokens against the target's
distributions p_0 .. p_K (p_i at the position of draft i, p_K after the last draft):
* greedy requests keep draft i while it equals argmax p_i;
* random requests keep draft i when a uniform draw u_i <= p_i(d_i) (the draft's own
  probability is taken as 1, since it is not available);
* at the first rejected position i the emitted token is the Gumbel-max draw
  argmax_x adj(x) / E_x with adj = p_i with the draft token's entry set to 0 and E_x
  independent Exp(1) noise, which draws from adj renormalised; greedy requests emit argmax p_i;
* when every draft is kept, a bonus token comes from p_K (greedy: its argmax; random: the
  Gumbel-max draw from p_K).
Output: [K + 1] tokens, the kept drafts then the recovered or bonus token, -1 after.

Readings taken: random numbers are inputs (``uniforms`` [K], ``exp_noise`` [K + 1, V]); argmax
ties go to the lower token id; probabilities are fp64.

Pinned by (tests/test_oracle_chain_sampler.py): the greedy branch equals the first-mismatch rule
of the tree acceptance on a chain; the first emitted token is distributed exactly as p_0 (closed
form over the accept / recover branches); chi-square over many noise draws for the Gumbel-max
draw and for the first emitted token.
"""
import numpy as np


def _argmax(v):
    return int(np.argmax(v))          # numpy returns the first (lowest) index among ties


def gumbel_max(weights, exp_noise):
    """argmax_x weights[x] / exp_noise[x]: a draw from weights renormalised."""
    w = np.asarray(weights, dtype=np.float64)
    return _argmax(np.where(w > 0, w / np.asarray(exp_noise, dtype=np.float64), -1.0))


def chain_verify(target_probs, draft_tokens, greedy, uniforms=None, exp_noise=None):
    """target_probs [K + 1, V] fp64; draft_tokens [K]; returns (output [K + 1], n_accepted)."""
    p = np.asarray(target_probs, dtype=np.float64)
    d = [int(t) for t in draft_tokens]
    K = len(d)
    out = [-1] * (K + 1)
    for i in range(K):
        if greedy:
            keep = d[i] == _argmax(p[i])
        else:
            keep = float(uniforms[i]) <= p[i, d[i]]
        if keep:
            out[i] = d[i]
            continue
        if greedy:
            out[i] = _argmax(p[i])
        else:
            adj = p[i].copy()
            adj[d[i]] = 0.0
            out[i] = gumbel_max(adj, exp_noise[i])
        return out, i
    out[K] = _argmax(p[K]) if greedy else gumbel_max(p[K], exp_noise[K])
    return out, K


# ----------------------------------------------------------------------------------------------
# The specified chain sampler (both sides take every decision identically).
#
# Readings taken, so that the GPU reproduces every token bit for bit from the same logits:
# * probabilities are the deterministic fixed-point softmax of oracle.dsm: W_x, S from the row's
#   logits at temperature T; a random request keeps draft d while u < p(d), i.e. U32 * S < 2**32 * W_d
#   (exact integers), U32 a Philox4x32-10 word;
# * the Gumbel-max noise E_x ~ Exp(1) comes from Philox words w through EXP_NOISE (below), and the
#   recovered / bonus token is the argmax over x of fp32(W_x) / E_x (fp32 round-to-nearest division;
#   ties to the lower id; the rejected draft's W is 0);
# * greedy requests use the argmax of the logits (fp32 total order, ties to the lower id).
# Counters (key = seed): the accept word of draft i of request r is word 0 of
# (ACCEPT_C0, 256 r + i, step low, step high); the noise of token x of row i is word x & 3 of
# (x >> 2, 256 r + i, step low, step high).
#
# EXP_NOISE(w): u = (2 (w >> 9) + 1) * 2**-24 (the top 23 bits of w, centred: u in (0, 1), exact in
# fp32); S = 2 (w >> 9) + 1 = 2**e * m with m in [1, 2), folded into [sqrt(1/2), sqrt(2)) as in
# oracle.dsm.log31; E = fp32(fp32(24 - e) * LN2) - ln m with ln m by the same atanh series.  This is
# -ln u without cancellation near u = 1, and E > 0 for every w.  Quantising u to 2**-23 is the
# noise's counterpart of the fixed point's 2**-31 weights.
# ----------------------------------------------------------------------------------------------
from . import dsm  # noqa: E402
from .accept import argmax as _argmax_f32  # noqa: E402
from .philox import philox4x32_10, philox4x32_10_np, seed_key  # noqa: E402

ACCEPT_C0 = 0x7FFFFFFF
_f32 = np.float32


def exp_noise(w):
    """EXP_NOISE over an array of uint32 words -> fp32 array of E > 0 (Exp(1) draws)."""
    w = np.asarray(w, dtype=np.uint64)
    S = 2 * (w >> np.uint64(9)) + np.uint64(1)                          # odd, < 2**24
    e = (S[..., None] >= (np.uint64(1) << np.arange(1, 25, dtype=np.uint64))).sum(-1).astype(np.int64)
    m = (S.astype(np.float32) * np.ldexp(np.float32(1.0), -e).astype(np.float32)).astype(np.float32)
    fold = m > dsm.SQRT2
    m = np.where(fold, (m * _f32(0.5)).astype(np.float32), m)
    e = e + fold
    s = ((m - _f32(1.0)).astype(np.float32) / (m + _f32(1.0)).astype(np.float32)).astype(np.float32)
    s2 = (s * s).astype(np.float32)
    q = np.full_like(s, dsm.LOG_D[5])
    for j in range(4, -1, -1):
        q = ((q * s2).astype(np.float32) + dsm.LOG_D[j]).astype(np.float32)
    lnm = ((_f32(2.0) * s).astype(np.float32) * q).astype(np.float32)
    k = (24 - e).astype(np.float32)
    return ((k * dsm.LN2).astype(np.float32) - lnm).astype(np.float32)


def _row_words(seed, step, r, i, V):
    """The Philox words of row i of request r for tokens 0..V-1."""
    k0, k1 = seed_key(seed)
    blocks = np.arange((V + 3) // 4, dtype=np.uint64)
    x = philox4x32_10_np(blocks, 256 * r + i, step & 0xFFFFFFFF, (step >> 32) & 0xFFFFFFFF, k0, k1)
    return np.stack(x, -1).reshape(-1)[:V]


def gumbel_argmax_f32(W, E):
    """argmax_x fp32(W_x) / E_x (fp32 division), ties to the lower id."""
    score = (np.asarray(W, dtype=np.float64).astype(np.float32) / np.asarray(E, dtype=np.float32)).astype(np.float32)
    return int(np.argmax(score))


def chain_verify_specified(logits, draft_tokens, greedy, temperature, seed, step, r):
    """One request: logits [K + 1, V] fp32 (row i verifies draft i, row K gives the bonus),
    draft_tokens [K].  Returns (output [K + 1] with -1 after the last emitted token, n_accepted)."""
    z = np.asarray(logits, dtype=np.float32)
    d = [int(t) for t in draft_tokens]
    K = len(d)
    V = z.shape[1]
    out = [-1] * (K + 1)
    inv_t = None if greedy else dsm.inv_temperature(temperature)
    for i in range(K):
        if greedy:
            pred = _argmax_f32(z[i])
            if d[i] == pred:
                out[i] = d[i]
                continue
            out[i] = pred
            return out, i
        W, S = dsm.weights(z[i], inv_t)
        u32 = philox4x32_10((ACCEPT_C0, 256 * r + i, step & 0xFFFFFFFF, (step >> 32) & 0xFFFFFFFF),
                            seed_key(seed))[0]
        if u32 * S < (int(W[d[i]]) << 32):
            out[i] = d[i]
            continue
        adj = W.copy()
        adj[d[i]] = 0
        out[i] = gumbel_argmax_f32(adj, exp_noise(_row_words(seed, step, r, i, V)))
        return out, i
    if greedy:
        out[K] = _argmax_f32(z[K])
    else:
        W, _ = dsm.weights(z[K], inv_t)
        out[K] = gumbel_argmax_f32(W, exp_noise(_row_words(seed, step, r, K, V)))
    return out, K
