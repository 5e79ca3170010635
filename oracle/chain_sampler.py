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
