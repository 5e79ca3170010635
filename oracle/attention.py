"""RoPE and tree-masked verify attention, in fp64.

Sources:
* "EAGLE-3: Engineering Implementation of LLM Inference Acceleration",
  appendix C (``rope``: rotate-half rotary embedding, inv_j = theta**(-2j/D);
  grouped-query attention by repeating each KV head over Hq/Hkv query heads;
  scores scaled by 1/sqrt(D)).  theta = 500000 for the Llama-3 family.
* "Advanced speculative decoding: tree drafts and EAGLE", section
  "Implementation" (``forward_with_mask``: every tree node attends to the
  whole cached prefix plus the tree nodes its mask row allows; positions are
  prefix length + depth).

Readings taken:
* inv_j is computed in fp64 and rounded to fp32; the angle is the fp32
  product fp32(pos) * inv_j; cos and sin are evaluated in fp64 at that fp32
  angle.  Rotation and attention are fp64 from the bf16/fp32 input values.
* The prefix cache holds keys that are already rotated (they were rotated
  when their tree node was verified and then compacted).
* The verify call rotates the tree keys and returns them, so that
  compaction copies rotated keys into the cache.

Pinned by: a chain tree reduces to ordinary causal attention over
prefix + chain (textbook attention written with a dense causal mask), each
node's output equals attention over prefix + its own root-to-node path
computed as a separate sequence (the invariant the tree-drafts page checks to
1.5e-05), RoPE preserving norms and relative-position invariance, and RoPE
equal to the complex rotation of the half-split pairs with inv_j = theta**(-2j/D)
(tests/test_oracle_model.py).
"""
import math

import numpy as np

from .tree import anc_bits, depths

ROPE_THETA = 500000.0


def rope_inv(D, theta=ROPE_THETA):
    j = np.arange(D // 2, dtype=np.float64)
    return (float(theta) ** (-2.0 * j / D)).astype(np.float32)


def rope_angles(pos, D, theta=ROPE_THETA):
    """fp32 angles [len(pos), D/2]."""
    pos = np.asarray(pos, dtype=np.float32).reshape(-1, 1)
    return (pos * rope_inv(D, theta)[None, :]).astype(np.float32)


def rope_apply(x, pos, theta=ROPE_THETA):
    """Rotate-half RoPE.  x: [T, H, D] (any float dtype), pos: [T] -> fp64.

    Element j of the first half and element j of the second half form a pair that is rotated
    by the angle pos * inv_j."""
    x = np.asarray(x, dtype=np.float64)
    half = x.shape[-1] // 2
    ang = rope_angles(pos, 2 * half, theta).astype(np.float64)[:, None, :]    # [T, 1, D/2]
    c, s = np.cos(ang), np.sin(ang)
    lo, hi = x[..., :half], x[..., half:]
    return np.concatenate([lo * c - hi * s, hi * c + lo * s], axis=-1)


def attend(q, keys, values, scale):
    """Softmax attention of one query vector over [S, D] keys/values (fp64).

    Returns (output [D], natural-log LSE of the scaled scores)."""
    s = keys @ q * scale
    m = s.max()
    e = np.exp(s - m)
    den = e.sum()
    return (e @ values) / den, m + math.log(den)


def verify_attention(q, tree_k, tree_v, k_cache, v_cache, parents, prefix_len,
                     theta=ROPE_THETA, sm_scale=None, batch_rows=None):
    """Tree-masked verify attention.

    q        [B, N, Hq, D]      un-rotated queries of the tree nodes
    tree_k   [B, N, Hkv, D]     un-rotated keys of the tree nodes
    tree_v   [B, N, Hkv, D]
    k_cache  [B, Hkv, S_max, D] rotated prefix keys (positions 0..L-1 valid)
    v_cache  [B, Hkv, S_max, D]
    parents  [B, N] int          per-sequence parent arrays
    prefix_len [B] int           L per sequence
    batch_rows                   optional subset of b to compute (others left 0)
    Returns o [B, N, Hq, D], lse [B, N, Hq], k_rot [B, N, Hkv, D] (all fp64).
    """
    B, N, Hq, D = q.shape
    Hkv = tree_k.shape[2]
    rep = Hq // Hkv
    scale = 1.0 / math.sqrt(D) if sm_scale is None else float(sm_scale)
    o = np.zeros((B, N, Hq, D))
    lse = np.zeros((B, N, Hq))
    k_rot = np.zeros((B, N, Hkv, D))
    rows = range(B) if batch_rows is None else batch_rows
    for b in rows:
        L = int(prefix_len[b])
        par = [int(v) for v in parents[b]]
        pos = L + depths(par)
        qr = rope_apply(q[b], pos, theta)                          # [N, Hq, D]
        kr = rope_apply(tree_k[b], pos, theta)                     # [N, Hkv, D]
        k_rot[b] = kr
        vt = np.asarray(tree_v[b], dtype=np.float64)
        bits = anc_bits(par)
        for g in range(Hkv):
            kc = np.asarray(k_cache[b, g, :L], dtype=np.float64)
            vc = np.asarray(v_cache[b, g, :L], dtype=np.float64)
            for i in range(N):
                vis = [j for j in range(N) if (int(bits[i]) >> j) & 1]
                keys = np.concatenate([kc, kr[vis, g]], 0)
                vals = np.concatenate([vc, vt[vis, g]], 0)
                for h in range(g * rep, (g + 1) * rep):
                    o[b, i, h], lse[b, i, h] = attend(qr[i, h], keys, vals, scale)
    return o, lse, k_rot


def causal_attention(q, k, v, scale):
    """Textbook causal attention for one head: q, k, v [T, D] fp64 -> [T, D].

    Used as an independent check: a dense score matrix with a lower-triangular
    mask, softmax per row."""
    T = q.shape[0]
    s = (q @ k.T) * scale
    s = np.where(np.tril(np.ones((T, T), dtype=bool)), s, -np.inf)
    s = s - s.max(-1, keepdims=True)
    e = np.exp(s)
    return (e / e.sum(-1, keepdims=True)) @ v


def ttt_attention(q, ks, vs, scale):
    """Training-time-test attention of one simulated step (NEXT-3's kernel; no device side yet).

    Source: "EAGLE-3: Engineering Implementation of LLM Inference Acceleration", sections VII.5
    (Figure 6's mask: the query at position i attends to the native keys up to i and, of every
    simulated step, to the key at position i alone) and VIII (``forward_ttt``).
    q [T, Hq, D]; ks / vs: lists of [T, Hkv, D], entry 0 the native step's keys (causal), entry
    t >= 1 simulated step t's keys, of which the query at position i sees only position i.
    Written as the definition: attention over all steps' keys concatenated, with that mask built
    explicitly.  Returns [T, Hq, D] fp64.

    Pinned by: with no simulated step it is textbook causal attention, and it equals the
    per-position dot-product form the page uses (the page measures 1.19e-7 in fp32)."""
    q = np.asarray(q, dtype=np.float64)
    T, Hq, D = q.shape
    Hkv = ks[0].shape[1]
    S = len(ks)
    mask = np.zeros((T, S * T), dtype=bool)
    mask[:, :T] = np.tril(np.ones((T, T), dtype=bool))
    for t in range(1, S):
        mask[np.arange(T), t * T + np.arange(T)] = True
    K = np.concatenate([np.asarray(k, dtype=np.float64) for k in ks], 0)      # [S*T, Hkv, D]
    V = np.concatenate([np.asarray(v, dtype=np.float64) for v in vs], 0)
    out = np.empty((T, Hq, D))
    for h in range(Hq):
        g = h // (Hq // Hkv)
        s = (q[:, h] @ K[:, g].T) * scale
        s = np.where(mask, s, -np.inf)
        s = s - s.max(-1, keepdims=True)
        e = np.exp(s)
        out[:, h] = (e / e.sum(-1, keepdims=True)) @ V[:, g]
    return out
