"""Compaction of the accepted path's K/V into contiguous cache slots.

Source: "Advanced speculative decoding: tree drafts and EAGLE", section
"Implementation" (the cache update after acceptance: the verify pass already
produced the K/V of the accepted path's nodes at their final positions, so
those rows are copied into the cache rather than recomputed, and every other
node is discarded) and "EAGLE-3: Engineering Implementation of LLM
Inference Acceleration", section XI.4 (the target cache keeps exactly the
committed positions).

Definition used on both sides: for sequence b with prefix length L and path
path[0..n] (path[0] = root), cache slot L + j receives tree row path[j] for
every layer and KV head; slot_map[b, j] = L + j for j <= n and -1 after;
the new prefix length is L + n + 1.  Optional aux rows (the target hidden
states the next draft catch-up consumes) are gathered in path order.

Pinned by: the compacted cache equals the cache that appending the path's
tokens one position at a time would build (tests/test_oracle_basics.py).
"""
import numpy as np


def compact_kv(k_cache, v_cache, tree_k, tree_v, path, accept_len, prefix_len, width,
               aux_tree=None):
    """k_cache/v_cache [layers, B, Hkv, S_max, D]; tree_k/v [layers, B, N, Hkv, D];
    path [B, >= n+1]; accept_len [B]; prefix_len [B]; aux_tree [B, N, A] or None.

    Returns (k_cache', v_cache', slot_map [B, width], prefix_len', aux_out [B, width, A])."""
    k_out, v_out = np.array(k_cache, copy=True), np.array(v_cache, copy=True)
    B = len(prefix_len)
    slot_map = np.full((B, width), -1, dtype=np.int32)
    new_len = np.array(prefix_len, dtype=np.int64, copy=True)
    aux_out = None
    if aux_tree is not None:
        aux_out = np.zeros((B, width, aux_tree.shape[-1]), dtype=aux_tree.dtype)
    for b in range(B):
        L, n = int(prefix_len[b]), int(accept_len[b])
        for j in range(n + 1):
            src = int(path[b][j])
            k_out[:, b, :, L + j, :] = tree_k[:, b, src, :, :]
            v_out[:, b, :, L + j, :] = tree_v[:, b, src, :, :]
            slot_map[b, j] = L + j
            if aux_tree is not None:
                aux_out[b, j] = aux_tree[b, src]
        new_len[b] = L + n + 1
    return k_out, v_out, slot_map, new_len, aux_out
