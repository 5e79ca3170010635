"""Paged KV cache on the GPU: verify attention and compaction through a block table.

Addressing ("Speculative Decoding (EAGLE3) in the vLLM Neuron Framework", "EagleProposer: Draft Model
Management"): position pos of a sequence is slot block_table[pos // block_size] * block_size +
pos % block_size of a pool [n_slots, Hkv, D].  Paging changes where the keys and values are read and
written, not what is computed, so:
* paged verify attention == the oracle on the contiguous cache (bf16 tolerance), and == the same
  kernel on the contiguous cache bit for bit;
* paged compaction, read back through the block table, == oracle.compact on the contiguous cache,
  bit-exact, with slot_map = the pool slots of the new positions.
"""
import numpy as np
import pytest
import torch

import synth
from oracle import attention as oatt
from oracle import compact as ocomp
from oracle import ragged, tree
from tests._util import close, require_gpu

pytestmark = pytest.mark.gpu
ATOL, RTOL = 2e-2, 1e-2


def _block_tables(seed, B, max_blocks, n_pages):
    r = np.random.default_rng(seed)
    return r.permutation(n_pages)[: B * max_blocks].reshape(B, max_blocks).astype(np.int32)


def _pool_from(cache, bt, bs, lens, n_slots):
    """Scatter contiguous caches [B, Hkv, S, D] into a pool [n_slots, Hkv, D] through the tables;
    slots no sequence uses hold N(0, 1) noise (they must never be read)."""
    B, Hkv, S, D = cache.shape
    pool = torch.randn(n_slots, Hkv, D).to(cache.dtype)
    for b in range(B):
        slots = torch.as_tensor(ragged.slot_mapping(bt[b], bs, np.arange(lens[b])))
        pool[slots] = cache[b, :, : lens[b]].transpose(0, 1)
    return pool


@pytest.mark.parametrize("bs", [64, 128, 256])
@pytest.mark.parametrize("qk_rotated", [False, True])
@pytest.mark.parametrize("splits", [0, 3])
def test_paged_verify_attention(bs, qk_rotated, splits):
    from eagle_tree_speculative_spec_gb300 import eagle3_verify_attn
    dev = require_gpu()
    Hq, Hkv, D, N = 32, 8, 128, 60
    lens = [0, 1, 63, 64, 65, 200, 700]
    B, S = len(lens), 768
    inp = synth.verify_attn_batch(51, B, N, Hq, Hkv, D, lens, S_max=S)
    max_blocks = (max(lens) + bs - 1) // bs + 1
    n_pages = B * max_blocks + 3
    bt = _block_tables(bs, B, max_blocks, n_pages)
    kpool = _pool_from(inp["k_cache"], bt, bs, lens, n_pages * bs)
    vpool = _pool_from(inp["v_cache"], bt, bs, lens, n_pages * bs)
    q, tv = inp["q"].to(dev), inp["tree_v"].to(dev)
    par = torch.as_tensor(inp["parents"], device=dev)
    plen = torch.as_tensor(inp["prefix_len"], device=dev)

    def run(paged):
        tk = inp["tree_k"].to(dev).clone()
        out = torch.full(q.shape, float("nan"), dtype=torch.bfloat16, device=dev)
        lse = torch.full(q.shape[:3], float("nan"), dtype=torch.float32, device=dev)
        st = torch.zeros(1, dtype=torch.int32, device=dev)
        if paged:
            eagle3_verify_attn(q, tk, tv, kpool.to(dev), vpool.to(dev), par, plen, out, max_prefix_len=max(lens),
                               lse=lse, num_splits=splits, dev_status=st, qk_rotated=qk_rotated,
                               block_table=torch.as_tensor(bt, device=dev), block_size=bs)
        else:
            eagle3_verify_attn(q, tk, tv, inp["k_cache"].to(dev), inp["v_cache"].to(dev), par, plen, out,
                               max_prefix_len=max(lens), lse=lse, num_splits=splits, dev_status=st,
                               qk_rotated=qk_rotated)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        return out.cpu(), lse.cpu()

    o_p, l_p = run(True)
    o_c, l_c = run(False)
    assert torch.equal(o_p.view(torch.int16), o_c.view(torch.int16))        # bit for bit
    assert torch.equal(l_p, l_c)
    if qk_rotated:
        return                                 # the oracle rotates q / tree_k itself: compare the other path
    ref_o, ref_lse, _ = oatt.verify_attention(inp["q_f32"], inp["tree_k_f32"], inp["tree_v_f32"], inp["k_cache_f32"],
                                              inp["v_cache_f32"], inp["parents"], inp["prefix_len"])
    ok, err = close(o_p.float().numpy(), ref_o, ATOL, RTOL)
    assert ok, err
    ok, err = close(l_p.numpy(), ref_lse, ATOL, RTOL)
    assert ok, err


@pytest.mark.parametrize("bs", [16, 64])
def test_paged_compaction(bs):
    from eagle_tree_speculative_spec_gb300 import eagle3_compact_kv
    dev = require_gpu()
    r = np.random.default_rng(22)
    layers, B, Hkv, D, N, W, A = 3, 5, 2, 128, 60, 7, 96
    L = np.array([0, 3, 20, 41, 57], np.int32)
    max_blocks = (64 + bs - 1) // bs
    n_pages = B * max_blocks + 2
    n_slots = n_pages * bs
    bt = _block_tables(7, B, max_blocks, n_pages)
    S = max_blocks * bs
    kc = torch.randn(layers, B, Hkv, S, D).to(torch.bfloat16)
    vc = torch.randn(layers, B, Hkv, S, D).to(torch.bfloat16)
    kpool = torch.stack([_pool_from(kc[l], bt, bs, [S] * B, n_slots) for l in range(layers)])
    vpool = torch.stack([_pool_from(vc[l], bt, bs, [S] * B, n_slots) for l in range(layers)])
    tk = torch.randn(layers, B, N, Hkv, D).to(torch.bfloat16)
    tv = torch.randn(layers, B, N, Hkv, D).to(torch.bfloat16)
    aux_t = torch.randn(B, N, A).to(torch.bfloat16)
    path, alen = np.full((B, W), -1, np.int32), np.zeros(B, np.int32)
    for b in range(B):
        p = tree.path_to(synth.random_tree(r, N), int(r.integers(0, N)))
        path[b, : len(p)] = p
        alen[b] = len(p) - 1
    g_k, g_v = kpool.to(dev), vpool.to(dev)
    g_L = torch.as_tensor(L, device=dev)
    g_slot = torch.full((B, W), -9, dtype=torch.int32, device=dev)
    g_aux = torch.zeros(B, W, A, dtype=torch.bfloat16, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    eagle3_compact_kv(g_k, g_v, tk.to(dev), tv.to(dev), torch.as_tensor(path, device=dev),
                      torch.as_tensor(alen, device=dev), g_L, g_slot, aux_tree=aux_t.to(dev), aux_out=g_aux,
                      dev_status=st, block_table=torch.as_tensor(bt, device=dev), block_size=bs)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    bits = lambda t: t.view(torch.int16).numpy()
    k2, v2, slot, newL, aux_out = ocomp.compact_kv(bits(kc), bits(vc), bits(tk), bits(tv), path, alen, L, W, bits(aux_t))
    gk, gv = bits(g_k.cpu()), bits(g_v.cpu())
    for l in range(layers):
        for b in range(B):
            view_k = ragged.paged_view(gk[l], bt[b], bs, S).transpose(1, 0, 2)
            view_v = ragged.paged_view(gv[l], bt[b], bs, S).transpose(1, 0, 2)
            assert np.array_equal(view_k, k2[l, b]) and np.array_equal(view_v, v2[l, b])
    for b in range(B):
        n = alen[b]
        want = list(ragged.slot_mapping(bt[b], bs, np.arange(L[b], L[b] + n + 1))) + [-1] * (W - n - 1)
        assert g_slot[b].cpu().tolist() == want
        assert np.array_equal(bits(g_aux.cpu())[b, : n + 1], aux_out[b, : n + 1])
    assert np.array_equal(g_L.cpu().numpy(), newL)


def test_paged_compaction_flags_bad_pages():
    from eagle_tree_speculative_spec_gb300 import eagle3_compact_kv
    dev = require_gpu()
    layers, B, Hkv, D, N, W, bs = 1, 2, 1, 8, 4, 4, 4
    kp = torch.zeros(layers, 8 * bs, Hkv, D, dtype=torch.float32, device=dev)
    vp = torch.zeros_like(kp)
    tk = torch.ones(layers, B, N, Hkv, D, dtype=torch.float32, device=dev)
    tv = torch.ones_like(tk)
    bt = torch.tensor([[0, -1], [3, 5]], dtype=torch.int32, device=dev)      # sequence 0's second page is missing
    path = torch.tensor([[0, 1, 2, 3], [0, 1, -1, -1]], dtype=torch.int32, device=dev)
    alen = torch.tensor([3, 1], dtype=torch.int32, device=dev)
    L = torch.tensor([2, 3], dtype=torch.int32, device=dev)                  # sequence 0 writes 2..5: page 1
    slot = torch.zeros(B, W, dtype=torch.int32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    eagle3_compact_kv(kp, vp, tk, tv, path, alen, L, slot, dev_status=st, block_table=bt, block_size=bs)
    torch.cuda.synchronize()
    assert int(st.item()) & 0x4
    assert L.tolist() == [2, 5]
    assert slot.tolist() == [[-1, -1, -1, -1], [15, 20, -1, -1]]     # positions 3, 4: page 3 offset 3, page 5 offset 0
    assert float(kp[0, :bs].abs().sum()) == 0.0
