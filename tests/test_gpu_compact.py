"""GPU parity: eagle3_compact_kv against the oracle, bit-exact."""
import numpy as np
import pytest
import torch

import synth
from oracle import compact as ocomp
from oracle import tree
from tests._util import require_gpu

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("aux", [False, True])
def test_compact_matches_oracle(dtype, aux):
    from eagle_tree_speculative_spec_gb300 import eagle3_compact_kv
    dev = require_gpu()
    r = np.random.default_rng(21)
    layers, B, Hkv, S, D, N, W, A = 3, 5, 2, 48, 128, 60, 7, 96
    kc = torch.randn(layers, B, Hkv, S, D).to(dtype)
    vc = torch.randn(layers, B, Hkv, S, D).to(dtype)
    tk = torch.randn(layers, B, N, Hkv, D).to(dtype)
    tv = torch.randn(layers, B, N, Hkv, D).to(dtype)
    aux_t = torch.randn(B, N, A).to(dtype) if aux else None
    L = np.array([0, 3, 20, 41, 47 - 6])
    path, alen = np.full((B, W), -1, np.int32), np.zeros(B, np.int32)
    for b in range(B):
        parents = synth.random_tree(r, N)
        p = tree.path_to(parents, int(r.integers(0, N)))
        path[b, : len(p)] = p
        alen[b] = len(p) - 1
    gpu = lambda t: t.to(dev).contiguous()
    g_kc, g_vc, g_tk, g_tv = gpu(kc), gpu(vc), gpu(tk), gpu(tv)
    g_path = torch.as_tensor(path, device=dev)
    g_alen = torch.as_tensor(alen, device=dev)
    g_L = torch.as_tensor(L.astype(np.int32), device=dev)
    g_slot = torch.full((B, W), -9, dtype=torch.int32, device=dev)
    g_aux_out = torch.zeros(B, W, A, dtype=dtype, device=dev) if aux else None
    eagle3_compact_kv(g_kc, g_vc, g_tk, g_tv, g_path, g_alen, g_L, g_slot,
                      aux_tree=gpu(aux_t) if aux else None, aux_out=g_aux_out)
    torch.cuda.synchronize()
    as_np = lambda t: t.view(torch.int16).numpy() if dtype == torch.bfloat16 else t.view(torch.int32).numpy()
    k2, v2, slot, newL, aux_out = ocomp.compact_kv(as_np(kc), as_np(vc), as_np(tk), as_np(tv), path, alen, L, W,
                                                   as_np(aux_t) if aux else None)
    assert (as_np(g_kc.cpu()) == k2).all()
    assert (as_np(g_vc.cpu()) == v2).all()
    assert (g_slot.cpu().numpy() == slot).all()
    assert (g_L.cpu().numpy() == newL).all()
    if aux:
        got = as_np(g_aux_out.cpu())
        for b in range(B):
            assert (got[b, : alen[b] + 1] == aux_out[b, : alen[b] + 1]).all()


def test_compact_capacity_flag():
    from eagle_tree_speculative_spec_gb300 import eagle3_compact_kv
    dev = require_gpu()
    layers, B, Hkv, S, D, N, W = 1, 2, 1, 10, 8, 4, 4
    kc = torch.zeros(layers, B, Hkv, S, D, dtype=torch.float32, device=dev)
    vc = torch.zeros_like(kc)
    tk = torch.ones(layers, B, N, Hkv, D, dtype=torch.float32, device=dev)
    tv = torch.ones_like(tk)
    path = torch.tensor([[0, 1, 2, 3], [0, 1, -1, -1]], dtype=torch.int32, device=dev)
    alen = torch.tensor([3, 1], dtype=torch.int32, device=dev)
    L = torch.tensor([8, 2], dtype=torch.int32, device=dev)       # row 0: 8 + 4 > 10
    slot = torch.zeros(B, W, dtype=torch.int32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    eagle3_compact_kv(kc, vc, tk, tv, path, alen, L, slot, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & 0x4
    assert L.tolist() == [8, 4]
    assert slot.tolist() == [[-1, -1, -1, -1], [2, 3, -1, -1]]
    assert float(kc[0, 0].abs().sum()) == 0.0 and float(kc[0, 1, 0, 2:4].sum()) == 16.0
