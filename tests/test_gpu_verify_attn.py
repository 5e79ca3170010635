"""GPU parity: eagle3_verify_attn against the fp64 oracle (bf16 tolerance 2e-2 abs / 1e-2 rel)."""
import numpy as np
import pytest
import torch

import synth
from oracle import attention as oatt
from tests._util import close, require_gpu

pytestmark = pytest.mark.gpu
ATOL, RTOL = 2e-2, 1e-2


def _run(inp, max_prefix, num_splits=0, lse=True):
    from eagle_tree_speculative_spec_gb300 import eagle3_verify_attn
    dev = require_gpu()
    q, tk, tv = inp["q"].to(dev), inp["tree_k"].to(dev).clone(), inp["tree_v"].to(dev)
    kc, vc = inp["k_cache"].to(dev), inp["v_cache"].to(dev)
    parents = torch.as_tensor(inp["parents"], device=dev)
    plen = torch.as_tensor(inp["prefix_len"], device=dev)
    out = torch.full(q.shape, float("nan"), dtype=torch.bfloat16, device=dev)
    lse_t = torch.full(q.shape[:3], float("nan"), dtype=torch.float32, device=dev) if lse else None
    eagle3_verify_attn(q, tk, tv, kc, vc, parents, plen, out, max_prefix_len=max_prefix, lse=lse_t,
                       num_splits=num_splits)
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), (lse_t.cpu().numpy() if lse else None), tk.float().cpu().numpy()


def _check(inp, got, rows):
    o, lse, krot = got
    ref_o, ref_lse, ref_k = oatt.verify_attention(inp["q_f32"], inp["tree_k_f32"], inp["tree_v_f32"],
                                                  inp["k_cache_f32"], inp["v_cache_f32"], inp["parents"],
                                                  inp["prefix_len"], batch_rows=rows)
    for b in rows:
        ok, err = close(o[b], ref_o[b], ATOL, RTOL)
        assert ok, f"out b={b} max err {err}"
        ok, err = close(krot[b], ref_k[b], 1e-2, 1e-2)
        assert ok, f"rotated tree_k b={b} max err {err}"
        if lse is not None:
            ok, err = close(lse[b], ref_lse[b], ATOL, RTOL)
            assert ok, f"lse b={b} max err {err}"


@pytest.mark.parametrize("splits", [0, 1, 2, 3])
def test_verify_small_ragged(splits):
    Hq, Hkv, D, N = 32, 8, 128, 60
    lens = [0, 1, 63, 64, 65, 200]
    inp = synth.verify_attn_batch(31, len(lens), N, Hq, Hkv, D, lens, S_max=300)
    got = _run(inp, max(lens), num_splits=splits)
    _check(inp, got, range(len(lens)))


@pytest.mark.parametrize("N", [1, 2, 17, 64])
def test_verify_node_counts(N):
    inp = synth.verify_attn_batch(32, 2, N, 32, 8, 128, [100, 37], S_max=200)
    got = _run(inp, 100)
    _check(inp, got, range(2))


@pytest.mark.parametrize("N", [33, 64])
def test_verify_deep_chain(N):
    """A chain of N nodes has N distinct RoPE positions: the kernel's per-block angle table holds 32,
    the deeper positions take the direct path."""
    inp = synth.verify_attn_batch(34, 2, N, 32, 8, 128, [90, 5], S_max=200)
    inp["parents"] = np.stack([synth.chain_tree(N)] * 2)
    _check(inp, _run(inp, 90), range(2))


def test_verify_other_gqa_ratio():
    inp = synth.verify_attn_batch(33, 2, 40, 16, 2, 128, [130, 77], S_max=200)   # rep 8: 320 rows > 256
    with pytest.raises(Exception):
        _run(inp, 130)
    inp = synth.verify_attn_batch(33, 2, 30, 16, 2, 128, [130, 77], S_max=200)   # rep 8 x 30 nodes = 240 rows
    _check(inp, _run(inp, 130), range(2))


def _full_size_batch(seed, B, N, Hq, Hkv, D, L, S_max, rows):
    """A batch whose sampled rows come from the shared generator (the oracle's inputs) and whose
    other rows are seeded N(0, 1) draws made on the device, each with its own random tree: every
    sequence is distinct, and only the sampled ones are generated on the host."""
    dev = require_gpu()
    q = torch.empty((B, N, Hq, D), dtype=torch.bfloat16, device=dev)
    tk = torch.empty((B, N, Hkv, D), dtype=torch.bfloat16, device=dev)
    tv = torch.empty_like(tk)
    kc = torch.zeros((B, Hkv, S_max, D), dtype=torch.bfloat16, device=dev)
    vc = torch.zeros_like(kc)
    parents = np.empty((B, N), np.int32)
    host = {k: [] for k in ("q", "tree_k", "tree_v", "k_cache", "v_cache", "parents")}
    g = torch.Generator(device=dev)
    for b in range(B):
        if b in rows:
            vals = synth.verify_attn_row(seed, b, N, Hq, Hkv, D, L, S_max)
            for name, dst, x in zip(("q", "tree_k", "tree_v", "k_cache", "v_cache"), (q, tk, tv, kc, vc), vals[:5]):
                t, f = synth.to_bf16(x)
                dst[b].copy_(t)
                host[name].append(f)
            parents[b] = vals[5]
            host["parents"].append(vals[5])
        else:
            parents[b] = synth.random_tree(synth.rng(seed, b), N)
            g.manual_seed(seed * 1000003 + b)
            for dst in (q[b], tk[b], tv[b], kc[b, :, :L], vc[b, :, :L]):
                dst.copy_(torch.randn(dst.shape, generator=g, device=dev))
    sub = {k + "_f32": np.stack(v) for k, v in host.items() if k != "parents"}
    sub["parents"] = np.stack(host["parents"])
    sub["prefix_len"] = np.full(len(rows), L, np.int32)
    dev_inp = dict(q=q, tree_k=tk, tree_v=tv, k_cache=kc, v_cache=vc, parents=parents,
                   prefix_len=np.full(B, L, np.int32))
    return dev_inp, sub


@pytest.mark.parametrize("B", [1, 8, 64])
@pytest.mark.parametrize("L", [512, 4096, 16384])
def test_verify_full_size(B, L):
    """Llama-3.1-8B shapes (32/8 heads, head_dim 128, N = 60) over the verify workload's grid of
    batch sizes and prefix lengths (up to 64 x 16384: 8.6 GB of KV cache); the oracle checks sampled
    sequences."""
    rows = sorted({0, B // 2, B - 1})
    inp, sub = _full_size_batch(3, B, 60, 32, 8, 128, L, L + 64, rows)
    o, lse, krot = _run(inp, L)
    _check(sub, (o[rows], lse[rows], krot[rows]), range(len(rows)))


def _run_rotated(inp, lens, num_splits=0):
    """q and tree_k rotated at prefix_len + depth by the oracle's RoPE, then the qk_rotated call."""
    from eagle_tree_speculative_spec_gb300 import eagle3_verify_attn
    dev = require_gpu()
    par = np.asarray(inp["parents"])
    B = par.shape[0]
    depth = np.zeros(par.shape, np.int64)
    for i in range(1, par.shape[1]):
        depth[:, i] = depth[np.arange(B), par[:, i]] + 1
    pos = np.asarray(inp["prefix_len"])[:, None] + depth                   # [B, N]
    rot = lambda t: np.stack([oatt.rope_apply(t[b], pos[b]) for b in range(B)], 0)
    q_r = torch.as_tensor(rot(inp["q_f32"]), dtype=torch.float32).to(torch.bfloat16)
    k_r = torch.as_tensor(rot(inp["tree_k_f32"]), dtype=torch.float32).to(torch.bfloat16)
    tk = k_r.to(dev).clone()
    out = torch.full(inp["q"].shape, float("nan"), dtype=torch.bfloat16, device=dev)
    eagle3_verify_attn(q_r.to(dev), tk, inp["tree_v"].to(dev), inp["k_cache"].to(dev), inp["v_cache"].to(dev),
                       torch.as_tensor(par, device=dev), torch.as_tensor(inp["prefix_len"], device=dev), out,
                       max_prefix_len=max(lens), num_splits=num_splits, qk_rotated=True)
    torch.cuda.synchronize()
    assert torch.equal(tk.cpu(), k_r)                                        # tree_k is not rewritten
    return out.float().cpu().numpy()


def _check_out(inp, o, rows):
    ref_o, _, _ = oatt.verify_attention(inp["q_f32"], inp["tree_k_f32"], inp["tree_v_f32"], inp["k_cache_f32"],
                                        inp["v_cache_f32"], inp["parents"], inp["prefix_len"], batch_rows=rows)
    for b in rows:
        ok, err = close(o[b], ref_o[b], ATOL, RTOL)
        assert ok, f"out b={b} max err {err}"


@pytest.mark.parametrize("B,L", [(3, 200), (64, 2048)])
def test_verify_qk_rotated(B, L):
    """qk_rotated: q and tree_k arrive rotated at prefix_len + depth (as the RoPE projection leaves
    them); the output equals the oracle's on the un-rotated inputs and tree_k is left as given."""
    lens = [L] * B if B > 8 else [L, 0, L // 3]
    inp = synth.verify_attn_batch(35, B, 60, 32, 8, 128, lens, S_max=max(lens) + 64)
    _check_out(inp, _run_rotated(inp, lens), sorted({0, B // 2, B - 1}))


@pytest.mark.parametrize("splits", [2, 3])
def test_verify_qk_rotated_splits_ragged(splits):
    lens = [0, 1, 64, 65, 200]
    inp = synth.verify_attn_batch(36, len(lens), 60, 32, 8, 128, lens, S_max=300)
    _check_out(inp, _run_rotated(inp, lens, num_splits=splits), range(len(lens)))


def test_verify_qk_rotated_other_ratio():
    """qk_rotated loads Q in boxes of (128 / rep) slots: rep = 8 works, rep = 3 is refused."""
    lens = [130, 77]
    inp = synth.verify_attn_batch(37, 2, 30, 16, 2, 128, lens, S_max=200)    # rep 8, 240 rows
    _check_out(inp, _run_rotated(inp, lens), range(2))
    inp = synth.verify_attn_batch(37, 2, 20, 12, 4, 128, lens, S_max=200)    # rep 3
    with pytest.raises(Exception):
        _run_rotated(inp, lens)
