"""GPU parity of eagle3_draft_tree.

Replay mode: the GPU returns every draft row's fp32 logits; the oracle's tree selection run on
those logits must reproduce the GPU tree bit for bit (tokens, parents, depth, scores, masks).
Float mode: the oracle draft model (fp64) runs the same rows (the catch-up rows and the frontier
rows of the GPU's tree) and its logits and appended K/V must agree with the GPU within the bf16
tolerance (2e-2 abs + 1e-2 rel).
"""
import numpy as np
import pytest
import torch

import synth
from oracle import draft_tree as odt
from oracle import llama as ollama
from tests._util import close, require_gpu

pytestmark = pytest.mark.gpu


def _setup(seed, B, d, Hq, Hkv, F, V, tc, draft_len, S, D=128, Vd=None):
    """Vd: a reduced draft vocabulary of Vd sorted target ids (d2t); the draft's LM head is then
    those rows of the generated [V, d] head."""
    embed = synth.normal(seed, 500, (V, d), 0.02)
    w = synth.eagle3_weights(seed, d, Hq, Hkv, D, F, V, embed=embed)
    d2t = None
    if Vd is not None:
        d2t = np.sort(synth.rng(seed, 78).choice(V, Vd, replace=False)).astype(np.int32)
        w["lm_head"] = np.ascontiguousarray(w["lm_head"][d2t])
    names = {"w_fc": "fc", "embed": "embed", "input_norm": "input_norm", "hidden_norm": "hidden_norm",
             "w_o": "wo", "post_norm": "post_norm", "w_gate": "w_gate", "w_up": "w_up", "w_down": "w_down",
             "final_norm": "final_norm", "lm_head": "lm_head"}
    gpu_w, f32_w = {}, {}
    for gname, oname in names.items():
        t, f = synth.to_bf16(w[oname])
        gpu_w[gname], f32_w[oname] = t, f
    qkv = np.concatenate([w["wq"], w["wk"], w["wv"]], 0)
    t, f = synth.to_bf16(qkv)
    gpu_w["w_qkv"] = t
    f32_w["wq"], f32_w["wk"], f32_w["wv"] = f[: Hq * D], f[Hq * D: (Hq + Hkv) * D], f[(Hq + Hkv) * D:]
    r = synth.rng(seed, 77)
    tc_max = max(tc)
    aux_t, aux = synth.to_bf16(r.standard_normal((B, tc_max, 3 * d), dtype=np.float32))
    next_tokens = r.integers(0, V, (B, tc_max)).astype(np.int32)
    kc = np.zeros((B, Hkv, S, D), np.float32)
    vc = np.zeros((B, Hkv, S, D), np.float32)
    for b in range(B):
        kc[b, :, : draft_len[b]] = r.standard_normal((Hkv, draft_len[b], D), dtype=np.float32)
        vc[b, :, : draft_len[b]] = r.standard_normal((Hkv, draft_len[b], D), dtype=np.float32)
    kc_t, kc_f = synth.to_bf16(kc)
    vc_t, vc_f = synth.to_bf16(vc)
    return dict(gpu_w=gpu_w, f32_w=f32_w, aux_t=aux_t, aux=aux, next_tokens=next_tokens, kc_t=kc_t, kc=kc_f,
                vc_t=vc_t, vc=vc_f, tc=np.asarray(tc, np.int32), draft_len=np.asarray(draft_len, np.int32), d2t=d2t)


def _run_gpu(s, Hq, F, V, depth, K, N, max_len):
    from eagle_tree_speculative_spec_gb300 import eagle3_draft_tree
    dev = require_gpu()
    B, tc_max = s["next_tokens"].shape
    w = {k: v.to(dev).contiguous() for k, v in s["gpu_w"].items()}
    kc, vc = s["kc_t"].to(dev).clone(), s["vc_t"].to(dev).clone()
    dl = torch.as_tensor(s["draft_len"], device=dev).clone()
    out = dict(tokens=torch.full((B, N), -9, dtype=torch.int32, device=dev),
               parents=torch.full((B, N), -9, dtype=torch.int32, device=dev),
               depth=torch.full((B, N), -9, dtype=torch.int32, device=dev),
               anc=torch.zeros((B, N), dtype=torch.int64, device=dev),
               score=torch.full((B, N), float("nan"), dtype=torch.float32, device=dev))
    d2t = None if s["d2t"] is None else torch.as_tensor(s["d2t"], device=dev)
    Vd = V if d2t is None else d2t.numel()
    dbg = torch.full((depth, K * B, Vd), float("nan"), dtype=torch.float32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    eagle3_draft_tree(w, s["aux_t"].to(dev), torch.as_tensor(s["next_tokens"], device=dev),
                      torch.as_tensor(s["tc"], device=dev), kc, vc, dl, out["tokens"], out["parents"], out["depth"],
                      out["anc"], out["score"], n_heads=Hq, ffn=F, vocab=V, depth=depth, top_k=K,
                      max_draft_len=max_len, dbg_logits=dbg, dev_status=st, d2t=d2t)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    res = {k: v.cpu().numpy() for k, v in out.items()}
    res["dbg"] = dbg.cpu().numpy()
    res["kc"] = kc.float().cpu().numpy()
    res["vc"] = vc.float().cpu().numpy()
    res["draft_len"] = dl.cpu().numpy()
    return res


def _replay(g, b, B, depth, K, N, d2t=None):
    def expand(t, front):
        if t == 1:
            return g["dbg"][0][b: b + 1]
        return np.stack([g["dbg"][t - 1][r * B + b] for r in range(len(front))], 0)
    return odt.select_tree(expand, depth, K, N, d2t=d2t)


def _check_replay(g, s, b, B, depth, K, N):
    ref = _replay(g, b, B, depth, K, N, s["d2t"])
    root = s["next_tokens"][b, s["tc"][b] - 1]
    assert g["tokens"][b, 0] == root
    assert (g["tokens"][b, 1:] == ref["tokens"][1:]).all(), (b, g["tokens"][b], ref["tokens"])
    assert (g["parents"][b] == ref["parents"]).all()
    assert (g["depth"][b] == ref["depth"]).all()
    assert (g["score"][b].view(np.int32) == ref["score"].view(np.int32)).all()
    assert (g["anc"][b].view(np.uint64) == ref["anc"]).all()
    return ref


def _oracle_draft(s, Hq, Hkv, D=128):
    w = {k: v.astype(np.float64) for k, v in s["f32_w"].items()}
    return ollama.Eagle3Draft(w, Hq, Hkv, D)


@pytest.mark.parametrize("cfg", [
    dict(B=3, d=256, Hq=4, Hkv=2, F=512, V=1000, depth=4, K=4, N=12, tc=[1, 2, 1], draft_len=[5, 0, 17], S=64),
    dict(B=2, d=1024, Hq=8, Hkv=2, F=2048, V=8192, depth=6, K=10, N=60, tc=[1, 3], draft_len=[40, 129], S=200),
    dict(B=3, d=256, Hq=4, Hkv=2, F=512, V=1000, depth=4, K=4, N=12, tc=[2, 1, 1], draft_len=[9, 3, 0], S=64,
         Vd=300),
])
def test_draft_tree_replay_and_float(cfg):
    B, d, Hq, Hkv, F, V = cfg["B"], cfg["d"], cfg["Hq"], cfg["Hkv"], cfg["F"], cfg["V"]
    depth, K, N = cfg["depth"], cfg["K"], cfg["N"]
    s = _setup(11, B, d, Hq, Hkv, F, V, cfg["tc"], cfg["draft_len"], cfg["S"], Vd=cfg.get("Vd"))
    max_len = max(cfg["draft_len"])
    g = _run_gpu(s, Hq, F, V, depth, K, N, max_len)
    draft = _oracle_draft(s, Hq, Hkv)
    for b in range(B):
        ref = _check_replay(g, s, b, B, depth, K, N)
        # ---- float parity along the GPU's tree
        L0, tcb = int(s["draft_len"][b]), int(s["tc"][b])
        cache = ollama.KV(1)
        cache.append(0, np.moveaxis(s["kc"][b, :, :L0], 1, 0), np.moveaxis(s["vc"][b, :, :L0], 1, 0))
        gfeat = draft.fuse(s["aux"][b, :tcb])
        a, k, v = draft.layer(s["next_tokens"][b, :tcb], gfeat, np.arange(L0, L0 + tcb), cache,
                              ollama.chain_visible(tcb))
        cache.append(0, k, v)
        assert g["draft_len"][b] == L0 + tcb
        ok, err = close(np.moveaxis(g["kc"][b, :, L0: L0 + tcb], 1, 0), k, 2e-2, 1e-2)
        assert ok, f"appended K b={b} err {err}"
        ok, err = close(np.moveaxis(g["vc"][b, :, L0: L0 + tcb], 1, 0), v, 2e-2, 1e-2)
        assert ok, f"appended V b={b} err {err}"
        log = []

        def gpu_logits(t, front):
            if t == 1:
                return g["dbg"][0][b: b + 1]
            return np.stack([g["dbg"][t - 1][r * B + b] for r in range(len(front))], 0)

        res = odt.draft_tree_for_sequence(draft, cache, a[-1], int(s["next_tokens"][b, tcb - 1]), L0 + tcb,
                                          depth, K, N, logits_log=log, select_logits=gpu_logits, d2t=s["d2t"])
        assert (res["tokens"][1:] == ref["tokens"][1:]).all()
        for t in range(1, depth + 1):
            got = gpu_logits(t, [None] * len(log[t - 1]))
            ok, err = close(got, log[t - 1], 2e-2, 1e-2)
            assert ok, f"logits b={b} depth {t} max err {err}"


@pytest.mark.parametrize("B,Vd", [(1, None), (64, None), (64, 32000)])
def test_draft_tree_full_shapes_replay(B, Vd):
    """Llama-3.1-8B draft head shapes (d 4096, 32/8 heads, FFN 14336, V 128256), depth 6, top-k 10,
    60 nodes, 2048-token draft prefix, one catch-up row: the tree must equal the oracle's
    selection on the GPU's logits for every sequence checked.  Vd: the 32,000-token reduced draft
    vocabulary of the LLaMA-3.1-8B recipe."""
    d, Hq, Hkv, F, V, depth, K, N = 4096, 32, 8, 14336, 128256, 6, 10, 60
    L = 2048
    s = _setup(4, B, d, Hq, Hkv, F, V, [1] * B, [L] * B, L + 64, Vd=Vd)
    g = _run_gpu(s, Hq, F, V, depth, K, N, L)
    rows = range(B) if B <= 4 else [0, 1, 31, 63]
    for b in rows:
        _check_replay(g, s, b, B, depth, K, N)
    assert (g["draft_len"] == L + 1).all()
    # every sequence: a valid tree of 60 nodes, depth <= 6, parents precede children
    assert (g["parents"][:, 0] == -1).all() and (g["depth"] <= depth).all()
    for b in range(B):
        assert all(0 <= g["parents"][b, i] < i for i in range(1, N))


@pytest.mark.parametrize("B", [24, 200])
def test_draft_tree_rows_not_multiple_of_four_floats(B):
    """Logit rows of 1001 floats (not a multiple of 16 bytes, so no shared-memory ring) with more rows
    than the cluster top-k takes: B = 24 (96 frontier rows) runs the register-fed top-k with 256-thread
    CTAs; B = 200 (200 root rows, then 800 frontier rows, more than one wave of those) also runs its
    128-thread variant.  The tree must equal the oracle's selection on the GPU's logits."""
    d, Hq, Hkv, F, V, depth, K, N = 256, 4, 2, 512, 1001, 3, 4, 10
    L = 20
    s = _setup(6, B, d, Hq, Hkv, F, V, [1] * B, [L] * B, L + 32)
    g = _run_gpu(s, Hq, F, V, depth, K, N, L)
    for b in sorted({0, 1, B // 2, B - 1}):
        _check_replay(g, s, b, B, depth, K, N)
    assert (g["draft_len"] == L + 1).all()
