"""GPU parity: eagle3_accept against the oracle, bit-exact (tokens, paths, lengths)."""
import numpy as np
import pytest
import torch

import synth
from oracle import accept as oacc
from tests._util import require_gpu

pytestmark = pytest.mark.gpu


def _run(mode, zt, zd, tokens, parents, W, temperature=1.0, seed=1, step=0, dev_status=None):
    from eagle_tree_speculative_spec_gb300 import eagle3_accept
    dev = require_gpu()
    B, N, V = zt.shape
    t = lambda a, dt: torch.as_tensor(np.ascontiguousarray(a), dtype=dt, device=dev)
    out = dict(accept_len=torch.full((B,), -7, dtype=torch.int32, device=dev),
               path=torch.full((B, W), -7, dtype=torch.int32, device=dev),
               emitted=torch.full((B, W), -7, dtype=torch.int32, device=dev),
               next_root=torch.full((B,), -7, dtype=torch.int32, device=dev))
    eagle3_accept(mode, t(zt, torch.float32), t(tokens, torch.int32), t(parents, torch.int32),
                  out["accept_len"], out["path"], out["emitted"], out["next_root"],
                  draft_logits=None if zd is None else t(zd, torch.float32), temperature=temperature,
                  seed=seed, step=step, dev_status=dev_status)
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in out.items()}


def _expect(mode, zt, zd, tokens, parents, W, b, temperature, seed, step):
    res = oacc.accept(mode, tokens[b], parents[b], zt[b], None if zd is None else zd[b],
                      temperature, seed, step, b)
    path, emitted = oacc.pad(res, W)
    return res, path, emitted


def _compare(got, mode, zt, zd, tokens, parents, W, rows, temperature=1.0, seed=1, step=0):
    for b in rows:
        res, path, emitted = _expect(mode, zt, zd, tokens, parents, W, b, temperature, seed, step)
        assert got["accept_len"][b] == res["accept_len"], (b, got["accept_len"][b], res)
        assert (got["path"][b] == path).all(), (b, got["path"][b], path)
        assert (got["emitted"][b] == emitted).all(), (b, got["emitted"][b], emitted)
        assert got["next_root"][b] == res["next_root"]


@pytest.mark.parametrize("V", [1000, 1001, 4099])
@pytest.mark.parametrize("mode", [oacc.GREEDY, oacc.TOPK, oacc.SAMPLED])
def test_accept_small(mode, V):
    B, N, W = 6, 60, 8
    zt, zd, parents, tokens = synth.accept_batch(11, B, N, V, sampled=(mode == oacc.SAMPLED))
    got = _run(mode, zt, zd if mode == oacc.SAMPLED else None, tokens, parents, W)
    _compare(got, mode, zt, zd, tokens, parents, W, range(B))


@pytest.mark.parametrize("temperature", [0.5, 2.0])
@pytest.mark.parametrize("mode", [oacc.TOPK, oacc.SAMPLED])
def test_accept_temperature_and_steps(mode, temperature):
    B, N, V, W = 4, 30, 2000, 8
    zt, zd, parents, tokens = synth.accept_batch(12, B, N, V, sampled=(mode == oacc.SAMPLED))
    for step in (0, 1, 2**33 + 5):
        got = _run(mode, zt, zd if mode == oacc.SAMPLED else None, tokens, parents, W,
                   temperature=temperature, seed=2**40 + 3, step=step)
        _compare(got, mode, zt, zd, tokens, parents, W, range(B), temperature, 2**40 + 3, step)


def test_accept_chain_and_root_only():
    V, W = 500, 6
    r = np.random.default_rng(3)
    for N in (1, 2, 5):
        parents = np.tile(synth.chain_tree(N), (3, 1))
        zt = (3 * r.standard_normal((3, N, V))).astype(np.float32)
        tokens = np.zeros((3, N), np.int32)
        for b in range(3):
            for i in range(1, N):   # make the chain fully greedy-accepted in row 0
                tokens[b, i] = int(np.argmax(zt[b, i - 1])) if b == 0 else int(r.integers(0, V))
        for mode in (oacc.GREEDY, oacc.TOPK):
            got = _run(mode, zt, None, tokens, parents, W)
            _compare(got, mode, zt, None, tokens, parents, W, range(3))
        assert _run(oacc.GREEDY, zt, None, tokens, parents, W)["accept_len"][0] == N - 1


def test_accept_bad_tree_is_flagged():
    V, N, W = 300, 6, 7
    zt, zd, parents, tokens = synth.accept_batch(13, 3, N, V)
    parents[1, 3] = 5          # parent index after the child
    tokens[2, 2] = V + 4       # token out of range
    status = torch.zeros(1, dtype=torch.int32, device=require_gpu())
    got = _run(oacc.GREEDY, zt, None, tokens, parents, W, dev_status=status)
    st = int(status.item())
    assert st & 0x1 and st & 0x2
    for b in (1, 2):
        assert got["accept_len"][b] == 0 and got["next_root"][b] == -1
        assert got["path"][b].tolist() == [0] + [-1] * (W - 1)
    _compare(got, oacc.GREEDY, zt, None, tokens, parents, W, [0])


def test_accept_path_truncation_flag():
    V, N = 200, 6
    r = np.random.default_rng(4)
    zt = (3 * r.standard_normal((1, N, V))).astype(np.float32)
    parents = synth.chain_tree(N)[None]
    tokens = np.zeros((1, N), np.int32)
    for i in range(1, N):
        tokens[0, i] = int(np.argmax(zt[0, i - 1]))
    status = torch.zeros(1, dtype=torch.int32, device=require_gpu())
    got = _run(oacc.GREEDY, zt, None, tokens, parents, 3, dev_status=status)
    assert int(status.item()) & 0x10
    assert got["path"][0].tolist() == [0, 1, 2]


@pytest.mark.parametrize("mode", [oacc.GREEDY, oacc.TOPK, oacc.SAMPLED])
def test_accept_full_size(mode):
    """Acceptance on synthetic logits at full size: B = 64, N = 60, V = 128256; the oracle
    checks a sample of the sequences (every launch covers all 64)."""
    B, N, V, W = 64, 60, 128256, 7
    zt, zd, parents, tokens = synth.accept_batch(1, B, N, V, sampled=(mode == oacc.SAMPLED))
    got = _run(mode, zt, zd if mode == oacc.SAMPLED else None, tokens, parents, W, seed=1)
    rows = [0, 1, 17, 31, 42, 63] if mode == oacc.SAMPLED else list(range(0, 64, 4)) + [63]
    _compare(got, mode, zt, zd, tokens, parents, W, rows, seed=1)
    assert (got["accept_len"] >= 0).all() and (got["accept_len"] <= 6).all()


@pytest.mark.parametrize("mode", [oacc.TOPK, oacc.SAMPLED])
def test_accept_device_step_counter(mode):
    """A device step counter replaces the host `step` and advances by one per call, so a captured graph
    draws fresh numbers on every replay: three replays give the oracle's results for steps s, s+1, s+2."""
    from eagle_tree_speculative_spec_gb300 import eagle3_accept
    dev = require_gpu()
    B, N, V, W = 4, 30, 2000, 8
    zt, zd, parents, tokens = synth.accept_batch(13, B, N, V, sampled=(mode == oacc.SAMPLED))
    t = lambda a, dt: torch.as_tensor(np.ascontiguousarray(a), dtype=dt, device=dev)
    zt_d, tok_d, par_d = t(zt, torch.float32), t(tokens, torch.int32), t(parents, torch.int32)
    zd_d = t(zd, torch.float32) if mode == oacc.SAMPLED else None
    s0 = 2**32 - 2                                  # the carry into the counter's high word is exercised
    counter = torch.tensor([s0], dtype=torch.int64, device=dev)
    out = dict(accept_len=torch.empty(B, dtype=torch.int32, device=dev),
               path=torch.empty(B, W, dtype=torch.int32, device=dev),
               emitted=torch.empty(B, W, dtype=torch.int32, device=dev),
               next_root=torch.empty(B, dtype=torch.int32, device=dev))
    stream = torch.cuda.Stream(device=dev)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        eagle3_accept(mode, zt_d, tok_d, par_d, out["accept_len"], out["path"], out["emitted"], out["next_root"],
                      draft_logits=zd_d, seed=3, step=12345, step_counter=counter,
                      stream=torch.cuda.current_stream())
    for r in range(3):
        g.replay()
        torch.cuda.synchronize()
        got = {k: v.cpu().numpy() for k, v in out.items()}
        _compare(got, mode, zt, zd, tokens, parents, W, range(B), seed=3, step=s0 + r)
    assert int(counter.item()) == s0 + 3


def _chi2_pvalue(hist, p):
    """Chi-square p-value of a histogram against probabilities p (cells with p = 0 must be empty)."""
    from scipy import stats
    assert hist[p == 0].sum() == 0
    keep = p > 0
    exp = p[keep] * hist.sum()
    return stats.chisquare(hist[keep], exp).pvalue


@pytest.mark.parametrize("mode", [oacc.TOPK, oacc.SAMPLED])
def test_accept_emits_the_target_distribution(mode):
    """Losslessness through the C ABI ("Speculative Decoding (EAGLE3) in the vLLM Neuron Framework",
    "Rejection Sampling"): 16384 sequences share one small tree and its logits and differ only in
    their Philox streams (the sequence index), so one call draws 16384 independent acceptances.  The
    first emitted token follows the target's p at the root (chi-square p-value > 1e-3, total
    variation < 0.02); for TOPK the token emitted after an accepted child follows that child's p.
    SAMPLED children are drawn from the draft's distribution by the oracle's draw."""
    from oracle import dsm
    r = np.random.default_rng(21)
    V, B, W, seed = 8, 16384, 4, 4242
    parents1 = [-1, 0, 0, 0, 1, 1, 2] if mode == oacc.TOPK else [-1, 0, 0, 0]
    N = len(parents1)
    zt1 = (1.5 * r.standard_normal((N, V))).astype(np.float32)
    if mode == oacc.TOPK:
        # deterministic top-k children: the root's three likeliest tokens, then each child's likeliest
        top = lambda z, k: [int(x) for x in np.argsort(-z, kind="stable")[:k]]
        tokens1 = [0] + top(zt1[0], 3) + top(zt1[1], 2) + top(zt1[2], 1)
    zd1 = (zt1 + r.standard_normal((N, V))).astype(np.float32)
    zt = np.ascontiguousarray(np.broadcast_to(zt1, (B, N, V)))
    zd = np.ascontiguousarray(np.broadcast_to(zd1, (B, N, V))) if mode == oacc.SAMPLED else None
    parents = np.tile(np.asarray(parents1, np.int32), (B, 1))
    if mode == oacc.TOPK:
        tokens = np.tile(np.asarray(tokens1, np.int32), (B, 1))
    else:
        tokens = np.zeros((B, N), np.int32)
        for b in range(B):
            kids = oacc.draw_children(zd1[0], 1.0, N - 1, seed=seed, step=0, b=b, node=0)
            assert len(kids) == N - 1
            tokens[b, 1:] = kids
    got = _run(mode, zt, zd, tokens, parents, W, seed=seed, step=0)
    _compare(got, mode, zt, zd, tokens, parents, W, [0, 1, B - 1], seed=seed)
    inv_t = dsm.inv_temperature(1.0)
    first = np.bincount(got["emitted"][:, 0], minlength=V).astype(np.float64)
    p0 = np.asarray(dsm.probabilities(zt1[0], inv_t), np.float64)
    assert _chi2_pvalue(first, p0) > 1e-3
    assert 0.5 * np.abs(first / B - p0).sum() < 0.02
    if mode == oacc.TOPK:
        for c in (1, 2):   # children of the root that have children of their own
            sel = (got["accept_len"] >= 1) & (got["path"][:, 1] == c)
            assert sel.sum() > 500
            h = np.bincount(got["emitted"][sel, 1], minlength=V).astype(np.float64)
            pc = np.asarray(dsm.probabilities(zt1[c], inv_t), np.float64)
            assert _chi2_pvalue(h, pc) > 1e-3
