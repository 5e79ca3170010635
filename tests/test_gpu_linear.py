"""GPU numerics of the tcgen05 linear layer against an fp64 matmul of the same bf16 inputs
(bf16 outputs: 2e-2 abs + 1e-2 rel; fp32 outputs: 1e-3 abs + 1e-3 rel)."""
import numpy as np
import pytest
import torch

from tests._util import close, require_gpu

pytestmark = pytest.mark.gpu


def _inputs(m, n, k, seed, swiglu=False):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(m, k, generator=g).to(torch.bfloat16)
    w = (0.02 * torch.randn(n, k, generator=g)).to(torch.bfloat16)
    w2 = (0.02 * torch.randn(n, k, generator=g)).to(torch.bfloat16) if swiglu else None
    return x, w, w2


def _ref(x, w):
    return x.double().numpy() @ w.double().numpy().T


def _silu(v):
    return v / (1.0 + np.exp(-v))


def _run(m, n, k, epi, seed=0, splits=0):
    from eagle_tree_speculative_spec_gb300 import EPI_BF16_RESIDUAL, EPI_F32, EPI_SWIGLU, eagle3_linear
    dev = require_gpu()
    x, w, w2 = _inputs(m, n, k, seed, swiglu=epi == EPI_SWIGLU)
    res = torch.randn(m, n).to(torch.bfloat16) if epi == EPI_BF16_RESIDUAL else None
    out = torch.full((m, n), float("nan"), dtype=torch.float32 if epi == EPI_F32 else torch.bfloat16, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    eagle3_linear(x.to(dev), w.to(dev), out, epilogue=epi, w2=None if w2 is None else w2.to(dev),
                  residual=None if res is None else res.to(dev), splits=splits, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    got = out.float().cpu().numpy()
    if epi == EPI_SWIGLU:
        want = _silu(_ref(x, w)) * _ref(x, w2)
    else:
        want = _ref(x, w)
        if res is not None:
            want = want + res.double().numpy()
    return got, want


def test_linear_single_tile():
    from eagle_tree_speculative_spec_gb300 import EPI_BF16
    got, want = _run(128, 256, 64, EPI_BF16)
    ok, err = close(got, want, 2e-2, 1e-2)
    assert ok, err


@pytest.mark.parametrize("m,n,k,splits", [
    (128, 256, 128, 1), (5, 1000, 64, 0), (130, 300, 200, 0), (10, 4096, 12288, 0), (10, 4096, 12288, 3),
    (640, 6144, 8192, 0), (257, 512, 4096, 2), (1, 256, 64, 0)])
def test_linear_bf16(m, n, k, splits):
    from eagle_tree_speculative_spec_gb300 import EPI_BF16
    got, want = _run(m, n, k, EPI_BF16, seed=m + n + k, splits=splits)
    ok, err = close(got, want, 2e-2, 1e-2)
    assert ok, err


@pytest.mark.parametrize("m,n,k", [(10, 128256, 4096), (130, 1000, 4096), (64, 4096, 64)])
def test_linear_f32_logits(m, n, k):
    from eagle_tree_speculative_spec_gb300 import EPI_F32
    got, want = _run(m, n, k, EPI_F32, seed=1)
    ok, err = close(got, want, 1e-3, 1e-3)
    assert ok, err


@pytest.mark.parametrize("m,n,k,splits", [(10, 4096, 4096, 0), (640, 4096, 14336, 0), (70, 256, 256, 1)])
def test_linear_residual(m, n, k, splits):
    from eagle_tree_speculative_spec_gb300 import EPI_BF16_RESIDUAL
    got, want = _run(m, n, k, EPI_BF16_RESIDUAL, seed=2, splits=splits)
    ok, err = close(got, want, 2e-2, 1e-2)
    assert ok, err


@pytest.mark.parametrize("m,n,k,splits", [(10, 14336, 4096, 0), (640, 14336, 4096, 0), (33, 300, 512, 3)])
def test_linear_swiglu(m, n, k, splits):
    from eagle_tree_speculative_spec_gb300 import EPI_SWIGLU
    got, want = _run(m, n, k, EPI_SWIGLU, seed=3, splits=splits)
    ok, err = close(got, want, 2e-2, 1e-2)
    assert ok, err


def test_linear_in_place_residual():
    """out may be the residual buffer itself (x = x + o_proj(attn))."""
    from eagle_tree_speculative_spec_gb300 import EPI_BF16_RESIDUAL, eagle3_linear
    dev = require_gpu()
    x, w, _ = _inputs(64, 512, 512, 9)
    r = torch.randn(64, 512).to(torch.bfloat16)
    buf = r.to(dev).clone()
    eagle3_linear(x.to(dev), w.to(dev), buf, epilogue=EPI_BF16_RESIDUAL, residual=buf)
    torch.cuda.synchronize()
    ok, err = close(buf.float().cpu().numpy(), _ref(x, w) + r.double().numpy(), 2e-2, 1e-2)
    assert ok, err


@pytest.mark.parametrize("m,n,k,epi", [
    (768, 4096, 12288, "bf16"), (300, 1000, 12296, "bf16"), (130, 4096, 14336, "residual"),
    (200, 4096, 12288, "f32"), (640, 2048, 12288, "swiglu"), (1, 4096, 14336, "bf16"),
    (3584, 2816, 12288, "bf16"),      # 308 tiles: 152 data-parallel, the rest shared out (4 tail tiles)
    (64, 128256, 4096, "f32")])       # one M tile, 501 tiles: 304 data-parallel in front
def test_linear_stream_k(m, n, k, epi):
    """Long-K shapes whose output tiles leave the last wave partly empty (and which a split of the
    last wave's tiles cannot fill), and single-M-tile launches, run the stream-K schedule: tiles cut
    between CTAs are finished by the CTA holding their first k-block, which adds the others' fp32
    slots in CTA order; the last two shapes have data-parallel waves in front."""
    import eagle_tree_speculative_spec_gb300 as e3
    code = {"bf16": e3.EPI_BF16, "residual": e3.EPI_BF16_RESIDUAL, "f32": e3.EPI_F32, "swiglu": e3.EPI_SWIGLU}[epi]
    got, want = _run(m, n, k, code, seed=5)
    atol, rtol = (1e-3, 1e-3) if epi == "f32" else (2e-2, 1e-2)
    ok, err = close(got, want, atol, rtol)
    assert ok, err


@pytest.mark.parametrize("m,rows_per_seq,n_heads,rope_heads", [(120, 60, 6, 5), (3840, 60, 48, 40), (7, 7, 3, 2)])
def test_linear_rope_epilogue(m, rows_per_seq, n_heads, rope_heads):
    """EPI_BF16_ROPE: the fused projection leaves its first rope_heads 128-wide heads rotated at
    position base[row // rows_per_seq] + depth[row] (rotate-half RoPE, angles fp32(pos * inv_j)),
    the rest plain; against the fp64 product rotated by the oracle's RoPE."""
    from oracle import attention as oatt
    from eagle_tree_speculative_spec_gb300 import EPI_BF16_ROPE, eagle3_linear
    dev = require_gpu()
    n, k = n_heads * 128, 256
    x, w, _ = _inputs(m, n, k, 5)
    g = np.random.default_rng(6)
    n_seq = (m + rows_per_seq - 1) // rows_per_seq
    base = g.integers(0, 20000, n_seq).astype(np.int32)
    depth = g.integers(0, 7, m).astype(np.int32)
    out = torch.full((m, n), float("nan"), dtype=torch.bfloat16, device=dev)
    eagle3_linear(x.to(dev), w.to(dev), out, epilogue=EPI_BF16_ROPE, rope_cols=rope_heads * 128,
                  rope_rows_per_seq=rows_per_seq, rope_theta=500000.0,
                  rope_base=torch.as_tensor(base, device=dev), rope_depth=torch.as_tensor(depth, device=dev))
    torch.cuda.synchronize()
    want = _ref(x, w)
    pos = base[np.arange(m) // rows_per_seq] + depth
    rot = want[:, : rope_heads * 128].reshape(m, rope_heads, 128)
    want[:, : rope_heads * 128] = oatt.rope_apply(rot, pos, 500000.0).reshape(m, rope_heads * 128)
    ok, err = close(out.float().cpu().numpy(), want, 2e-2, 1e-2)
    assert ok, f"max err {err}"


def test_linear_rope_epilogue_padded_pitch():
    """The RoPE epilogue through the C ABI with a padded output pitch (ld_out = n + 64): the padding
    columns are left alone."""
    import ctypes
    from oracle import attention as oatt
    from eagle_tree_speculative_spec_gb300 import EPI_BF16_ROPE
    from eagle_tree_speculative_spec_gb300 import _lib as E
    dev = require_gpu()
    m, n, k, rows_per_seq = 100, 512, 256, 50
    x, w, _ = _inputs(m, n, k, 7)
    base = torch.tensor([40, 900], dtype=torch.int32, device=dev)
    depth = torch.arange(m, dtype=torch.int32, device=dev) % 7
    out = torch.full((m, n + 64), 3.0, dtype=torch.bfloat16, device=dev)
    xd, wd = x.to(dev), w.to(dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    a = E.LinearArgs(m=m, n=n, k=k, epilogue=EPI_BF16_ROPE, splits=0, ld_x=0, ld_w=0, ld_out=n + 64, ld_res=0,
                     x=xd.data_ptr(), w=wd.data_ptr(), w2=None, out=out.data_ptr(), residual=None,
                     dev_status=st.data_ptr(), rope_cols=256, rope_rows_per_seq=rows_per_seq, rope_theta=10000.0,
                     rope_base=base.data_ptr(), rope_depth=depth.data_ptr())
    ws = torch.empty(1 << 20, dtype=torch.uint8, device=dev)
    assert E.lib().eagle3_linear(ctypes.byref(a), ws.data_ptr(), ws.numel(), None) == 0
    torch.cuda.synchronize()
    got = out.float().cpu().numpy()
    assert (got[:, n:] == 3.0).all()
    want = _ref(x, w)
    pos = base.cpu().numpy()[np.arange(m) // rows_per_seq] + depth.cpu().numpy()
    want[:, :256] = oatt.rope_apply(want[:, :256].reshape(m, 2, 128), pos, 10000.0).reshape(m, 256)
    ok, err = close(got[:, :n], want, 2e-2, 1e-2)
    assert ok, f"max err {err}"


@pytest.mark.parametrize("m,n,k,splits", [
    (10, 128256, 4096, 0),    # one M tile, many N tiles: stream-K (owners finish the cut tiles)
    (10, 32000, 4096, 0),     # one M tile, few N tiles: split-K (the reduce kernel writes the outputs)
    (640, 128256, 512, 0),    # many tiles: data-parallel, TMA-stored
    (130, 1001, 256, 0),      # unaligned row pitch: direct stores
    (33, 300, 512, 3)])       # forced split-K, rows spanning a warp's outputs
def test_linear_f32_row_max(m, n, k, splits):
    """The fp32 epilogue's row maxima: each row's word ends at the order key of the row's largest
    output (bit-exact against the maximum of the outputs the same call wrote), however the plan
    finishes the tiles."""
    from eagle_tree_speculative_spec_gb300 import EPI_F32, eagle3_linear
    dev = require_gpu()
    x, w, _ = _inputs(m, n, k, 11)
    out = torch.full((m, n), float("nan"), dtype=torch.float32, device=dev)
    rmax = torch.zeros(m, dtype=torch.int32, device=dev)
    eagle3_linear(x.to(dev), w.to(dev), out, epilogue=EPI_F32, splits=splits, row_max=rmax)
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    bits = got.view(np.uint32).astype(np.uint64)
    keys = np.where(bits >> 31, ~bits & 0xFFFFFFFF, bits | 0x80000000)
    assert np.array_equal(rmax.cpu().numpy().view(np.uint32).astype(np.uint64), keys.max(1))
    ok, err = close(got, _ref(x, w), 1e-3, 1e-3)
    assert ok, err


@pytest.mark.parametrize("m,n,k,epi_name", [
    (1280, 4096, 2048, "residual"),   # 160 tiles: 152 whole, 8 tail tiles split 8 ways
    (1280, 2048, 2048, "swiglu"),     # 10 x 16 SwiGLU tiles (gate / up halves paired in the reduce)
    (1290, 4100, 1024, "bf16"),       # ragged edges: 187 tiles, 35 tail tiles split 4 ways
    (1280, 4096, 2048, "f32"),        # fp32 logits with the row maxima published by the reduce
    (3840, 4096, 14336, "residual"),  # the target's down projection: 24 tail tiles split 6 ways
    (1290, 4100, 12288, "residual")])  # ragged, long k: 35 tail tiles split 4 ways (stream-K's shape before)
def test_linear_split_tail(m, n, k, epi_name):
    """Whole waves of tiles run data-parallel and the partial last wave's tiles are split along k,
    their partials added in split order by a second kernel: the same products as the fp64 matmul."""
    import eagle_tree_speculative_spec_gb300 as e3
    epi = {"residual": e3.EPI_BF16_RESIDUAL, "swiglu": e3.EPI_SWIGLU, "bf16": e3.EPI_BF16, "f32": e3.EPI_F32}[epi_name]
    dev = require_gpu()
    x, w, w2 = _inputs(m, n, k, 13, swiglu=epi == e3.EPI_SWIGLU)
    res = torch.randn(m, n).to(torch.bfloat16) if epi == e3.EPI_BF16_RESIDUAL else None
    out = torch.full((m, n), float("nan"), dtype=torch.float32 if epi == e3.EPI_F32 else torch.bfloat16, device=dev)
    rmax = torch.zeros(m, dtype=torch.int32, device=dev) if epi == e3.EPI_F32 else None
    e3.eagle3_linear(x.to(dev), w.to(dev), out, epilogue=epi, w2=None if w2 is None else w2.to(dev),
                     residual=None if res is None else res.to(dev), row_max=rmax)
    torch.cuda.synchronize()
    got = out.float().cpu().numpy()
    if epi == e3.EPI_SWIGLU:
        want = _silu(_ref(x, w)) * _ref(x, w2)
    else:
        want = _ref(x, w) + (res.double().numpy() if res is not None else 0.0)
    tol = (1e-3, 1e-3) if epi == e3.EPI_F32 else (2e-2, 1e-2)
    ok, err = close(got, want, *tol)
    assert ok, err
    if rmax is not None:
        bits = got.view(np.uint32).astype(np.uint64)
        keys = np.where(bits >> 31, ~bits & 0xFFFFFFFF, bits | 0x80000000)
        assert np.array_equal(rmax.cpu().numpy().view(np.uint32).astype(np.uint64), keys.max(1))


@pytest.mark.parametrize("m,n,k,epi_name", [
    (130, 1000, 256, "residual"),      # data-parallel, a partial 256-column block, direct-store tails
    (1280, 4096, 2048, "residual"),    # split tail: the reduce kernel writes outputs and row sums
    (768, 4096, 12288, "bf16"),        # stream-K: owners finish the cut tiles
    (1290, 4100, 12288, "residual"),   # ragged split tail at long k (35 tail tiles, 4 ranges)
    (300, 1000, 512, "bf16")])         # unaligned pitch of the output: direct stores
def test_linear_row_ssq(m, n, k, epi_name):
    """row_ssq: for each row and block of 256 output columns, the sum of squares of the bf16 outputs
    the same call stored (any plan) — the per-row statistic a folded RMSNorm of the next projection
    needs."""
    import eagle_tree_speculative_spec_gb300 as e3
    epi = {"residual": e3.EPI_BF16_RESIDUAL, "bf16": e3.EPI_BF16}[epi_name]
    dev = require_gpu()
    x, w, _ = _inputs(m, n, k, 17)
    res = torch.randn(m, n).to(torch.bfloat16) if epi == e3.EPI_BF16_RESIDUAL else None
    out = torch.full((m, n), float("nan"), dtype=torch.bfloat16, device=dev)
    blocks = (n + 255) // 256
    ssq = torch.full((blocks, m), float("nan"), dtype=torch.float32, device=dev)
    e3.eagle3_linear(x.to(dev), w.to(dev), out, epilogue=epi, residual=None if res is None else res.to(dev),
                     row_ssq=ssq)
    torch.cuda.synchronize()
    o = out.double().cpu().numpy()
    want = np.stack([(o[:, 256 * b:256 * (b + 1)] ** 2).sum(1) for b in range(blocks)])
    got = ssq.cpu().numpy()
    assert np.isfinite(got).all()
    assert np.allclose(got, want, rtol=1e-5, atol=1e-6), np.abs(got - want).max()
    ok, err = close(o, _ref(x, w) + (res.double().numpy() if res is not None else 0.0), 2e-2, 1e-2)
    assert ok, err


@pytest.mark.parametrize("m,n,k,epi_name", [
    (130, 1000, 256, "bf16"), (1280, 2048, 2048, "swiglu"), (768, 4096, 12288, "residual"),
    (640, 16384, 512, "f32"), (120, 768, 256, "rope"), (1290, 4100, 1024, "bf16")])
def test_linear_folded_rmsnorm(m, n, k, epi_name):
    """row_ssq_in: every output row is scaled by rsqrt(sum of the row's block sums / dim + eps)
    before the epilogue, i.e. RMSNorm(x) W^T = diag(rsqrt(mean(x^2) + eps)) x W^T with x's sums of
    squares given per block (data-parallel, split-tail, stream-K and TMA-stored fp32 plans)."""
    from oracle import attention as oatt
    import eagle_tree_speculative_spec_gb300 as e3
    epi = {"bf16": e3.EPI_BF16, "swiglu": e3.EPI_SWIGLU, "residual": e3.EPI_BF16_RESIDUAL, "f32": e3.EPI_F32,
           "rope": e3.EPI_BF16_ROPE}[epi_name]
    dev = require_gpu()
    x, w, w2 = _inputs(m, n, k, 19, swiglu=epi == e3.EPI_SWIGLU)
    xd = x.double().numpy()
    blocks, eps = 3, 1e-5
    # the row sums of squares of x, cut into three uneven blocks (their order is the addition order)
    cuts = [0, k // 3, (2 * k) // 3, k]
    sums = np.stack([(xd[:, cuts[b]:cuts[b + 1]] ** 2).sum(1) for b in range(blocks)]).astype(np.float32)
    scale = 1.0 / np.sqrt(sums.astype(np.float64).sum(0) / k + eps)
    res = torch.randn(m, n).to(torch.bfloat16) if epi == e3.EPI_BF16_RESIDUAL else None
    out = torch.full((m, n), float("nan"), dtype=torch.float32 if epi == e3.EPI_F32 else torch.bfloat16, device=dev)
    kw = {}
    if epi == e3.EPI_BF16_ROPE:
        g = np.random.default_rng(21)
        base = g.integers(0, 5000, (m + 59) // 60).astype(np.int32)
        depth = g.integers(0, 7, m).astype(np.int32)
        kw = dict(rope_cols=512, rope_rows_per_seq=60, rope_theta=500000.0,
                  rope_base=torch.as_tensor(base, device=dev), rope_depth=torch.as_tensor(depth, device=dev))
    e3.eagle3_linear(x.to(dev), w.to(dev), out, epilogue=epi, w2=None if w2 is None else w2.to(dev),
                     residual=None if res is None else res.to(dev), row_ssq_in=torch.as_tensor(sums, device=dev),
                     ssq_dim=k, ssq_eps=eps, **kw)
    torch.cuda.synchronize()
    acc = _ref(x, w) * scale[:, None]
    if epi == e3.EPI_SWIGLU:
        want = _silu(acc) * (_ref(x, w2) * scale[:, None])
    elif epi == e3.EPI_BF16_ROPE:
        want = acc.copy()
        pos = base[np.arange(m) // 60] + depth
        want[:, :512] = oatt.rope_apply(acc[:, :512].reshape(m, 4, 128), pos, 500000.0).reshape(m, 512)
    else:
        want = acc + (res.double().numpy() if res is not None else 0.0)
    tol = (1e-3, 1e-3) if epi == e3.EPI_F32 else (2e-2, 1e-2)
    ok, err = close(out.float().cpu().numpy(), want, *tol)
    assert ok, err


def test_linear_folded_rmsnorm_rejects_k_split():
    """A caller-requested k split with a per-row epilogue input or output is refused on the host."""
    import eagle_tree_speculative_spec_gb300 as e3
    dev = require_gpu()
    x, w, _ = _inputs(64, 512, 256, 1)
    out = torch.empty(64, 512, dtype=torch.bfloat16, device=dev)
    ssq = torch.zeros(2, 64, dtype=torch.float32, device=dev)
    with pytest.raises(e3.Eagle3Error):
        e3.eagle3_linear(x.to(dev), w.to(dev), out, splits=2, row_ssq=ssq)
