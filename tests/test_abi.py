"""The C ABI: the library loads, exports every symbol the header declares, and rejects bad
arguments on the host before launching anything (no GPU needed)."""
import ctypes

import pytest

from tests._util import built_lib, header_functions
from eagle_tree_speculative_spec_gb300 import _lib as B


def test_header_symbols_exported():
    L = built_lib()
    names = header_functions()
    assert {"eagle3_accept", "eagle3_compact_kv", "eagle3_verify_attn", "eagle3_status_string"} <= set(names)
    for n in names:
        assert hasattr(L, n), n


def test_status_strings():
    L = built_lib()
    for s in range(7):
        assert L.eagle3_status_string(s)
    assert L.eagle3_version() >= 100


def _accept(**kw):
    base = dict(mode=0, batch=2, n_nodes=5, vocab=100, max_path=7, temperature=1.0, seed=1, step=0,
                target_logits=16, draft_logits=None, tokens=16, parents=16, accept_len=16, path=16,
                emitted=16, next_root=16, dev_status=None)
    base.update(kw)
    return B.AcceptArgs(**base)


@pytest.mark.parametrize("kw,want", [
    (dict(batch=0), 0),
    (dict(n_nodes=65), 2),
    (dict(n_nodes=0), 1),
    (dict(vocab=0), 1),
    (dict(max_path=0), 1),
    (dict(mode=7), 1),
    (dict(mode=1, temperature=0.0), 1),
    (dict(mode=1, temperature=-1.0), 1),
    (dict(mode=2, draft_logits=None), 1),
    (dict(target_logits=None), 1),
    (dict(mode=2, draft_logits=16), 6),     # SAMPLED without its workspace
])
def test_accept_host_validation(kw, want):
    L = built_lib()
    a = _accept(**kw)
    assert L.eagle3_accept(ctypes.byref(a), None, 0, None) == want


def test_accept_workspace_size():
    L = built_lib()
    assert L.eagle3_accept_workspace_size(ctypes.byref(_accept(mode=0))) == 0
    assert L.eagle3_accept_workspace_size(ctypes.byref(_accept(mode=2, draft_logits=16))) == 2 * 2 * 100 * 4


def _verify(**kw):
    base = dict(batch=2, n_nodes=60, n_heads=32, n_kv_heads=8, head_dim=128, s_max=4096, max_prefix_len=1024,
                num_splits=0, rope_theta=500000.0, sm_scale=0.0, q=16, tree_k=16, tree_v=16, k_cache=16,
                v_cache=16, parents=16, prefix_len=16, out=16, lse=None, dev_status=None)
    base.update(kw)
    return B.VerifyAttnArgs(**base)


@pytest.mark.parametrize("kw,want", [
    (dict(batch=0), 0),
    (dict(head_dim=64), 2),
    (dict(n_nodes=65), 2),
    (dict(n_heads=30), 1),
    (dict(max_prefix_len=4090), 3),          # A27-style capacity check: L + N > S_max
    (dict(q=None), 1),
    (dict(q=18), 1),                         # not 16-byte aligned
    (dict(rope_theta=0.0), 1),
])
def test_verify_host_validation(kw, want):
    L = built_lib()
    a = _verify(**kw)
    assert L.eagle3_verify_attn(ctypes.byref(a), None, 0, None) == want


def test_compact_host_validation():
    L = built_lib()
    a = B.CompactArgs(n_layers=2, batch=1, n_nodes=5, n_kv_heads=2, head_dim=8, elem_bytes=3, s_max=10,
                      max_path=3, cache_layer_stride=1000, tree_layer_stride=1000)
    assert L.eagle3_compact_kv(ctypes.byref(a), None) == 2
    a.elem_bytes = 2
    assert L.eagle3_compact_kv(ctypes.byref(a), None) == 1        # null pointers
    a.batch = 0
    assert L.eagle3_compact_kv(ctypes.byref(a), None) == 0


def _linear(**kw):
    base = dict(m=128, n=768, k=256, epilogue=4, splits=0, ld_x=0, ld_w=0, ld_out=0, ld_res=0, x=16, w=16, w2=None,
                out=16, residual=None, dev_status=None, rope_cols=640, rope_rows_per_seq=60, rope_theta=500000.0,
                rope_base=16, rope_depth=16)
    base.update(kw)
    return B.LinearArgs(**base)


@pytest.mark.parametrize("kw,want", [
    (dict(m=0), 0),
    (dict(rope_cols=100), 1),          # not whole 128-wide heads
    (dict(rope_cols=896), 1),          # beyond the output columns
    (dict(rope_rows_per_seq=0), 1),
    (dict(rope_theta=0.0), 1),
    (dict(splits=2), 1),               # the RoPE epilogue runs unsplit
    (dict(rope_base=None), 1),
    (dict(rope_depth=None), 1),
    (dict(out=24), 2),                 # outputs leave by TMA: 16-byte aligned only
    (dict(ld_out=772), 2),             # ... with a whole-16-byte row pitch
    (dict(epilogue=5), 1),
])
def test_linear_rope_host_validation(kw, want):
    L = built_lib()
    a = _linear(**kw)
    assert L.eagle3_linear(ctypes.byref(a), None, 0, None) == want


def _draft(**kw):
    base = dict(batch=2, hidden=256, n_heads=4, n_kv_heads=2, head_dim=128, ffn=512, vocab=1000, depth=4, top_k=4,
                n_nodes=12, tc_max=2, s_max=64, max_draft_len=32, rope_theta=500000.0, rms_eps=1e-5, aux=16,
                next_tokens=16, tc=16, draft_k_cache=16, draft_v_cache=16, draft_len=16, tokens=16, parents=16,
                depth_out=16, anc_mask=16, score=16, dbg_logits=None, dev_status=None, draft_vocab=0, d2t=None)
    base.update(kw)
    return B.DraftTreeArgs(**base)


@pytest.mark.parametrize("kw,want", [
    (dict(batch=0), 0),
    (dict(batch=0, draft_vocab=300, d2t=16), 0),
    (dict(draft_vocab=-1), 1),
    (dict(draft_vocab=1001, d2t=16), 1),      # larger than the target vocabulary
    (dict(draft_vocab=300), 1),               # a reduced vocabulary needs its map
    (dict(draft_vocab=3, d2t=16), 2),         # top_k above the draft vocabulary
    (dict(head_dim=64), 2),
    (dict(max_draft_len=63), 3),              # max_draft_len + tc_max > s_max
    (dict(tokens=None), 1),
])
def test_draft_tree_host_validation(kw, want):
    L = built_lib()
    a = _draft(**kw)
    assert L.eagle3_draft_tree(None, ctypes.byref(a), None, 0, None) == want


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    """Without the built library every call raises: there is no fallback implementation."""
    monkeypatch.setattr(B, "_lib", None)
    monkeypatch.setattr(B, "LIB_PATH", str(tmp_path / "libeagle3.so"))
    with pytest.raises(RuntimeError, match="no fallback"):
        B.lib()
    with pytest.raises(RuntimeError):
        B.eagle3_draft_tree_workspace_size(_draft())
