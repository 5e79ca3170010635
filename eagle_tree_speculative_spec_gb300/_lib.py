"""Thin ctypes binding of libeagle3 (argument marshalling only).

Every function here has the name of the C entry point it calls, takes torch
tensors that already live on the GPU, checks dtype / shape / contiguity,
fills the C argument struct with their data pointers and launches on the
current torch stream.  No computation happens in Python: if the library is
missing, the calls raise instead of falling back to anything else.
"""
import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libeagle3.so")
_lib = None


class Eagle3Error(RuntimeError):
    def __init__(self, status, what):
        super().__init__(f"{what}: {status_string(status)} (status {status})")
        self.status = status


def lib():
    """Load libeagle3.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with __graft_entry__.build() "
                               "(there is no fallback implementation)")
        _lib = ctypes.CDLL(LIB_PATH)
        _declare(_lib)
    return _lib


# ----------------------------------------------------------------------------- C structs
GREEDY, TOPK, SAMPLED = 0, 1, 2
DEV_BAD_TREE, DEV_BAD_TOKEN, DEV_CAPACITY, DEV_TIMEOUT, DEV_PATH_TRUNC = 0x1, 0x2, 0x4, 0x8, 0x10

_p = ctypes.c_void_p
_i32, _i64, _u64, _f32 = ctypes.c_int32, ctypes.c_int64, ctypes.c_uint64, ctypes.c_float


class AcceptArgs(ctypes.Structure):
    _fields_ = [("mode", _i32), ("batch", _i32), ("n_nodes", _i32), ("vocab", _i32), ("max_path", _i32),
                ("temperature", _f32), ("seed", _u64), ("step", _u64),
                ("target_logits", _p), ("draft_logits", _p), ("tokens", _p), ("parents", _p),
                ("accept_len", _p), ("path", _p), ("emitted", _p), ("next_root", _p), ("dev_status", _p),
                ("step_counter", _p)]


class AcceptLazyArgs(ctypes.Structure):
    _fields_ = [("accept", AcceptArgs), ("hidden", _i32), ("hidden_states", _p), ("lm_head", _p),
                ("dbg_level_logits", _p)]


class CompactArgs(ctypes.Structure):
    _fields_ = [("n_layers", _i32), ("batch", _i32), ("n_nodes", _i32), ("n_kv_heads", _i32),
                ("head_dim", _i32), ("elem_bytes", _i32), ("s_max", _i32), ("max_path", _i32),
                ("cache_layer_stride", _i64), ("tree_layer_stride", _i64), ("tree_node_stride", _i64),
                ("k_cache", _p), ("v_cache", _p), ("tree_k", _p), ("tree_v", _p),
                ("path", _p), ("accept_len", _p), ("prefix_len", _p), ("slot_map", _p), ("committed", _p),
                ("aux_dim", _i32), ("aux_tree", _p), ("aux_out", _p), ("dev_status", _p),
                ("block_table", _p), ("max_blocks", _i32), ("block_size", _i32), ("n_slots", _i32)]


class VerifyAttnArgs(ctypes.Structure):
    _fields_ = [("batch", _i32), ("n_nodes", _i32), ("n_heads", _i32), ("n_kv_heads", _i32),
                ("head_dim", _i32), ("s_max", _i32), ("max_prefix_len", _i32), ("num_splits", _i32),
                ("q_node_stride", _i64), ("kv_node_stride", _i64), ("rope_theta", _f32), ("sm_scale", _f32),
                ("q", _p), ("tree_k", _p), ("tree_v", _p), ("k_cache", _p), ("v_cache", _p),
                ("parents", _p), ("prefix_len", _p), ("out", _p), ("lse", _p), ("dev_status", _p),
                ("qk_rotated", _i32), ("block_table", _p), ("max_blocks", _i32), ("block_size", _i32),
                ("n_slots", _i32)]


class LinearArgs(ctypes.Structure):
    _fields_ = [("m", _i32), ("n", _i32), ("k", _i32), ("epilogue", _i32), ("splits", _i32),
                ("ld_x", _i64), ("ld_w", _i64), ("ld_out", _i64), ("ld_res", _i64),
                ("x", _p), ("w", _p), ("w2", _p), ("out", _p), ("residual", _p), ("dev_status", _p),
                ("rope_cols", _i32), ("rope_rows_per_seq", _i32), ("rope_theta", ctypes.c_float),
                ("rope_base", _p), ("rope_depth", _p), ("row_max", _p),
                ("row_ssq", _p), ("row_ssq_in", _p), ("ssq_blocks", _i32), ("ssq_dim", _i32), ("ssq_eps", _f32)]


EPI_BF16, EPI_F32, EPI_BF16_RESIDUAL, EPI_SWIGLU, EPI_BF16_ROPE = 0, 1, 2, 3, 4
DEV_BAD_COUNTS = 0x20


class SpecDecodeMetadataArgs(ctypes.Structure):
    _fields_ = [("n_requests", _i32), ("max_rows", _i32), ("cu_num_scheduled_tokens", _p), ("num_draft_tokens", _p),
                ("cu_num_draft_tokens", _p), ("logits_indices", _p), ("target_logits_indices", _p),
                ("bonus_logits_indices", _p), ("num_rows", _p), ("dev_status", _p)]


class TttAttnArgs(ctypes.Structure):
    _fields_ = [("batch", _i32), ("seq_len", _i32), ("n_heads", _i32), ("n_kv_heads", _i32), ("head_dim", _i32),
                ("n_steps", _i32), ("sm_scale", _f32), ("q", _p), ("k", _p), ("v", _p), ("out", _p),
                ("dev_status", _p)]


class ChainVerifyArgs(ctypes.Structure):
    _fields_ = [("n_requests", _i32), ("vocab", _i32), ("max_drafts", _i32), ("temperature", _f32),
                ("seed", _u64), ("step", _u64), ("logits", _p), ("draft_tokens", _p), ("cu_num_draft_tokens", _p),
                ("is_greedy", _p), ("output_tokens", _p), ("num_accepted", _p), ("dev_status", _p),
                ("step_counter", _p)]

DRAFT_WEIGHT_NAMES = ("w_fc", "embed", "input_norm", "hidden_norm", "w_qkv", "w_o", "post_norm", "w_gate",
                      "w_up", "w_down", "final_norm", "lm_head")


class DraftWeights(ctypes.Structure):
    _fields_ = [(n, _p) for n in DRAFT_WEIGHT_NAMES]


class DraftTreeArgs(ctypes.Structure):
    _fields_ = [("batch", _i32), ("hidden", _i32), ("n_heads", _i32), ("n_kv_heads", _i32), ("head_dim", _i32),
                ("ffn", _i32), ("vocab", _i32), ("depth", _i32), ("top_k", _i32), ("n_nodes", _i32),
                ("tc_max", _i32), ("s_max", _i32), ("max_draft_len", _i32), ("rope_theta", _f32), ("rms_eps", _f32),
                ("aux", _p), ("next_tokens", _p), ("tc", _p), ("draft_k_cache", _p), ("draft_v_cache", _p),
                ("draft_len", _p), ("tokens", _p), ("parents", _p), ("depth_out", _p), ("anc_mask", _p),
                ("score", _p), ("dbg_logits", _p), ("dev_status", _p), ("draft_vocab", _i32), ("d2t", _p)]


F32_EPI_NONE, F32_EPI_RESIDUAL, F32_EPI_SWIGLU = 0, 1, 2


class F32LinearArgs(ctypes.Structure):
    _fields_ = [("m", _i64), ("n", _i64), ("k", _i64), ("epilogue", _i32), ("ld_x", _i64), ("ld_out", _i64),
                ("ld_res", _i64), ("x", _p), ("w", _p), ("w2", _p), ("residual", _p), ("out", _p)]


class F32AttnArgs(ctypes.Structure):
    _fields_ = [("n_rows", _i32), ("n_heads", _i32), ("n_kv_heads", _i32), ("head_dim", _i32), ("cache_len", _i32),
                ("s_max", _i32), ("scale", _f32), ("ld_q", _i64), ("ld_kv", _i64), ("q", _p), ("k_new", _p),
                ("v_new", _p), ("k_cache", _p), ("v_cache", _p), ("visible", _p), ("out", _p)]


class RmsnormArgs(ctypes.Structure):
    _fields_ = [("rows", _i32), ("dim", _i32), ("n_src", _i32), ("eps", _f32), ("ld_in", _i64), ("ld_out", _i64),
                ("ld_tap", _i64), ("input", _p), ("w", _p), ("gather", _p), ("out", _p), ("tap_out", _p),
                ("dev_status", _p)]


def _declare(L):
    P = ctypes.POINTER
    L.eagle3_status_string.restype = ctypes.c_char_p
    L.eagle3_status_string.argtypes = [ctypes.c_int]
    L.eagle3_version.restype = ctypes.c_int
    L.eagle3_accept_workspace_size.restype = ctypes.c_size_t
    L.eagle3_accept_workspace_size.argtypes = [P(AcceptArgs)]
    L.eagle3_accept.restype = ctypes.c_int
    L.eagle3_accept.argtypes = [P(AcceptArgs), _p, ctypes.c_size_t, _p]
    L.eagle3_accept_lazy_workspace_size.restype = ctypes.c_size_t
    L.eagle3_accept_lazy_workspace_size.argtypes = [P(AcceptLazyArgs)]
    L.eagle3_accept_lazy.restype = ctypes.c_int
    L.eagle3_accept_lazy.argtypes = [P(AcceptLazyArgs), _p, ctypes.c_size_t, _p]
    L.eagle3_compact_kv.restype = ctypes.c_int
    L.eagle3_compact_kv.argtypes = [P(CompactArgs), _p]
    L.eagle3_verify_attn_workspace_size.restype = ctypes.c_size_t
    L.eagle3_verify_attn_workspace_size.argtypes = [P(VerifyAttnArgs)]
    L.eagle3_verify_attn.restype = ctypes.c_int
    L.eagle3_verify_attn.argtypes = [P(VerifyAttnArgs), _p, ctypes.c_size_t, _p]
    L.eagle3_ttt_attn_workspace_size.restype = ctypes.c_size_t
    L.eagle3_ttt_attn_workspace_size.argtypes = [P(TttAttnArgs)]
    L.eagle3_ttt_attn.restype = ctypes.c_int
    L.eagle3_ttt_attn.argtypes = [P(TttAttnArgs), _p, ctypes.c_size_t, _p]
    L.eagle3_spec_decode_metadata.restype = ctypes.c_int
    L.eagle3_spec_decode_metadata.argtypes = [P(SpecDecodeMetadataArgs), _p]
    L.eagle3_chain_verify.restype = ctypes.c_int
    L.eagle3_chain_verify.argtypes = [P(ChainVerifyArgs), _p]
    L.eagle3_test_verify_attn_timeout.restype = ctypes.c_int
    L.eagle3_test_verify_attn_timeout.argtypes = [P(VerifyAttnArgs), _p, ctypes.c_size_t, _i32, _i64, _p]
    L.eagle3_verify_attn_noalloc.restype = ctypes.c_int
    L.eagle3_verify_attn_noalloc.argtypes = [P(VerifyAttnArgs), _p]
    L.eagle3_linear_workspace_size.restype = ctypes.c_size_t
    L.eagle3_linear_workspace_size.argtypes = [P(LinearArgs)]
    L.eagle3_linear.restype = ctypes.c_int
    L.eagle3_linear.argtypes = [P(LinearArgs), _p, ctypes.c_size_t, _p]
    L.eagle3_draft_tree_workspace_size.restype = ctypes.c_size_t
    L.eagle3_draft_tree_workspace_size.argtypes = [P(DraftTreeArgs)]
    L.eagle3_draft_tree.restype = ctypes.c_int
    L.eagle3_draft_tree.argtypes = [P(DraftWeights), P(DraftTreeArgs), _p, ctypes.c_size_t, _p]
    L.eagle3_rmsnorm.restype = ctypes.c_int
    L.eagle3_rmsnorm.argtypes = [P(RmsnormArgs), _p]
    L.eagle3_f32_linear.restype = ctypes.c_int
    L.eagle3_f32_linear.argtypes = [P(F32LinearArgs), _p]
    L.eagle3_f32_rmsnorm.restype = ctypes.c_int
    L.eagle3_f32_rmsnorm.argtypes = [_i64, _i64, _p, _i64, _p, _p, _f32, _p, _i64, _p]
    L.eagle3_f32_rope.restype = ctypes.c_int
    L.eagle3_f32_rope.argtypes = [_i64, _i32, _i32, _p, _i64, _p, _f32, _p]
    L.eagle3_f32_gather.restype = ctypes.c_int
    L.eagle3_f32_gather.argtypes = [_i64, _i64, _p, _p, _p, _i64, _p]
    L.eagle3_f32_argmax.restype = ctypes.c_int
    L.eagle3_f32_argmax.argtypes = [_i64, _i64, _p, _p, _p]
    L.eagle3_f32_attn.restype = ctypes.c_int
    L.eagle3_f32_attn.argtypes = [P(F32AttnArgs), _p]


def status_string(status):
    try:
        return lib().eagle3_status_string(int(status)).decode()
    except Exception:
        return "unknown"


# ----------------------------------------------------------------------------- helpers
def _ptr(t, dtype=None, name="tensor"):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def _check(status, what):
    if status != 0:
        raise Eagle3Error(status, what)


def _workspace(nbytes, device):
    if nbytes == 0:
        return None
    return torch.empty(nbytes, dtype=torch.uint8, device=device)


# ----------------------------------------------------------------------------- entry points
def eagle3_accept(mode, target_logits, tokens, parents, accept_len, path, emitted, next_root, *,
                  draft_logits=None, temperature=1.0, seed=0, step=0, dev_status=None, step_counter=None,
                  workspace=None, stream=None):
    """Acceptance of a verified tree.  target_logits [B, N, V] fp32; tokens / parents [B, N]
    int32; outputs accept_len [B], path / emitted [B, W], next_root [B] int32."""
    B, N, V = target_logits.shape
    a = AcceptArgs(mode=int(mode), batch=B, n_nodes=N, vocab=V, max_path=path.shape[1],
                   temperature=float(temperature), seed=int(seed), step=int(step),
                   target_logits=_ptr(target_logits, torch.float32, "target_logits"),
                   draft_logits=_ptr(draft_logits, torch.float32, "draft_logits"),
                   tokens=_ptr(tokens, torch.int32, "tokens"), parents=_ptr(parents, torch.int32, "parents"),
                   accept_len=_ptr(accept_len, torch.int32, "accept_len"), path=_ptr(path, torch.int32, "path"),
                   emitted=_ptr(emitted, torch.int32, "emitted"),
                   next_root=_ptr(next_root, torch.int32, "next_root"),
                   dev_status=_ptr(dev_status, torch.int32, "dev_status"),
                   step_counter=_ptr(step_counter, torch.int64, "step_counter"))
    if tuple(tokens.shape) != (B, N) or tuple(parents.shape) != (B, N):
        raise ValueError("tokens and parents must be [B, N]")
    if emitted.shape != path.shape or accept_len.numel() != B or next_root.numel() != B:
        raise ValueError("output shapes do not match the batch")
    L = lib()
    need = L.eagle3_accept_workspace_size(ctypes.byref(a))
    if workspace is None:
        workspace = _workspace(need, target_logits.device)
    ws_ptr = None if workspace is None else workspace.data_ptr()
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(L.eagle3_accept(ctypes.byref(a), ws_ptr, ws_bytes, _stream(stream)), "eagle3_accept")


def accept_lazy_args(mode, hidden_states, lm_head, tokens, parents, accept_len, path, emitted, next_root, *,
                     temperature=1.0, seed=0, step=0, dev_status=None, step_counter=None, dbg_level_logits=None):
    """AcceptLazyArgs: hidden_states [B, N, d] bf16 (final-normed), lm_head [V, d] bf16."""
    B, N, d = hidden_states.shape
    V = lm_head.shape[0]
    bf = torch.bfloat16
    if lm_head.shape[1] != d or tuple(tokens.shape) != (B, N) or tuple(parents.shape) != (B, N):
        raise ValueError("shapes: hidden_states [B, N, d], lm_head [V, d], tokens / parents [B, N]")
    acc = AcceptArgs(mode=int(mode), batch=B, n_nodes=N, vocab=V, max_path=path.shape[1],
                     temperature=float(temperature), seed=int(seed), step=int(step), target_logits=None,
                     draft_logits=None, tokens=_ptr(tokens, torch.int32, "tokens"),
                     parents=_ptr(parents, torch.int32, "parents"), accept_len=_ptr(accept_len, torch.int32, "accept_len"),
                     path=_ptr(path, torch.int32, "path"), emitted=_ptr(emitted, torch.int32, "emitted"),
                     next_root=_ptr(next_root, torch.int32, "next_root"),
                     dev_status=_ptr(dev_status, torch.int32, "dev_status"),
                     step_counter=_ptr(step_counter, torch.int64, "step_counter"))
    return AcceptLazyArgs(accept=acc, hidden=d, hidden_states=_ptr(hidden_states, bf, "hidden_states"),
                          lm_head=_ptr(lm_head, bf, "lm_head"),
                          dbg_level_logits=_ptr(dbg_level_logits, torch.float32, "dbg_level_logits"))


def eagle3_accept_lazy(mode, hidden_states, lm_head, tokens, parents, accept_len, path, emitted, next_root, *,
                       temperature=1.0, seed=0, step=0, dev_status=None, step_counter=None, dbg_level_logits=None,
                       workspace=None, stream=None):
    """Acceptance with a lazy target LM head (GREEDY or TOPK): logits only for the visited nodes."""
    a = accept_lazy_args(mode, hidden_states, lm_head, tokens, parents, accept_len, path, emitted, next_root,
                         temperature=temperature, seed=seed, step=step, dev_status=dev_status,
                         step_counter=step_counter, dbg_level_logits=dbg_level_logits)
    L = lib()
    need = L.eagle3_accept_lazy_workspace_size(ctypes.byref(a))
    if workspace is None:
        workspace = _workspace(need, hidden_states.device)
    ws_ptr = None if workspace is None else workspace.data_ptr()
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(L.eagle3_accept_lazy(ctypes.byref(a), ws_ptr, ws_bytes, _stream(stream)), "eagle3_accept_lazy")


def eagle3_compact_kv(k_cache, v_cache, tree_k, tree_v, path, accept_len, prefix_len, slot_map, *,
                      aux_tree=None, aux_out=None, committed=None, tree_node_stride=0, tree_layer_stride=0,
                      dev_status=None, stream=None, block_table=None, block_size=0):
    """k_cache / v_cache [layers, B, Hkv, S_max, D] (bf16 or fp32), or with block_table [B, max_blocks]
    paged pools [layers, n_slots, Hkv, D]; tree_k / tree_v: [layers, B, N, Hkv, D] tensors, or flat
    views into fused QKV buffers described by tree_node_stride / tree_layer_stride (elements; then
    pass tree_k / tree_v as 1-D tensors starting at the first key / value element); path / slot_map
    [B, W]; accept_len, prefix_len [B] int32; aux_tree [B, N, A], aux_out [B, W, A]."""
    paged = block_table is not None
    if paged:
        layers, n_slots, Hkv, D = k_cache.shape
        B, S = path.shape[0], 0
    else:
        layers, B, Hkv, S, D = k_cache.shape
        n_slots = 0
    if tree_k.dim() == 5:
        N = tree_k.shape[2]
        if tuple(tree_k.shape) != (layers, B, N, Hkv, D) or tree_v.shape != tree_k.shape:
            raise ValueError("cache / tree shapes do not match")
        tls, tns = B * N * Hkv * D, Hkv * D
    else:
        if not (tree_node_stride and tree_layer_stride):
            raise ValueError("flat tree_k / tree_v need tree_node_stride and tree_layer_stride")
        tls, tns = int(tree_layer_stride), int(tree_node_stride)
        N = (tls // tns) // B
    if tree_k.dtype != k_cache.dtype or v_cache.dtype != k_cache.dtype or tree_v.dtype != k_cache.dtype:
        raise TypeError("caches and tree K/V must share one dtype")
    if v_cache.shape != k_cache.shape:
        raise ValueError("k_cache and v_cache differ in shape")
    A = 0 if aux_tree is None else aux_tree.shape[-1]
    a = CompactArgs(n_layers=layers, batch=B, n_nodes=N, n_kv_heads=Hkv, head_dim=D,
                    elem_bytes=k_cache.element_size(), s_max=S, max_path=path.shape[1],
                    cache_layer_stride=(n_slots if paged else B * S) * Hkv * D, tree_layer_stride=tls,
                    tree_node_stride=tns,
                    k_cache=_ptr(k_cache, None, "k_cache"), v_cache=_ptr(v_cache, None, "v_cache"),
                    tree_k=tree_k.data_ptr(), tree_v=tree_v.data_ptr(),
                    path=_ptr(path, torch.int32, "path"), accept_len=_ptr(accept_len, torch.int32, "accept_len"),
                    prefix_len=_ptr(prefix_len, torch.int32, "prefix_len"),
                    slot_map=_ptr(slot_map, torch.int32, "slot_map"),
                    committed=_ptr(committed, torch.int32, "committed"), aux_dim=A,
                    aux_tree=_ptr(aux_tree, None, "aux_tree"), aux_out=_ptr(aux_out, None, "aux_out"),
                    dev_status=_ptr(dev_status, torch.int32, "dev_status"),
                    block_table=_ptr(block_table, torch.int32, "block_table"),
                    max_blocks=block_table.shape[1] if paged else 0, block_size=int(block_size) if paged else 0,
                    n_slots=n_slots)
    for t in (tree_k, tree_v):
        if not t.is_cuda:
            raise ValueError("tree_k / tree_v must be CUDA tensors")
    _check(lib().eagle3_compact_kv(ctypes.byref(a), _stream(stream)), "eagle3_compact_kv")


def _view_ptr(t, dtype, name):
    """Data pointer of a (possibly strided) view whose innermost dimension is contiguous."""
    if not t.is_cuda or t.dtype != dtype or t.stride(-1) != 1:
        raise ValueError(f"{name} must be a {dtype} CUDA tensor with a contiguous last dimension")
    return t.data_ptr()


def verify_attn_args(q, tree_k, tree_v, k_cache, v_cache, parents, prefix_len, out, *, max_prefix_len,
                     lse=None, rope_theta=500000.0, sm_scale=0.0, num_splits=0, dev_status=None, qk_rotated=False,
                     block_table=None, block_size=0):
    """q [B, N, Hq, D] and tree_k / tree_v [B, N, Hkv, D] may be node-strided views (e.g. slices of a
    fused [B, N, (Hq + 2 Hkv) * D] projection output); everything else is dense.  qk_rotated: q and
    tree_k already carry RoPE at prefix_len + depth (EPI_BF16_ROPE projection).  Paged cache:
    block_table [B, max_blocks] int32 and k_cache / v_cache pools [n_slots, Hkv, D]."""
    B, N, Hq, D = q.shape
    Hkv = tree_k.shape[2]
    if block_table is not None:
        n_slots = k_cache.shape[0]
        S = 0
        cache_shape = (n_slots, Hkv, D)
        if block_table.dim() != 2 or block_table.shape[0] != B:
            raise ValueError("block_table must be [B, max_blocks]")
    else:
        S = k_cache.shape[2]
        cache_shape = (B, Hkv, S, D)
    for name, t, shape in (("tree_k", tree_k, (B, N, Hkv, D)), ("tree_v", tree_v, (B, N, Hkv, D)),
                           ("k_cache", k_cache, cache_shape), ("v_cache", v_cache, cache_shape),
                           ("out", out, (B, N, Hq, D)), ("parents", parents, (B, N))):
        if tuple(t.shape) != shape:
            raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {shape}")
    bf = torch.bfloat16
    qs = q.stride()
    ks = tree_k.stride()
    if qs[3] != 1 or qs[2] != D or qs[0] != N * qs[1]:
        raise ValueError("q must be node-strided with dense heads")
    if ks[3] != 1 or ks[2] != D or ks[0] != N * ks[1] or tree_v.stride() != tree_k.stride():
        raise ValueError("tree_k / tree_v must share one node stride with dense heads")
    return VerifyAttnArgs(batch=B, n_nodes=N, n_heads=Hq, n_kv_heads=Hkv, head_dim=D, s_max=S,
                          max_prefix_len=int(max_prefix_len), num_splits=int(num_splits),
                          q_node_stride=qs[1], kv_node_stride=ks[1],
                          rope_theta=float(rope_theta), sm_scale=float(sm_scale),
                          q=_view_ptr(q, bf, "q"), tree_k=_view_ptr(tree_k, bf, "tree_k"),
                          tree_v=_view_ptr(tree_v, bf, "tree_v"),
                          k_cache=_ptr(k_cache, bf, "k_cache"), v_cache=_ptr(v_cache, bf, "v_cache"),
                          parents=_ptr(parents, torch.int32, "parents"),
                          prefix_len=_ptr(prefix_len, torch.int32, "prefix_len"),
                          out=_ptr(out, bf, "out"), lse=_ptr(lse, torch.float32, "lse"),
                          dev_status=_ptr(dev_status, torch.int32, "dev_status"), qk_rotated=1 if qk_rotated else 0,
                          block_table=_ptr(block_table, torch.int32, "block_table"),
                          max_blocks=0 if block_table is None else block_table.shape[1],
                          block_size=int(block_size) if block_table is not None else 0,
                          n_slots=0 if block_table is None else k_cache.shape[0])


def eagle3_verify_attn_workspace_size(args):
    return lib().eagle3_verify_attn_workspace_size(ctypes.byref(args))


def eagle3_verify_attn(q, tree_k, tree_v, k_cache, v_cache, parents, prefix_len, out, *, max_prefix_len,
                       lse=None, rope_theta=500000.0, sm_scale=0.0, num_splits=0, dev_status=None,
                       workspace=None, stream=None, qk_rotated=False, block_table=None, block_size=0):
    """Tree-masked verify attention for one layer (bf16, head_dim 128); rotates tree_k in place
    unless qk_rotated (q and tree_k already rotated).  With block_table the caches are paged pools."""
    a = verify_attn_args(q, tree_k, tree_v, k_cache, v_cache, parents, prefix_len, out,
                         max_prefix_len=max_prefix_len, lse=lse, rope_theta=rope_theta, sm_scale=sm_scale,
                         num_splits=num_splits, dev_status=dev_status, qk_rotated=qk_rotated,
                         block_table=block_table, block_size=block_size)
    L = lib()
    need = L.eagle3_verify_attn_workspace_size(ctypes.byref(a))
    if workspace is None:
        workspace = _workspace(need, q.device)
    ws_ptr = None if workspace is None else workspace.data_ptr()
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(L.eagle3_verify_attn(ctypes.byref(a), ws_ptr, ws_bytes, _stream(stream)), "eagle3_verify_attn")


def eagle3_test_verify_attn_timeout(q, tree_k, tree_v, k_cache, v_cache, parents, prefix_len, out, *,
                                    max_prefix_len, stall_tile, wait_limit_cycles, num_splits=0, dev_status=None,
                                    workspace=None, stream=None, qk_rotated=False):
    """Test hook (include/eagle3_testing.h): eagle3_verify_attn with prefix tile `stall_tile` never
    loaded and every bounded wait limited to wait_limit_cycles, so the timeout path runs."""
    a = verify_attn_args(q, tree_k, tree_v, k_cache, v_cache, parents, prefix_len, out,
                         max_prefix_len=max_prefix_len, num_splits=num_splits, dev_status=dev_status,
                         qk_rotated=qk_rotated)
    L = lib()
    need = L.eagle3_verify_attn_workspace_size(ctypes.byref(a))
    if workspace is None:
        workspace = _workspace(need, q.device)
    ws_ptr = None if workspace is None else workspace.data_ptr()
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(L.eagle3_test_verify_attn_timeout(ctypes.byref(a), ws_ptr, ws_bytes, int(stall_tile),
                                             int(wait_limit_cycles), _stream(stream)),
           "eagle3_test_verify_attn_timeout")


def eagle3_spec_decode_metadata(cu_num_scheduled_tokens, num_draft_tokens, cu_num_draft_tokens, logits_indices,
                                target_logits_indices, bonus_logits_indices, num_rows, *, dev_status=None, stream=None):
    """Index bookkeeping of a ragged verify batch (int32 CUDA tensors; logits_indices and
    target_logits_indices have the capacity max_rows)."""
    R = cu_num_scheduled_tokens.numel()
    i32 = torch.int32
    a = SpecDecodeMetadataArgs(n_requests=R, max_rows=logits_indices.numel(),
                               cu_num_scheduled_tokens=_ptr(cu_num_scheduled_tokens, i32, "cu_num_scheduled_tokens"),
                               num_draft_tokens=_ptr(num_draft_tokens, i32, "num_draft_tokens"),
                               cu_num_draft_tokens=_ptr(cu_num_draft_tokens, i32, "cu_num_draft_tokens"),
                               logits_indices=_ptr(logits_indices, i32, "logits_indices"),
                               target_logits_indices=_ptr(target_logits_indices, i32, "target_logits_indices"),
                               bonus_logits_indices=_ptr(bonus_logits_indices, i32, "bonus_logits_indices"),
                               num_rows=_ptr(num_rows, i32, "num_rows"), dev_status=_ptr(dev_status, i32, "dev_status"))
    if target_logits_indices.numel() != logits_indices.numel():
        raise ValueError("logits_indices and target_logits_indices share the capacity max_rows")
    _check(lib().eagle3_spec_decode_metadata(ctypes.byref(a), _stream(stream)), "eagle3_spec_decode_metadata")


def eagle3_ttt_attn(q, k, v, out, *, sm_scale=0.0, dev_status=None, workspace=None, stream=None):
    """Training-time-test attention: q [Bt, T, Hq, D], k / v [S, Bt, T, Hkv, D] (step 0 native, then
    the simulated steps), out [Bt, T, Hq, D]; bf16, rotated."""
    Bt, T, Hq, D = q.shape
    S, _, _, Hkv, _ = k.shape
    bf = torch.bfloat16
    if tuple(k.shape) != (S, Bt, T, Hkv, D) or v.shape != k.shape or out.shape != q.shape:
        raise ValueError("shapes: q / out [Bt, T, Hq, D], k / v [S, Bt, T, Hkv, D]")
    a = TttAttnArgs(batch=Bt, seq_len=T, n_heads=Hq, n_kv_heads=Hkv, head_dim=D, n_steps=S, sm_scale=float(sm_scale),
                    q=_ptr(q, bf, "q"), k=_ptr(k, bf, "k"), v=_ptr(v, bf, "v"), out=_ptr(out, bf, "out"),
                    dev_status=_ptr(dev_status, torch.int32, "dev_status"))
    L = lib()
    need = L.eagle3_ttt_attn_workspace_size(ctypes.byref(a))
    if workspace is None:
        workspace = _workspace(need, q.device)
    ws_ptr = None if workspace is None else workspace.data_ptr()
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(L.eagle3_ttt_attn(ctypes.byref(a), ws_ptr, ws_bytes, _stream(stream)), "eagle3_ttt_attn")


def eagle3_chain_verify(logits, draft_tokens, cu_num_draft_tokens, output_tokens, *, is_greedy=None, num_accepted=None,
                        temperature=1.0, seed=0, step=0, dev_status=None, step_counter=None, stream=None):
    """Chain rejection sampling of a ragged batch: logits [rows, V] fp32, draft_tokens [sum d] and
    cu_num_draft_tokens [R] int32, output_tokens [R, K + 1] int32."""
    R, W = output_tokens.shape
    i32 = torch.int32
    a = ChainVerifyArgs(n_requests=R, vocab=logits.shape[1], max_drafts=W - 1, temperature=float(temperature),
                        seed=int(seed), step=int(step), logits=_ptr(logits, torch.float32, "logits"),
                        draft_tokens=_ptr(draft_tokens, i32, "draft_tokens") if draft_tokens.numel() else None,
                        cu_num_draft_tokens=_ptr(cu_num_draft_tokens, i32, "cu_num_draft_tokens"),
                        is_greedy=_ptr(is_greedy, i32, "is_greedy"), output_tokens=_ptr(output_tokens, i32, "output_tokens"),
                        num_accepted=_ptr(num_accepted, i32, "num_accepted"), dev_status=_ptr(dev_status, i32, "dev_status"),
                        step_counter=_ptr(step_counter, torch.int64, "step_counter"))
    if cu_num_draft_tokens.numel() != R:
        raise ValueError("one cu_num_draft_tokens entry per output row")
    _check(lib().eagle3_chain_verify(ctypes.byref(a), _stream(stream)), "eagle3_chain_verify")


def eagle3_linear(x, w, out, *, epilogue=EPI_BF16, w2=None, residual=None, splits=0, dev_status=None,
                  workspace=None, stream=None, rope_cols=0, rope_rows_per_seq=1, rope_theta=500000.0,
                  rope_base=None, rope_depth=None, row_max=None, row_ssq=None, row_ssq_in=None, ssq_dim=0,
                  ssq_eps=1e-5):
    """out = epilogue(x W^T) on the tensor cores.  x [m, k] bf16, w (and w2) [n, k] bf16,
    out [m, n] bf16 (fp32 for EPI_F32), residual [m, n] bf16 for EPI_BF16_RESIDUAL.
    EPI_BF16_ROPE rotates columns [0, rope_cols) per 128-wide head at row position
    rope_base[row // rope_rows_per_seq] + rope_depth[row] (int32 device tensors).  row_max (EPI_F32,
    int32 [m] holding the uint32 words, zeroed by the caller): each row's maximum output order key.
    row_ssq (fp32 [ceil(n / 256), m], bf16 epilogues): per row and 256-column block, the sum of
    squares of the bf16 outputs.  row_ssq_in (fp32 [blocks, m]): scale each output row by
    rsqrt(sum / ssq_dim + ssq_eps) before the epilogue (an RMSNorm folded into this projection)."""
    m, k = x.shape
    n = w.shape[0]
    if w.shape[1] != k or (w2 is not None and tuple(w2.shape) != (n, k)):
        raise ValueError("weight shapes do not match x")
    if tuple(out.shape) != (m, n):
        raise ValueError(f"out must be [{m}, {n}]")
    want = torch.float32 if epilogue == EPI_F32 else torch.bfloat16
    bf = torch.bfloat16
    a = LinearArgs(m=m, n=n, k=k, epilogue=int(epilogue), splits=int(splits), ld_x=0, ld_w=0, ld_out=0, ld_res=0,
                   x=_ptr(x, bf, "x"), w=_ptr(w, bf, "w"), w2=_ptr(w2, bf, "w2"), out=_ptr(out, want, "out"),
                   residual=_ptr(residual, bf, "residual"), dev_status=_ptr(dev_status, torch.int32, "dev_status"),
                   rope_cols=int(rope_cols), rope_rows_per_seq=int(rope_rows_per_seq), rope_theta=float(rope_theta),
                   rope_base=_ptr(rope_base, torch.int32, "rope_base"),
                   rope_depth=_ptr(rope_depth, torch.int32, "rope_depth"),
                   row_max=_ptr(row_max, torch.int32, "row_max"), row_ssq=_ptr(row_ssq, torch.float32, "row_ssq"),
                   row_ssq_in=_ptr(row_ssq_in, torch.float32, "row_ssq_in"),
                   ssq_blocks=0 if row_ssq_in is None else int(row_ssq_in.shape[0]), ssq_dim=int(ssq_dim),
                   ssq_eps=float(ssq_eps))
    L = lib()
    need = L.eagle3_linear_workspace_size(ctypes.byref(a))
    if workspace is None:
        workspace = _workspace(need, x.device)
    ws_ptr = None if workspace is None else workspace.data_ptr()
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(L.eagle3_linear(ctypes.byref(a), ws_ptr, ws_bytes, _stream(stream)), "eagle3_linear")


def draft_tree_args(aux, next_tokens, tc, k_cache, v_cache, draft_len, tokens, parents, depth_out, anc_mask, score, *,
                    n_heads, ffn, vocab, depth, top_k, max_draft_len, rope_theta=500000.0, rms_eps=1e-5,
                    dbg_logits=None, dev_status=None, d2t=None):
    B, tc_max, d3 = aux.shape
    Hkv, S, D = k_cache.shape[1:]
    N = tokens.shape[1]
    bf, i32 = torch.bfloat16, torch.int32
    return DraftTreeArgs(batch=B, hidden=d3 // 3, n_heads=n_heads, n_kv_heads=Hkv, head_dim=D, ffn=ffn, vocab=vocab,
                         depth=depth, top_k=top_k, n_nodes=N, tc_max=tc_max, s_max=S, max_draft_len=int(max_draft_len),
                         rope_theta=float(rope_theta), rms_eps=float(rms_eps),
                         aux=_ptr(aux, bf, "aux"), next_tokens=_ptr(next_tokens, i32, "next_tokens"),
                         tc=_ptr(tc, i32, "tc"), draft_k_cache=_ptr(k_cache, bf, "k_cache"),
                         draft_v_cache=_ptr(v_cache, bf, "v_cache"), draft_len=_ptr(draft_len, i32, "draft_len"),
                         tokens=_ptr(tokens, i32, "tokens"), parents=_ptr(parents, i32, "parents"),
                         depth_out=_ptr(depth_out, i32, "depth_out"), anc_mask=_ptr(anc_mask, torch.int64, "anc_mask"),
                         score=_ptr(score, torch.float32, "score"),
                         dbg_logits=_ptr(dbg_logits, torch.float32, "dbg_logits"),
                         dev_status=_ptr(dev_status, i32, "dev_status"),
                         draft_vocab=0 if d2t is None else int(d2t.numel()), d2t=_ptr(d2t, i32, "d2t"))


def draft_weights(w):
    """DraftWeights from a dict of contiguous bf16 CUDA tensors named as in DRAFT_WEIGHT_NAMES."""
    return DraftWeights(**{n: _ptr(w[n], torch.bfloat16, n) for n in DRAFT_WEIGHT_NAMES})


def eagle3_draft_tree_workspace_size(args):
    return lib().eagle3_draft_tree_workspace_size(ctypes.byref(args))


def eagle3_draft_tree(weights, aux, next_tokens, tc, k_cache, v_cache, draft_len, tokens, parents, depth_out,
                      anc_mask, score, *, n_heads, ffn, vocab, depth, top_k, max_draft_len, rope_theta=500000.0,
                      rms_eps=1e-5, dbg_logits=None, dev_status=None, d2t=None, workspace=None, stream=None):
    """Draft head + dynamic tree.  weights: dict of bf16 tensors (see DRAFT_WEIGHT_NAMES);
    aux [B, tc_max, 3d] bf16; next_tokens [B, tc_max] / tc [B] / draft_len [B] int32; caches
    [B, Hkv, S, D] bf16; outputs [B, N] (anc_mask int64 bit patterns of the uint64 masks).
    d2t: optional [Vd] int32 CUDA tensor, the target ids of a reduced draft vocabulary (lm_head is
    then [Vd, d] and dbg_logits rows have Vd entries)."""
    a = draft_tree_args(aux, next_tokens, tc, k_cache, v_cache, draft_len, tokens, parents, depth_out, anc_mask, score,
                        n_heads=n_heads, ffn=ffn, vocab=vocab, depth=depth, top_k=top_k, max_draft_len=max_draft_len,
                        rope_theta=rope_theta, rms_eps=rms_eps, dbg_logits=dbg_logits, dev_status=dev_status, d2t=d2t)
    wts = draft_weights(weights)
    L = lib()
    need = L.eagle3_draft_tree_workspace_size(ctypes.byref(a))
    if workspace is None:
        workspace = _workspace(need, aux.device)
    ws_ptr = None if workspace is None else workspace.data_ptr()
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(L.eagle3_draft_tree(ctypes.byref(wts), ctypes.byref(a), ws_ptr, ws_bytes, _stream(stream)),
           "eagle3_draft_tree")


def eagle3_rmsnorm(x, w, out, *, eps=1e-5, gather=None, tap_out=None, dev_status=None, stream=None):
    """out[r] = w * rmsnorm(x[gather[r] if gather else r]); tap_out[r] = that input row (optional)."""
    rows = out.shape[0]
    dim = w.shape[0]
    bf = torch.bfloat16
    a = RmsnormArgs(rows=rows, dim=dim, n_src=x.shape[0], eps=float(eps), ld_in=x.stride(0), ld_out=out.stride(0),
                    ld_tap=0 if tap_out is None else tap_out.stride(0), input=x.data_ptr(), w=_ptr(w, bf, "w"),
                    gather=_ptr(gather, torch.int32, "gather"), out=out.data_ptr(),
                    tap_out=None if tap_out is None else tap_out.data_ptr(),
                    dev_status=_ptr(dev_status, torch.int32, "dev_status"))
    for name, t in (("x", x), ("out", out), ("tap_out", tap_out)):
        if t is not None and (not t.is_cuda or t.dtype != bf or t.stride(-1) != 1):
            raise ValueError(f"{name} must be a bf16 CUDA tensor with unit inner stride")
    _check(lib().eagle3_rmsnorm(ctypes.byref(a), _stream(stream)), "eagle3_rmsnorm")


def eagle3_verify_attn_noalloc(q, tree_k, tree_v, k_cache, v_cache, parents, prefix_len, out, *, max_prefix_len,
                               lse=None, rope_theta=500000.0, sm_scale=0.0, num_splits=0, dev_status=None,
                               stream=None, qk_rotated=False):
    """eagle3_verify_attn without a workspace: the library's static scratch holds the split partials."""
    a = verify_attn_args(q, tree_k, tree_v, k_cache, v_cache, parents, prefix_len, out,
                         max_prefix_len=max_prefix_len, lse=lse, rope_theta=rope_theta, sm_scale=sm_scale,
                         num_splits=num_splits, dev_status=dev_status, qk_rotated=qk_rotated)
    _check(lib().eagle3_verify_attn_noalloc(ctypes.byref(a), _stream(stream)), "eagle3_verify_attn_noalloc")


# ----------------------------------------------------------------------------- fp32 small-model blocks
def _rows_pitch(t, what):
    """Row pitch (elements) of a 2-D view whose rows are contiguous."""
    if t.dim() != 2 or t.stride(1) != 1:
        raise ValueError(f"{what} must be a 2-D view with contiguous rows")
    return t.stride(0)


def _vptr(t, dtype, name):
    """Pointer of a 2-D row view (rows contiguous, any row pitch), or None."""
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    _rows_pitch(t, name)
    return t.data_ptr()


def eagle3_f32_linear(x, w, out, *, epilogue=F32_EPI_NONE, w2=None, residual=None, stream=None):
    """out = epilogue(x W^T) in fp32; x [m, k], w (and w2) [n, k], out / residual [m, n] row views."""
    m, k = x.shape
    n = w.shape[0]
    a = F32LinearArgs(m=m, n=n, k=k, epilogue=int(epilogue), ld_x=_rows_pitch(x, "x"), ld_out=_rows_pitch(out, "out"),
                      ld_res=0 if residual is None else _rows_pitch(residual, "residual"),
                      x=_vptr(x, torch.float32, "x"), w=_ptr(w, torch.float32, "w"), w2=_ptr(w2, torch.float32, "w2"),
                      residual=_vptr(residual, torch.float32, "residual"), out=_vptr(out, torch.float32, "out"))
    _check(lib().eagle3_f32_linear(ctypes.byref(a), _stream(stream)), "eagle3_f32_linear")


def eagle3_f32_rmsnorm(x, w, out, *, eps=1e-5, gather=None, stream=None):
    rows = out.shape[0] if gather is None else gather.numel()
    dim = w.numel()
    _check(lib().eagle3_f32_rmsnorm(rows, dim, _vptr(x, torch.float32, "x"), _rows_pitch(x, "x"),
                                    _ptr(gather, torch.int32, "gather"), _ptr(w, torch.float32, "w"), eps,
                                    _vptr(out, torch.float32, "out"), _rows_pitch(out, "out"), _stream(stream)),
           "eagle3_f32_rmsnorm")


def eagle3_f32_rope(x, heads, head_dim, pos, *, theta=500000.0, stream=None):
    """x [rows, >= heads * head_dim] row view, rotated in place at positions pos [rows] int32."""
    _check(lib().eagle3_f32_rope(x.shape[0], heads, head_dim, _vptr(x, torch.float32, "x"), _rows_pitch(x, "x"),
                                 _ptr(pos, torch.int32, "pos"), theta, _stream(stream)), "eagle3_f32_rope")


def eagle3_f32_gather(table, idx, out, *, stream=None):
    _check(lib().eagle3_f32_gather(idx.numel(), table.shape[1], _ptr(table, torch.float32, "table"),
                                   _ptr(idx, torch.int32, "idx"), _vptr(out, torch.float32, "out"),
                                   _rows_pitch(out, "out"), _stream(stream)), "eagle3_f32_gather")


def eagle3_f32_argmax(logits, out, *, stream=None):
    _check(lib().eagle3_f32_argmax(logits.shape[0], logits.shape[1], _vptr(logits, torch.float32, "logits"),
                                   _ptr(out, torch.int32, "out"), _stream(stream)), "eagle3_f32_argmax")


def eagle3_f32_attn(q, k_new, v_new, k_cache, v_cache, visible, out, *, n_heads, n_kv_heads, head_dim, cache_len,
                    scale=0.0, stream=None):
    """q [T, >= Hq*D] and k_new / v_new [T, >= Hkv*D] row views (rotated); k_cache / v_cache
    [Hkv, s_max, D]; visible [T] int64 bitmasks over the new rows; out [T, Hq, D]."""
    a = F32AttnArgs(n_rows=q.shape[0], n_heads=n_heads, n_kv_heads=n_kv_heads, head_dim=head_dim,
                    cache_len=int(cache_len), s_max=k_cache.shape[1], scale=float(scale),
                    ld_q=_rows_pitch(q, "q"), ld_kv=_rows_pitch(k_new, "k_new"),
                    q=_vptr(q, torch.float32, "q"), k_new=_vptr(k_new, torch.float32, "k_new"),
                    v_new=_vptr(v_new, torch.float32, "v_new"), k_cache=_ptr(k_cache, torch.float32, "k_cache"),
                    v_cache=_ptr(v_cache, torch.float32, "v_cache"), visible=_ptr(visible, torch.int64, "visible"),
                    out=_ptr(out, torch.float32, "out"))
    if _rows_pitch(v_new, "v_new") != a.ld_kv:
        raise ValueError("k_new and v_new must share a row pitch")
    _check(lib().eagle3_f32_attn(ctypes.byref(a), _stream(stream)), "eagle3_f32_attn")
