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
                ("accept_len", _p), ("path", _p), ("emitted", _p), ("next_root", _p), ("dev_status", _p)]


class CompactArgs(ctypes.Structure):
    _fields_ = [("n_layers", _i32), ("batch", _i32), ("n_nodes", _i32), ("n_kv_heads", _i32),
                ("head_dim", _i32), ("elem_bytes", _i32), ("s_max", _i32), ("max_path", _i32),
                ("cache_layer_stride", _i64), ("tree_layer_stride", _i64),
                ("k_cache", _p), ("v_cache", _p), ("tree_k", _p), ("tree_v", _p),
                ("path", _p), ("accept_len", _p), ("prefix_len", _p), ("slot_map", _p),
                ("aux_dim", _i32), ("aux_tree", _p), ("aux_out", _p), ("dev_status", _p)]


class VerifyAttnArgs(ctypes.Structure):
    _fields_ = [("batch", _i32), ("n_nodes", _i32), ("n_heads", _i32), ("n_kv_heads", _i32),
                ("head_dim", _i32), ("s_max", _i32), ("max_prefix_len", _i32), ("num_splits", _i32),
                ("rope_theta", _f32), ("sm_scale", _f32),
                ("q", _p), ("tree_k", _p), ("tree_v", _p), ("k_cache", _p), ("v_cache", _p),
                ("parents", _p), ("prefix_len", _p), ("out", _p), ("lse", _p), ("dev_status", _p)]


class LinearArgs(ctypes.Structure):
    _fields_ = [("m", _i32), ("n", _i32), ("k", _i32), ("epilogue", _i32), ("splits", _i32),
                ("ld_x", _i64), ("ld_w", _i64), ("ld_out", _i64), ("ld_res", _i64),
                ("x", _p), ("w", _p), ("w2", _p), ("out", _p), ("residual", _p), ("dev_status", _p)]


EPI_BF16, EPI_F32, EPI_BF16_RESIDUAL, EPI_SWIGLU = 0, 1, 2, 3


def _declare(L):
    P = ctypes.POINTER
    L.eagle3_status_string.restype = ctypes.c_char_p
    L.eagle3_status_string.argtypes = [ctypes.c_int]
    L.eagle3_version.restype = ctypes.c_int
    L.eagle3_accept_workspace_size.restype = ctypes.c_size_t
    L.eagle3_accept_workspace_size.argtypes = [P(AcceptArgs)]
    L.eagle3_accept.restype = ctypes.c_int
    L.eagle3_accept.argtypes = [P(AcceptArgs), _p, ctypes.c_size_t, _p]
    L.eagle3_compact_kv.restype = ctypes.c_int
    L.eagle3_compact_kv.argtypes = [P(CompactArgs), _p]
    L.eagle3_verify_attn_workspace_size.restype = ctypes.c_size_t
    L.eagle3_verify_attn_workspace_size.argtypes = [P(VerifyAttnArgs)]
    L.eagle3_verify_attn.restype = ctypes.c_int
    L.eagle3_verify_attn.argtypes = [P(VerifyAttnArgs), _p, ctypes.c_size_t, _p]
    L.eagle3_linear_workspace_size.restype = ctypes.c_size_t
    L.eagle3_linear_workspace_size.argtypes = [P(LinearArgs)]
    L.eagle3_linear.restype = ctypes.c_int
    L.eagle3_linear.argtypes = [P(LinearArgs), _p, ctypes.c_size_t, _p]


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
                  draft_logits=None, temperature=1.0, seed=0, step=0, dev_status=None,
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
                   dev_status=_ptr(dev_status, torch.int32, "dev_status"))
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


def eagle3_compact_kv(k_cache, v_cache, tree_k, tree_v, path, accept_len, prefix_len, slot_map, *,
                      aux_tree=None, aux_out=None, dev_status=None, stream=None):
    """k_cache / v_cache [layers, B, Hkv, S_max, D]; tree_k / tree_v [layers, B, N, Hkv, D]
    (bf16 or fp32, same dtype); path / slot_map [B, W]; accept_len, prefix_len [B] int32."""
    layers, B, Hkv, S, D = k_cache.shape
    N = tree_k.shape[2]
    if tree_k.dtype != k_cache.dtype or v_cache.dtype != k_cache.dtype or tree_v.dtype != k_cache.dtype:
        raise TypeError("caches and tree K/V must share one dtype")
    if tuple(tree_k.shape) != (layers, B, N, Hkv, D) or tree_v.shape != tree_k.shape or v_cache.shape != k_cache.shape:
        raise ValueError("cache / tree shapes do not match")
    A = 0 if aux_tree is None else aux_tree.shape[-1]
    a = CompactArgs(n_layers=layers, batch=B, n_nodes=N, n_kv_heads=Hkv, head_dim=D,
                    elem_bytes=k_cache.element_size(), s_max=S, max_path=path.shape[1],
                    cache_layer_stride=B * Hkv * S * D, tree_layer_stride=B * N * Hkv * D,
                    k_cache=_ptr(k_cache, None, "k_cache"), v_cache=_ptr(v_cache, None, "v_cache"),
                    tree_k=_ptr(tree_k, None, "tree_k"), tree_v=_ptr(tree_v, None, "tree_v"),
                    path=_ptr(path, torch.int32, "path"), accept_len=_ptr(accept_len, torch.int32, "accept_len"),
                    prefix_len=_ptr(prefix_len, torch.int32, "prefix_len"),
                    slot_map=_ptr(slot_map, torch.int32, "slot_map"), aux_dim=A,
                    aux_tree=_ptr(aux_tree, None, "aux_tree"), aux_out=_ptr(aux_out, None, "aux_out"),
                    dev_status=_ptr(dev_status, torch.int32, "dev_status"))
    _check(lib().eagle3_compact_kv(ctypes.byref(a), _stream(stream)), "eagle3_compact_kv")


def verify_attn_args(q, tree_k, tree_v, k_cache, v_cache, parents, prefix_len, out, *, max_prefix_len,
                     lse=None, rope_theta=500000.0, sm_scale=0.0, num_splits=0, dev_status=None):
    B, N, Hq, D = q.shape
    Hkv = tree_k.shape[2]
    S = k_cache.shape[2]
    for name, t, shape in (("tree_k", tree_k, (B, N, Hkv, D)), ("tree_v", tree_v, (B, N, Hkv, D)),
                           ("k_cache", k_cache, (B, Hkv, S, D)), ("v_cache", v_cache, (B, Hkv, S, D)),
                           ("out", out, (B, N, Hq, D)), ("parents", parents, (B, N))):
        if tuple(t.shape) != shape:
            raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {shape}")
    bf = torch.bfloat16
    return VerifyAttnArgs(batch=B, n_nodes=N, n_heads=Hq, n_kv_heads=Hkv, head_dim=D, s_max=S,
                          max_prefix_len=int(max_prefix_len), num_splits=int(num_splits),
                          rope_theta=float(rope_theta), sm_scale=float(sm_scale),
                          q=_ptr(q, bf, "q"), tree_k=_ptr(tree_k, bf, "tree_k"), tree_v=_ptr(tree_v, bf, "tree_v"),
                          k_cache=_ptr(k_cache, bf, "k_cache"), v_cache=_ptr(v_cache, bf, "v_cache"),
                          parents=_ptr(parents, torch.int32, "parents"),
                          prefix_len=_ptr(prefix_len, torch.int32, "prefix_len"),
                          out=_ptr(out, bf, "out"), lse=_ptr(lse, torch.float32, "lse"),
                          dev_status=_ptr(dev_status, torch.int32, "dev_status"))


def eagle3_verify_attn_workspace_size(args):
    return lib().eagle3_verify_attn_workspace_size(ctypes.byref(args))


def eagle3_verify_attn(q, tree_k, tree_v, k_cache, v_cache, parents, prefix_len, out, *, max_prefix_len,
                       lse=None, rope_theta=500000.0, sm_scale=0.0, num_splits=0, dev_status=None,
                       workspace=None, stream=None):
    """Tree-masked verify attention for one layer (bf16, head_dim 128); rotates tree_k in place."""
    a = verify_attn_args(q, tree_k, tree_v, k_cache, v_cache, parents, prefix_len, out,
                         max_prefix_len=max_prefix_len, lse=lse, rope_theta=rope_theta, sm_scale=sm_scale,
                         num_splits=num_splits, dev_status=dev_status)
    L = lib()
    need = L.eagle3_verify_attn_workspace_size(ctypes.byref(a))
    if workspace is None:
        workspace = _workspace(need, q.device)
    ws_ptr = None if workspace is None else workspace.data_ptr()
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(L.eagle3_verify_attn(ctypes.byref(a), ws_ptr, ws_bytes, _stream(stream)), "eagle3_verify_attn")


def eagle3_linear(x, w, out, *, epilogue=EPI_BF16, w2=None, residual=None, splits=0, dev_status=None,
                  workspace=None, stream=None):
    """out = epilogue(x W^T) on the tensor cores.  x [m, k] bf16, w (and w2) [n, k] bf16,
    out [m, n] bf16 (fp32 for EPI_F32), residual [m, n] bf16 for EPI_BF16_RESIDUAL."""
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
                   residual=_ptr(residual, bf, "residual"), dev_status=_ptr(dev_status, torch.int32, "dev_status"))
    L = lib()
    need = L.eagle3_linear_workspace_size(ctypes.byref(a))
    if workspace is None:
        workspace = _workspace(need, x.device)
    ws_ptr = None if workspace is None else workspace.data_ptr()
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(L.eagle3_linear(ctypes.byref(a), ws_ptr, ws_bytes, _stream(stream)), "eagle3_linear")
