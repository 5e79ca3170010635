"""One EAGLE-3 draft-and-verify step, composed from the library's C entry points.

Sources: "EAGLE-3: Engineering Implementation of LLM Inference Acceleration", section XI (the
loop: catch-up of the committed positions into the draft cache, drafting, verification by the
target, acceptance, commit), "Advanced speculative decoding: tree drafts and EAGLE", section
"Implementation" (the target runs the whole tree in one pass with the tree mask, every node at
prefix length + depth; only the accepted path's K/V is appended to the cache) and "Speculative
Decoding (EAGLE3) in the vLLM Neuron Framework", section "Auxiliary Hidden State Extraction" (the
target's hidden states entering the tapped layers are kept for the draft's next catch-up).

A step, every part of it a libeagle3 call on the caller's stream:
  eagle3_draft_tree     catch-up rows -> draft cache; dynamic top-k tree (tokens, parents, depth)
  target verify forward, per layer l:
      eagle3_rmsnorm    attn norm (layer 0 gathers the embedding rows of the tree tokens and keeps
                        them as the residual stream; a tapped layer copies the stream entering it
                        into that tap's third of the aux rows)
      eagle3_linear     fused QKV projection; q and k leave it rotated at prefix_len + depth
      eagle3_verify_attn tree-masked attention over the layer's cache and the tree
      eagle3_linear     O projection + residual, post-norm, SwiGLU gate/up, down + residual
                        (fold_norms: the RMSNorms before QKV, gate/up and the LM head are folded
                        into those projections: the O and down projections emit each row's sum of
                        squares, the next projection reads the raw residual stream with the norm
                        weight folded into its weights and scales its output rows; only layer 0
                        (which gathers the embeddings) and the tapped layers keep a norm kernel)
  eagle3_rmsnorm + eagle3_linear   final norm, LM head (fp32 logits)
  eagle3_accept         greedy walk or lossless rejection sampling over the tree
                        (lazy_head: eagle3_accept_lazy instead of the LM head and eagle3_accept; the
                        head's logits are computed level by level, only for the nodes the walk visits)
  eagle3_compact_kv     the accepted path's K/V of every layer into the caches (read in place
                        from the fused QKV outputs), the path's aux rows and tokens into the next
                        step's catch-up inputs, prefix_len += accepted + 1

The outputs of one step are the inputs of the next (a real decoding loop): emitted tokens go to
``next_tok`` (the last one is the next root), the gathered aux rows to ``aux_in`` and the committed
count to ``tc``.  Every argument struct is built once; the ops can be issued eagerly or captured
into a CUDA graph.  Nothing here computes: Python only marshals pointers.
"""
import ctypes

import torch

from . import _lib

TARGET_LAYER_WEIGHTS = ("wqkv", "wo", "wg", "wu", "wd", "norm1", "norm2")


class SpeculativeStep:
    """Device state and the prepared C calls of one draft-and-verify step.

    cfg keys: layers, d, Hq, Hkv, D, F, V, taps (three layer ids > 0), B, N, depth, top_k, W (path
    width, >= depth + 1), mode (GREEDY, or TOPK: the tree's children are the draft's top-k tokens, so
    the sampled-children mode does not apply), temperature, seed, rope_theta, eps.
    target: dict with embed [V, d], lm_head [V, d], final_norm [d] and per-layer lists of
    wqkv [(Hq + 2 Hkv) D, d], wo [d, Hq D], wg / wu [F, d], wd [d, F], norm1 / norm2 [d] (bf16).
    draft: dict of the eagle3_draft_tree weights (bf16; see _lib.DRAFT_WEIGHT_NAMES).
    s_max: cache capacity; max_prefix: host bound on every prefix length over the run (the kernels
    read the exact lengths from device memory, so one set of prepared calls serves every step).

    The caller fills the caches and the per-sequence state (prefix_len, draft_len, aux_in,
    next_tok, tc) before the first step; the buffers are attributes of this object."""

    def __init__(self, cfg, target, draft, s_max, max_prefix, dev, fused_rope=True, d2t=None, fold_norms=False):
        c = self.cfg = dict(cfg)
        if len(c["taps"]) != 3 or min(c["taps"]) < 1 or max(c["taps"]) >= c["layers"]:
            raise ValueError("three aux taps in [1, layers) are needed")
        if c["W"] < c["depth"] + 1:
            raise ValueError("the path width must hold depth + 1 nodes")
        self.target, self.draft_w, self.dev = target, draft, dev
        self.fused_rope = fused_rope
        self.fold_norms = bool(fold_norms)
        self.S, self.max_prefix = int(s_max), int(max_prefix)
        self.d2t = d2t
        B, N, d, V, D = c["B"], c["N"], c["d"], c["V"], c["D"]
        Hq, Hkv, F, Lyr, W = c["Hq"], c["Hkv"], c["F"], c["layers"], c["W"]
        self.qkv_w = (Hq + 2 * Hkv) * D
        bf, i32 = torch.bfloat16, torch.int32
        S = self.S
        # caches and per-sequence state
        self.k_cache = torch.zeros(Lyr, B, Hkv, S, D, device=dev, dtype=bf)
        self.v_cache = torch.zeros_like(self.k_cache)
        self.dk_cache = torch.zeros(B, Hkv, S, D, device=dev, dtype=bf)
        self.dv_cache = torch.zeros_like(self.dk_cache)
        self.prefix_len = torch.zeros(B, dtype=i32, device=dev)
        self.draft_len = torch.zeros(B, dtype=i32, device=dev)
        self.aux_in = torch.zeros(B, W, 3 * d, device=dev, dtype=bf)
        self.next_tok = torch.zeros(B, W, dtype=i32, device=dev)
        self.tc = torch.ones(B, dtype=i32, device=dev)
        # per-step buffers
        self.tokens = torch.empty(B, N, dtype=i32, device=dev)
        self.parents = torch.empty(B, N, dtype=i32, device=dev)
        self.depth = torch.empty(B, N, dtype=i32, device=dev)
        self.anc = torch.empty(B, N, dtype=torch.int64, device=dev)
        self.score = torch.empty(B, N, dtype=torch.float32, device=dev)
        R = B * N
        self.x = torch.empty(R, d, device=dev, dtype=bf)
        self.h = torch.empty(R, d, device=dev, dtype=bf)
        self.qkv = torch.empty(Lyr, R, self.qkv_w, device=dev, dtype=bf)
        self.attn = torch.empty(R, Hq * D, device=dev, dtype=bf)
        self.act = torch.empty(R, F, device=dev, dtype=bf)
        self.aux_tree = torch.empty(R, 3 * d, device=dev, dtype=bf)
        self.logits = None                 # [R, V] fp32, allocated by a full-head prepare()
        self.lazy_head = False
        self.accept_len = torch.empty(B, dtype=i32, device=dev)
        self.path = torch.empty(B, W, dtype=i32, device=dev)
        self.next_root = torch.empty(B, dtype=i32, device=dev)
        self.slot_map = torch.empty(B, W, dtype=i32, device=dev)
        self.dev_status = torch.zeros(1, dtype=i32, device=dev)
        # folded RMSNorm: per row and 256-column block, the sum of squares of the residual stream as
        # stored (after the O projection, and after the down projection)
        self.ssq_blocks = (d + 255) // 256
        self.ssq_mid = torch.zeros(self.ssq_blocks, R, dtype=torch.float32, device=dev)
        self.ssq_next = torch.zeros(self.ssq_blocks, R, dtype=torch.float32, device=dev)
        self._folded = None
        self.step_counter = torch.zeros(1, dtype=torch.int64, device=dev)   # Philox step, advanced on device
        self.draft_ops, self.verify_ops = [], []
        self._keep = []

    # ------------------------------------------------------------------------------ views
    def tree_q(self, layer):
        """[B, N, Hq, D] view of layer's rotated queries inside the fused QKV output."""
        c = self.cfg
        return self.qkv[layer].view(c["B"], c["N"], self.qkv_w)[:, :, : c["Hq"] * c["D"]].unflatten(2, (c["Hq"], c["D"]))

    def tree_k(self, layer):
        c = self.cfg
        lo, hi = c["Hq"] * c["D"], (c["Hq"] + c["Hkv"]) * c["D"]
        return self.qkv[layer].view(c["B"], c["N"], self.qkv_w)[:, :, lo:hi].unflatten(2, (c["Hkv"], c["D"]))

    def tree_v(self, layer):
        c = self.cfg
        lo = (c["Hq"] + c["Hkv"]) * c["D"]
        return self.qkv[layer].view(c["B"], c["N"], self.qkv_w)[:, :, lo:].unflatten(2, (c["Hkv"], c["D"]))

    # ------------------------------------------------------------------------------ preparation
    def prepare(self, ws_linear_bytes=512 << 20, ws_attn_bytes=256 << 20, lazy_head=False):
        """Build every argument struct of the step once.  Ops are (kind, call) pairs; kind names
        the calls a profiler may want to time ("gemm", "gemm_gateup", "verify_attn") or is None.
        lazy_head: the acceptance computes the target LM head's logits itself, one level of the walk
        at a time and only for the nodes it visits (same decisions as the full head; the logits
        buffer is then not written)."""
        e3, c = _lib, self.cfg
        self.lazy_head = bool(lazy_head)
        self._keep = []
        L = e3.lib()
        B, N, d, D, Hq, Hkv = c["B"], c["N"], c["d"], c["D"], c["Hq"], c["Hkv"]
        R = B * N
        theta, eps = float(c.get("rope_theta", 500000.0)), float(c.get("eps", 1e-5))
        st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
        keep = self._keep
        dev_st = self.dev_status.data_ptr()

        def ws(t):
            return (ctypes.c_void_p(t.data_ptr()), ctypes.c_size_t(t.numel())) if t is not None else (None, 0)

        # ---- draft head and tree
        da = e3.draft_tree_args(self.aux_in, self.next_tok, self.tc, self.dk_cache, self.dv_cache,
                                self.draft_len, self.tokens, self.parents, self.depth, self.anc, self.score,
                                n_heads=Hq, ffn=c["F"], vocab=c["V"], depth=c["depth"], top_k=c["top_k"],
                                max_draft_len=self.max_prefix - 1, rope_theta=theta, rms_eps=eps,
                                dev_status=self.dev_status, d2t=self.d2t)
        need = L.eagle3_draft_tree_workspace_size(ctypes.byref(da))
        self.ws_draft = torch.empty(max(need, 16), dtype=torch.uint8, device=self.dev)
        dw = e3.draft_weights(self.draft_w)
        keep += [da, dw]
        wp, wb = ws(self.ws_draft)
        self.draft_ops = [(None, lambda a=da, w=dw: L.eagle3_draft_tree(ctypes.byref(w), ctypes.byref(a), wp, wb, st))]

        ops = []

        def norm(x, w, out, gather=None, tap=None):
            a = e3.RmsnormArgs(rows=out.shape[0], dim=w.shape[0], n_src=x.shape[0], eps=eps, ld_in=x.stride(0),
                               ld_out=out.stride(0), ld_tap=0 if tap is None else tap.stride(0),
                               input=x.data_ptr(), w=w.data_ptr(),
                               gather=None if gather is None else gather.data_ptr(), out=out.data_ptr(),
                               tap_out=None if tap is None else tap.data_ptr(), dev_status=dev_st)
            keep.append(a)
            ops.append((None, lambda a=a: L.eagle3_rmsnorm(ctypes.byref(a), st)))

        # linear workspace: the largest any projection of the step asks for
        self.ws_lin = torch.empty(ws_linear_bytes, dtype=torch.uint8, device=self.dev)
        lp, lb = ws(self.ws_lin)

        def lin(x, w, out, epi=0, w2=None, res=None, kind="gemm", rope_cols=0, ssq_out=None, ssq_in=None):
            a = e3.LinearArgs(m=x.shape[0], n=w.shape[0], k=x.shape[1], epilogue=epi, splits=0, ld_x=0, ld_w=0,
                              ld_out=0, ld_res=0, x=x.data_ptr(), w=w.data_ptr(),
                              w2=None if w2 is None else w2.data_ptr(), out=out.data_ptr(),
                              residual=None if res is None else res.data_ptr(), dev_status=dev_st,
                              rope_cols=rope_cols, rope_rows_per_seq=N, rope_theta=theta,
                              rope_base=self.prefix_len.data_ptr() if rope_cols else None,
                              rope_depth=self.depth.data_ptr() if rope_cols else None,
                              row_ssq=None if ssq_out is None else ssq_out.data_ptr(),
                              row_ssq_in=None if ssq_in is None else ssq_in.data_ptr(),
                              ssq_blocks=0 if ssq_in is None else self.ssq_blocks,
                              ssq_dim=0 if ssq_in is None else d, ssq_eps=eps)
            if L.eagle3_linear_workspace_size(ctypes.byref(a)) > ws_linear_bytes:
                raise ValueError("linear workspace too small for the step's shapes")
            keep.append(a)
            ops.append((kind, lambda a=a: L.eagle3_linear(ctypes.byref(a), lp, lb, st)))

        T = self.target
        taps = {t: i for i, t in enumerate(c["taps"])}
        fold = self.fold_norms
        if fold and self._folded is None:
            self._folded = self._fold_weights()
        Fw = self._folded
        # layer 0's norm reads the tree tokens' embedding rows and keeps them as the residual stream
        norm(T["embed"], T["norm1"][0], self.h, gather=self.tokens.view(-1), tap=self.x)
        self.ws_attn = torch.empty(ws_attn_bytes, dtype=torch.uint8, device=self.dev)
        ap, ab = ws(self.ws_attn)
        for l in range(c["layers"]):
            # the attention norm: a kernel on layer 0 (embedding gather) and on tapped layers (the tap
            # copies the stream entering the layer); otherwise folded into the QKV projection
            fold1 = fold and l > 0 and l not in taps
            if l > 0 and not fold1:
                tap = self.aux_tree[:, taps[l] * d:(taps[l] + 1) * d] if l in taps else None
                norm(self.x, T["norm1"][l], self.h, tap=tap)
            qkv = self.qkv[l]
            a_in, w_qkv = (self.x, Fw["wqkv"][l]) if fold1 else (self.h, T["wqkv"][l])
            s_in = self.ssq_next if fold1 else None
            if self.fused_rope:
                lin(a_in, w_qkv, qkv, epi=e3.EPI_BF16_ROPE, rope_cols=(Hq + Hkv) * D, ssq_in=s_in)
            else:
                lin(a_in, w_qkv, qkv, ssq_in=s_in)
            va = e3.verify_attn_args(self.tree_q(l), self.tree_k(l), self.tree_v(l), self.k_cache[l],
                                     self.v_cache[l], self.parents, self.prefix_len, self.attn.view(B, N, Hq, D),
                                     max_prefix_len=self.max_prefix, rope_theta=theta, dev_status=self.dev_status,
                                     qk_rotated=self.fused_rope)
            if L.eagle3_verify_attn_workspace_size(ctypes.byref(va)) > ws_attn_bytes:
                raise ValueError("attention workspace too small for the step's shapes")
            keep.append(va)
            ops.append(("verify_attn", lambda a=va: L.eagle3_verify_attn(ctypes.byref(a), ap, ab, st)))
            lin(self.attn, T["wo"][l], self.x, epi=e3.EPI_BF16_RESIDUAL, res=self.x,
                ssq_out=self.ssq_mid if fold else None)
            if fold:   # the post-attention norm folded into the gate / up projection
                lin(self.x, Fw["wg"][l], self.act, epi=e3.EPI_SWIGLU, w2=Fw["wu"][l], kind="gemm_gateup",
                    ssq_in=self.ssq_mid)
            else:
                norm(self.x, T["norm2"][l], self.h)
                lin(self.h, T["wg"][l], self.act, epi=e3.EPI_SWIGLU, w2=T["wu"][l], kind="gemm_gateup")
            lin(self.act, T["wd"][l], self.x, epi=e3.EPI_BF16_RESIDUAL, res=self.x,
                ssq_out=self.ssq_next if fold else None)
        fold_f = fold and not self.lazy_head   # the lazy head gathers normalised rows
        if not fold_f:
            norm(self.x, T["final_norm"], self.h)
        # ---- acceptance over the tree (the emitted row is the next step's catch-up tokens)
        if self.lazy_head:
            aa = e3.accept_lazy_args(c["mode"], self.h.view(B, N, d), T["lm_head"], self.tokens, self.parents,
                                     self.accept_len, self.path, self.next_tok, self.next_root,
                                     temperature=float(c.get("temperature", 1.0)), seed=int(c.get("seed", 0)),
                                     dev_status=self.dev_status, step_counter=self.step_counter)
            need = L.eagle3_accept_lazy_workspace_size(ctypes.byref(aa))
            accept_fn = L.eagle3_accept_lazy
        else:
            if self.logits is None:
                self.logits = torch.empty(R, c["V"], device=self.dev, dtype=torch.float32)
            if fold_f:
                lin(self.x, Fw["lm_head"], self.logits, epi=e3.EPI_F32, ssq_in=self.ssq_next)
            else:
                lin(self.h, T["lm_head"], self.logits, epi=e3.EPI_F32)
            aa = e3.AcceptArgs(mode=int(c["mode"]), batch=B, n_nodes=N, vocab=c["V"], max_path=c["W"],
                               temperature=float(c.get("temperature", 1.0)), seed=int(c.get("seed", 0)), step=0,
                               target_logits=self.logits.data_ptr(), draft_logits=None,
                               tokens=self.tokens.data_ptr(), parents=self.parents.data_ptr(),
                               accept_len=self.accept_len.data_ptr(), path=self.path.data_ptr(),
                               emitted=self.next_tok.data_ptr(), next_root=self.next_root.data_ptr(),
                               dev_status=dev_st, step_counter=self.step_counter.data_ptr())
            need = L.eagle3_accept_workspace_size(ctypes.byref(aa))
            accept_fn = L.eagle3_accept
        keep.append(aa)
        self.ws_acc = torch.empty(max(need, 16), dtype=torch.uint8, device=self.dev)
        cp, cb = ws(self.ws_acc)
        ops.append((None, lambda a=aa, f=accept_fn: f(ctypes.byref(a), cp, cb, st)))
        # ---- compaction: tree K/V read in place from the fused QKV outputs (node pitch qkv_w)
        kflat = torch.as_strided(self.qkv, (1,), (1,), storage_offset=Hq * D)
        vflat = torch.as_strided(self.qkv, (1,), (1,), storage_offset=(Hq + Hkv) * D)
        ca = e3.CompactArgs(n_layers=c["layers"], batch=B, n_nodes=N, n_kv_heads=Hkv, head_dim=D, elem_bytes=2,
                            s_max=self.S, max_path=c["W"], cache_layer_stride=B * Hkv * self.S * D,
                            tree_layer_stride=R * self.qkv_w, tree_node_stride=self.qkv_w,
                            k_cache=self.k_cache.data_ptr(), v_cache=self.v_cache.data_ptr(),
                            tree_k=kflat.data_ptr(), tree_v=vflat.data_ptr(), path=self.path.data_ptr(),
                            accept_len=self.accept_len.data_ptr(), prefix_len=self.prefix_len.data_ptr(),
                            slot_map=self.slot_map.data_ptr(), committed=self.tc.data_ptr(), aux_dim=3 * d,
                            aux_tree=self.aux_tree.data_ptr(), aux_out=self.aux_in.data_ptr(), dev_status=dev_st)
        keep.append(ca)
        ops.append((None, lambda a=ca: L.eagle3_compact_kv(ctypes.byref(a), st)))
        self.verify_ops = ops
        self.ops = self.draft_ops + self.verify_ops
        return self

    def _fold_weights(self):
        """Weights with the RMSNorm weight folded in, W' = W diag(g), made once (bf16 of the fp32
        product); a norm weight of all ones leaves W itself."""
        T, c = self.target, self.cfg

        def fold(w, g):
            if bool(torch.all(g == 1)):
                return w
            return (w.float() * g.float()[None, :]).to(torch.bfloat16).contiguous()
        return {"wqkv": [fold(T["wqkv"][l], T["norm1"][l]) for l in range(c["layers"])],
                "wg": [fold(T["wg"][l], T["norm2"][l]) for l in range(c["layers"])],
                "wu": [fold(T["wu"][l], T["norm2"][l]) for l in range(c["layers"])],
                "lm_head": fold(T["lm_head"], T["final_norm"])}

    # ------------------------------------------------------------------------------ issue
    @staticmethod
    def issue(ops, timed=None):
        """Issue prepared ops on the stream they were prepared for.  ``timed(kind, call)``, when
        given, wraps the calls whose kind is not None (e.g. to bracket them with events)."""
        for kind, call in ops:
            if kind is not None and timed is not None:
                timed(kind, call)
            else:
                status = call()
                if status:
                    raise _lib.Eagle3Error(status, "libeagle3 step call")

    def run(self, draft=True, timed=None):
        """One step: the draft (unless draft=False: the tree already in tokens / parents / depth
        is verified as it is), then the target's verification, acceptance and compaction."""
        if not self.verify_ops:
            self.prepare()
        self.issue(self.ops if draft else self.verify_ops, timed)

    def flops(self, catchup_rows=None, head_rows=None):
        """Algorithmic GEMM flops of one step: (target verify, draft head).  The draft counts the
        real catch-up rows (sum of tc over the batch; default one per sequence, the committed count
        of a step that accepted nothing), not the rows the launch pads to tc_max.  head_rows: rows of
        the target LM head (default every tree node; with the lazy head, the visited nodes)."""
        c = self.cfg
        d, F, V, Hq, D, qw = c["d"], c["F"], c["V"], c["Hq"], c["D"], self.qkv_w
        Vd = V if self.d2t is None else int(self.d2t.numel())
        R = c["B"] * c["N"]
        per_layer = 2 * R * (d * qw + Hq * D * d + 2 * d * F + F * d)
        target = c["layers"] * per_layer + 2 * (R if head_rows is None else head_rows) * d * V
        rows_d = c["B"] * c["top_k"]
        draft_layer = lambda m: 2 * m * (2 * d * qw + Hq * D * d + 2 * d * F + F * d)
        tc_rows = c["B"] if catchup_rows is None else catchup_rows
        draft = (2 * tc_rows * 3 * d * d + draft_layer(tc_rows) + 2 * c["B"] * d * Vd
                 + (c["depth"] - 1) * (draft_layer(rows_d) + 2 * rows_d * d * Vd))
        return target, draft
