"""Benchmark: one EAGLE-3 draft-and-verify step per iteration on GB300.

Workload (default): Llama-3.1-8B-shaped random-init target (32 layers, d 4096, GQA 32/8, FFN
14336, vocab 128256, bf16) and EAGLE-3 draft head (fc 12288->4096, one decoder layer, own LM
head), batch 64, 2048-token prefixes, 60-node dynamic trees (depth 6, top-k 10), temperature 1
(TOPK rejection sampling, Philox seed 2), compaction of the accepted path into the caches.  A
step is: eagle3_draft_tree -> 32 target layers over the tree (RMSNorm with fused aux taps,
tcgen05 QKV / O / SwiGLU / down GEMMs, eagle3_verify_attn) -> final norm -> LM head (fp32
logits) -> eagle3_accept -> eagle3_compact_kv; its outputs feed the next step (a real decoding
loop).  Metric: verified tree tokens per second (B * N per step).

Every number comes from CUDA events on the launching stream; the dominant kernel (the tcgen05
GEMM) and the verify attention are also timed per launch inside the timed region.
"""
import argparse
import json
import math
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

METRIC = "verified tree tokens/s per GB300 (draft+verify+accept); verify-attn HBM GB/s"
UNIT = "tokens/s"

CFG = dict(layers=32, d=4096, Hq=32, Hkv=8, D=128, F=14336, V=128256, taps=(2, 15, 29),
           B=64, N=60, L0=2048, depth=6, top_k=10, W=7, temperature=1.0, seed=2)


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), float(p["bf16_tflops_sustained"]), "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


# ----------------------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples (SM clock, max clock, throttle reasons), timestamped on arrival.

    The sampler is started before the warm-up so that its own start-up is not inside the timed
    region; summary() keeps only the samples that arrived inside [t0, t1]."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, index):
        self.index, self.rows, self.proc = index, [], None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 9:
                self.rows.append((time.time(), parts))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t0, t1):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = [r for (t, r) in self.rows if t0 <= t <= t1]
        if not rows:      # timed region shorter than one period: take the nearest samples
            rows = [r for (t, r) in self.rows][-2:]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        num = lambda v: v.replace(".", "", 1).isdigit()
        sm = sorted(float(r[1]) for r in rows if num(r[1]))
        mx = max([float(r[2]) for r in rows if num(r[2])] or [0.0])
        reasons = sorted({self.NAMES[i] for r in rows for i in range(4) if r[5 + i].strip() == "Active"})
        pw = sorted(float(r[3]) for r in rows if num(r[3]))
        return {"sm_mhz": sm[len(sm) // 2] if sm else None, "sm_max_mhz": mx, "reasons": reasons,
                "samples": len(rows), "power_w": pw[len(pw) // 2] if pw else None}


# ----------------------------------------------------------------------------------------- GPU arm
class Engine:
    """The bench workload around the package's SpeculativeStep: random-init Llama-3.1-8B-shaped
    target and EAGLE-3 head (N(0, 0.02), norms 1), N(0, 1) prefilled caches, and per-launch timing
    of the dominant kernels with CUDA events on the launching stream."""

    def __init__(self, cfg, steps_total, dev, timing=True, fused_rope=True, fold_norms=True):
        from eagle_tree_speculative_spec_gb300.step import SpeculativeStep
        import eagle_tree_speculative_spec_gb300 as e3
        self.e3, self.cfg, self.dev, self.timing = e3, cfg, dev, timing
        # the target's QKV projection rotates q and the tree keys (EPI_BF16_ROPE) and the verify
        # attention takes them as they are; False: the attention rotates them itself
        self.fused_rope = fused_rope
        c = cfg
        B, d, V, D = c["B"], c["d"], c["V"], c["D"]
        Hq, Hkv, F, Lyr = c["Hq"], c["Hkv"], c["F"], c["layers"]
        qkv_w = (Hq + 2 * Hkv) * D
        S = c["L0"] + c["W"] * (steps_total + 2) + 64
        # host-side length bound of every launch, fixed for the run so one captured graph serves every step
        # (the kernels read the exact per-sequence lengths from device memory)
        max_prefix = c["L0"] + c["W"] * (steps_total + 1)
        g = torch.Generator(device=dev)
        g.manual_seed(1234)
        bf = torch.bfloat16

        def w(*shape, std=0.02):
            return (torch.randn(*shape, generator=g, device=dev, dtype=torch.float32) * std).to(bf)

        ones = lambda n: torch.ones(n, device=dev, dtype=bf)
        embed = w(V, d)
        target = {"embed": embed, "wqkv": [w(qkv_w, d) for _ in range(Lyr)], "wo": [w(d, Hq * D) for _ in range(Lyr)],
                  "wg": [w(F, d) for _ in range(Lyr)], "wu": [w(F, d) for _ in range(Lyr)],
                  "wd": [w(d, F) for _ in range(Lyr)], "norm1": [ones(d) for _ in range(Lyr)],
                  "norm2": [ones(d) for _ in range(Lyr)], "final_norm": ones(d), "lm_head": w(V, d)}
        # draft head (shares the target embedding; own LM head)
        draft = {"w_fc": w(d, 3 * d), "embed": embed, "input_norm": ones(d), "hidden_norm": ones(d),
                 "w_qkv": w(qkv_w, 2 * d), "w_o": w(d, Hq * D), "post_norm": ones(d),
                 "w_gate": w(F, d), "w_up": w(F, d), "w_down": w(d, F), "final_norm": ones(d), "lm_head": w(V, d)}
        scfg = dict(c, mode=e3.TOPK)
        self.step_obj = st = SpeculativeStep(scfg, target, draft, S, max_prefix, dev, fused_rope=fused_rope,
                                             fold_norms=fold_norms)
        self.S, self.max_prefix = S, max_prefix
        # caches: prefixes of L0 positions of N(0, 1) keys / values (as if prefilled)
        st.k_cache[..., : c["L0"], :].normal_(generator=g)
        st.v_cache[..., : c["L0"], :].normal_(generator=g)
        st.dk_cache[..., : c["L0"] - 1, :].normal_(generator=g)
        st.dv_cache[..., : c["L0"] - 1, :].normal_(generator=g)
        st.prefix_len.fill_(c["L0"])
        st.draft_len.fill_(c["L0"] - 1)
        # catch-up input of the first step: the last prompt position's aux states and the root token
        st.aux_in[:, 0].normal_(generator=g)
        st.next_tok.copy_(torch.randint(0, V, st.next_tok.shape, generator=g, device=dev, dtype=torch.int32))
        st.tc.fill_(1)
        # the per-sequence state and outputs are the step's buffers
        for name in ("prefix_len", "draft_len", "aux_in", "next_tok", "tc", "accept_len", "dev_status", "tokens"):
            setattr(self, name, getattr(st, name))
        self.steps_done = 0
        self.kernel_ms = {"gemm": 0.0, "gemm_gateup": 0.0, "verify_attn": 0.0}
        self.kernel_calls = {"gemm": 0, "gemm_gateup": 0, "verify_attn": 0}
        self._ev = []
        # events are created once and reused: creating timing events inside the loop is not free
        self._pool = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                      for _ in range(4096)]

    # -- per-launch timing of the dominant kernels (CUDA events on the launching stream)
    def _timed(self, kind, fn, evs, external=False):
        if external:
            a, b = (torch.cuda.Event(enable_timing=True, external=True),
                    torch.cuda.Event(enable_timing=True, external=True))
        else:
            if len(self._ev) >= len(self._pool):
                self._pool += [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                               for _ in range(len(self._pool))]
            a, b = self._pool[len(self._ev)]
        a.record()
        status = fn()
        b.record()
        if status:
            raise RuntimeError(f"libeagle3 call failed with status {status}")
        evs.append((kind, a, b))

    def collect(self, evs=None):
        torch.cuda.synchronize()
        for kind, a, b in (self._ev if evs is None else evs):
            self.kernel_ms[kind] += a.elapsed_time(b)
            self.kernel_calls[kind] += 1
        if evs is None:
            self._ev = []

    def reset_counters(self):
        self.collect()
        self.kernel_ms = {k: 0.0 for k in self.kernel_ms}
        self.kernel_calls = {k: 0 for k in self.kernel_calls}

    def _issue(self, evs, external=False):
        timed = None if evs is None else (lambda kind, call: self._timed(kind, call, evs, external))
        self.step_obj.run(timed=timed)

    def step(self):
        """One eager step: every C call issued from the host."""
        if not self.step_obj.verify_ops:
            self.step_obj.prepare()
        self._issue(self._ev if self.timing else None)
        self.steps_done += 1

    def capture(self, n):
        """Capture n CUDA graphs of one step each (same kernels; each graph owns its timing events, so
        every replay of a timed loop over the n graphs can be read back afterwards)."""
        if not self.step_obj.verify_ops:
            self.step_obj.prepare()
        self.graphs = []
        pool = None
        for _ in range(n):
            try:
                g = torch.cuda.CUDAGraph(keep_graph=True)
            except TypeError:
                g = torch.cuda.CUDAGraph()
            evs = []
            with torch.cuda.graph(g, pool=pool, stream=torch.cuda.current_stream()):
                self._issue(evs if self.timing else None, external=True)
            pool = g.pool()
            self.graphs.append((g, evs))

    def replay(self, i):
        self.graphs[i % len(self.graphs)][0].replay()
        self.steps_done += 1

    def graph_kernels(self):
        """Kernel nodes of the first captured graph, by function name (driver graph API)."""
        return graph_kernel_names(self.graphs[0][0])

    def flops_per_step(self, catchup_rows=None):
        """Algorithmic GEMM flops of one step (target verify, draft head over the real catch-up rows)."""
        return self.step_obj.flops(catchup_rows)

    def attn_bytes_per_launch(self, L):
        """Algorithmic HBM bytes of one verify-attention launch (one layer, whole batch)."""
        c = self.cfg
        B, N, Hq, Hkv, D = c["B"], c["N"], c["Hq"], c["Hkv"], c["D"]
        kv_prefix = 2 * B * Hkv * L * D * 2
        tree_kv = 2 * B * N * Hkv * D * 2
        rot_write = 0 if self.fused_rope else B * N * Hkv * D * 2   # the in-call rotation writes tree_k back
        q_o = 2 * B * N * Hq * D * 2
        return kv_prefix + tree_kv + rot_write + q_o


class _KernelNodeParams(__import__("ctypes").Structure):
    import ctypes as _c
    _fields_ = [("func", _c.c_void_p), ("grid", _c.c_uint * 3), ("block", _c.c_uint * 3), ("smem", _c.c_uint),
                ("kernel_params", _c.c_void_p), ("extra", _c.c_void_p), ("kern", _c.c_void_p), ("ctx", _c.c_void_p)]


def graph_kernel_names(g):
    """{kernel name: launches} over the kernel nodes of a captured graph (driver graph API), or None."""
    import ctypes
    import re
    try:
        raw = g.raw_cuda_graph()
        cu = ctypes.CDLL("libcuda.so.1")
    except Exception:
        return None
    n = ctypes.c_size_t(0)
    if cu.cuGraphGetNodes(ctypes.c_void_p(raw), None, ctypes.byref(n)) != 0:
        return None
    nodes = (ctypes.c_void_p * max(1, n.value))()
    if cu.cuGraphGetNodes(ctypes.c_void_p(raw), nodes, ctypes.byref(n)) != 0:
        return None
    out = {}
    for i in range(n.value):
        t = ctypes.c_int(-1)
        if cu.cuGraphNodeGetType(ctypes.c_void_p(nodes[i]), ctypes.byref(t)) != 0 or t.value != 0:
            continue                                        # 0: CU_GRAPH_NODE_TYPE_KERNEL
        prm = _KernelNodeParams()
        name = ctypes.c_char_p()
        if cu.cuGraphKernelNodeGetParams_v2(ctypes.c_void_p(nodes[i]), ctypes.byref(prm)) != 0:
            key = "?"
        elif prm.func and cu.cuFuncGetName(ctypes.byref(name), ctypes.c_void_p(prm.func)) == 0 and name.value:
            key = name.value.decode()
        elif prm.kern and cu.cuKernelGetName(ctypes.byref(name), ctypes.c_void_p(prm.kern)) == 0 and name.value:
            key = name.value.decode()
        else:
            key = "?"
        m = re.search(r"([A-Za-z_][A-Za-z0-9_]*_kernel)", key)
        key = m.group(1) if m else key
        out[key] = out.get(key, 0) + 1
    return out


def max_over_ranks(x, dev):
    """The largest value over the ranks of the process group (the job's time is the slowest
    rank's); x itself with no group or a single rank."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(units_per_rank, world, ms):
    """Whole-job throughput: the units every rank processed over the slowest rank's time."""
    return units_per_rank * world / (ms / 1e3)


def external_events_ok():
    try:
        torch.cuda.Event(enable_timing=True, external=True)
        return True
    except TypeError:
        return False


def run_gpu(args):
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import __graft_entry__
    __graft_entry__.build()
    cfg = dict(CFG)
    cfg["B"] = args.batch
    # all work on one side stream: graph capture needs a stream other than the legacy default one
    stream = torch.cuda.Stream(device=dev)
    torch.cuda.set_stream(stream)
    eng = Engine(cfg, args.steps * 3 + 2 * max(args.warmup, args.steps) + 8, dev, fused_rope=not args.rope_in_attention,
                 fold_norms=not args.norm_kernels)
    use_graph = not args.eager
    if use_graph and not external_events_ok():
        eng.timing = False                      # timing events cannot live inside a graph: time kernels eagerly
    clocks = ClockSampler(local)
    clocks.start()
    eng.step()                                  # eager warm-up: kernel attributes, tensor maps, first touch
    # the timed loop's own bookkeeping ops run in the warm-up too: PyTorch loads its kernels lazily, and
    # on a cold host the first load takes long enough to leave the GPU idle inside the timed region
    warm_acc = torch.zeros((), dtype=torch.int64, device=dev)
    if use_graph:
        eng.capture(args.steps)
        for i in range(max(args.warmup, args.steps)):   # the first launch of a graph uploads it: do all
            eng.replay(i)
            warm_acc += (eng.accept_len.to(torch.int64) + 1).sum()
    else:
        for _ in range(args.warmup):
            eng.step()
            warm_acc += (eng.accept_len.to(torch.int64) + 1).sum()
    eng.reset_counters()
    torch.cuda.synchronize()
    prefix_before = int(eng.prefix_len.sum())
    if world > 1:
        dist.barrier()
    wall0 = time.time()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    step_ev = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    t0.record()
    accepted = torch.zeros((), dtype=torch.int64, device=dev)
    for i in range(args.steps):
        if use_graph:
            eng.replay(i)
        else:
            eng.step()
        accepted += (eng.accept_len.to(torch.int64) + 1).sum()
        step_ev[i].record()
    t1.record()
    torch.cuda.synchronize()
    ms = t0.elapsed_time(t1)
    step_ms = [round((t0 if i == 0 else step_ev[i - 1]).elapsed_time(step_ev[i]), 3) for i in range(args.steps)]
    wall1 = time.time()
    clocks.stop()
    clk = clocks.summary(wall0, wall1)
    # mean verified prefix over the timed steps (the prefix grows by the accepted length + 1 per step)
    L_mean = (prefix_before + int(eng.prefix_len.sum())) / (2.0 * cfg["B"])
    if use_graph and eng.timing:
        for _, evs in eng.graphs:
            eng.collect(evs)
    elif use_graph:                             # per-kernel times from eager steps after the timed region
        eng.timing = True
        for _ in range(min(args.steps, 5)):
            eng.step()
        eng.collect()
    else:
        eng.collect()
    kernels = eng.graph_kernels() if use_graph else None
    # the verify attention of layer 0 as it stands after the timed steps (prefix lengths of the run's
    # end), issued back to back on its prepared arguments: the kernel without the event nodes that
    # bracket it inside the step graph (its inputs, 0.6 GB of KV, are larger than L2)
    attn_op = next(call for kind, call in eng.step_obj.verify_ops if kind == "verify_attn")
    attn_alone_ms = _time_loop(attn_op, 20, 3)
    L_end = float(eng.prefix_len.float().mean())
    if world > 1:
        dist.barrier()
    ms = max_over_ranks(ms, dev)
    status = int(eng.dev_status.item())

    # ---- e2e through host buffers: every step's inputs come from pinned host memory and its outputs go
    # back to it, and the outputs of step i are the inputs of step i + 1 (the decoding loop's own data
    # flow, carried through the host): catch-up aux rows, the emitted tokens (last one = next root), the
    # committed counts; the accepted lengths are read back as the step's result
    c = cfg
    host_aux = eng.aux_in.cpu().pin_memory()
    host_tok = eng.next_tok.cpu().pin_memory()
    host_tc = eng.tc.cpu().pin_memory()
    out_len = torch.empty_like(eng.accept_len, device="cpu").pin_memory()
    eng.timing = False

    def e2e_step(i):
        eng.aux_in.copy_(host_aux, non_blocking=True)
        eng.next_tok.copy_(host_tok, non_blocking=True)
        eng.tc.copy_(host_tc, non_blocking=True)
        if use_graph:
            eng.replay(i)
        else:
            eng.step()
        host_aux.copy_(eng.aux_in, non_blocking=True)
        host_tok.copy_(eng.next_tok, non_blocking=True)
        host_tc.copy_(eng.tc, non_blocking=True)
        out_len.copy_(eng.accept_len, non_blocking=True)

    # untimed warm-up steps right before the timed ones, as for the device-timed loop: after the pause
    # above, the first steps run at a higher clock than the power cap then settles to
    for i in range(args.warmup):
        e2e_step(i)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record()
    for i in range(args.steps):
        e2e_step(i)
    e1.record()
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), dev)

    # ---- the same step with the lazy target LM head (eagle3_accept_lazy: the head's logits only for
    # the nodes the acceptance walk visits), continuing from the state the loops above left
    eng.step_obj.prepare(lazy_head=True)
    if use_graph:
        eng.capture(args.steps)
        for i in range(max(args.warmup, args.steps)):
            eng.replay(i)
    else:
        for _ in range(args.warmup):
            eng.step()
    torch.cuda.synchronize()
    l0, l1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    lazy_acc = torch.zeros((), dtype=torch.int64, device=dev)
    l0.record()
    for i in range(args.steps):
        if use_graph:
            eng.replay(i)
        else:
            eng.step()
        lazy_acc += (eng.accept_len.to(torch.int64) + 1).sum()
    l1.record()
    torch.cuda.synchronize()
    lazy_ms = max_over_ranks(l0.elapsed_time(l1), dev)
    status |= int(eng.dev_status.item())
    h2d = host_aux.numel() * 2 + host_tok.numel() * 4 + host_tc.numel() * 4
    d2h = h2d + out_len.numel() * 4

    units = cfg["B"] * cfg["N"] * args.steps * world
    value = job_rate(cfg["B"] * cfg["N"] * args.steps, world, ms)
    hbm, tf_burst, tf_sust, src = peaks()
    tgt_f, drf_f = eng.flops_per_step()
    # the target's projections are timed one by one; the draft head's run inside eagle3_draft_tree
    gemm_ms = (eng.kernel_ms["gemm"] + eng.kernel_ms["gemm_gateup"]) / max(1, args.steps)
    gemm_calls = (eng.kernel_calls["gemm"] + eng.kernel_calls["gemm_gateup"]) / max(1, args.steps)
    gemm_tflops = tgt_f / (gemm_ms / 1e3) / 1e12 if gemm_ms > 0 else None
    # the dominant launch: the SwiGLU gate + up projection of a target layer
    R = cfg["B"] * cfg["N"]
    gu_flops = 2.0 * R * (2 * cfg["F"]) * cfg["d"]
    gu_ms = eng.kernel_ms["gemm_gateup"] / max(1, eng.kernel_calls["gemm_gateup"])
    gu_tflops = gu_flops / (gu_ms / 1e3) / 1e12 if gu_ms > 0 else None
    attn_ms = eng.kernel_ms["verify_attn"] / max(1, eng.kernel_calls["verify_attn"])
    attn_gbs = eng.attn_bytes_per_launch(L_mean) / (attn_ms / 1e3) / 1e9 if attn_ms > 0 else None
    tau = float(accepted.item()) / (cfg["B"] * args.steps) - 1.0
    if kernels:
        launches_per_step = sum(kernels.values())
    else:
        launches_per_step = gemm_calls + cfg["layers"] * 2 + 3 * cfg["layers"] + 4 + _draft_launches(cfg)
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms / args.steps, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (random-init weights N(0,0.02), N(0,1) caches, uniform tokens)",
        "config": {"workload": "EAGLE-3 draft-and-verify step, Llama-3.1-8B-shaped target + EAGLE-3 head, "
                               "B=64, N=60 (depth 6, top-k 10), prefix 2048, T=1, compaction on",
                   "global_batch": cfg["B"] * world, "seq_len": cfg["L0"], "parallelism": f"replicas x{world}",
                   "l2": "inputs larger than L2 (16 GB of weights streamed per step)"},
        "roofline": {"bound": "tensor", "achieved": round(gu_tflops, 1) if gu_tflops else None,
                     "peak": tf_sust, "unit": "TFLOP/s",
                     "frac": round(gu_tflops / tf_sust, 4) if gu_tflops else None,
                     "traffic": GATEUP_TRAFFIC_BYTES,
                     "traffic_source": "ncu dram__bytes_read.sum + dram__bytes_write.sum of one launch of this "
                                       "kernel at this shape (a separate capture, not this run)",
                     "frac_of_burst": round(gu_tflops / tf_burst, 4) if gu_tflops else None,
                     "kernel": f"gemm_tc_kernel, SwiGLU gate+up projection M={R} N=2x{cfg['F']} K={cfg['d']} "
                               f"({gu_flops / 1e12:.3f} TFLOP per launch, {cfg['layers']} launches per step)",
                     "ms_per_launch": round(gu_ms, 4),
                     "peak_source": f"{src} bf16_tflops_sustained (kernel timed inside the step)",
                     "all_target_gemms": {"achieved": round(gemm_tflops, 1) if gemm_tflops else None,
                                          "frac": round(gemm_tflops / tf_sust, 4) if gemm_tflops else None,
                                          "launches_per_step": gemm_calls}},
        "verify_attn": {"achieved_gbs": round(attn_gbs, 1) if attn_gbs else None, "peak_gbs": hbm,
                        "frac": round(attn_gbs / hbm, 4) if attn_gbs else None,
                        "frac_of_8tbs": round(attn_gbs / 8000.0, 4) if attn_gbs else None,
                        "ms_per_launch": round(attn_ms, 4), "prefix_len": round(L_mean, 1),
                        "standalone": {"ms_per_launch": round(attn_alone_ms, 4), "prefix_len": round(L_end, 1),
                                       "frac": round(eng.attn_bytes_per_launch(L_end) / (attn_alone_ms / 1e3) / 1e9
                                                     / hbm, 4),
                                       "how": "layer 0's prepared call issued 20 times back to back after the "
                                              "timed steps (no event nodes around it)"}},
        "lazy_head": {"value": round(job_rate(cfg["B"] * cfg["N"] * args.steps, world, lazy_ms), 2), "unit": UNIT,
                      "ms_per_step": round(lazy_ms / args.steps, 4),
                      "tau": round(float(lazy_acc.item()) / (cfg["B"] * args.steps) - 1.0, 4),
                      "how": "the same step with eagle3_accept_lazy in place of the full LM head and "
                             "eagle3_accept (head logits only for the visited nodes; the lazy head reads rows "
                             "normalised by the norm kernel where the full head folds the norm, so decisions "
                             "agree up to that rounding), "
                             f"{args.steps} steps timed after the e2e loop"},
        "accepted_tokens_per_s": round(float(accepted.item()) * world / (ms / 1e3), 2),
        "tau": round(tau, 4),
        "e2e": {"value": round(units / (e2e_ms / 1e3), 2), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": int(round(launches_per_step * args.steps)),
        "launches_per_step": kernels if kernels else {"estimate": launches_per_step},
        "issue": "cuda-graph replay, one graph per step" if use_graph else "eager C-ABI calls",
        "clocks": clk,
        "step_ms": step_ms,
        "dev_status": status,
    }
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(cfg)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


# DRAM bytes (read + write) of one SwiGLU gate+up launch at the bench shape, from an ncu capture of the
# current GEMM kernel (to be set to None when the kernel changes)
GATEUP_TRAFFIC_BYTES = 267338240 + 100351232


def _draft_launches(cfg):
    # catch-up: meta, fc, prologue, qkv, attn, O, norm, swiglu, down, append, norm, lm, topk, select
    # per depth 2..D: prologue, qkv, attn, O, norm, swiglu, down, norm, lm, topk, select; final select;
    # split-K GEMMs add a reduce launch (counted in the GEMM events above as part of the call)
    return 14 + (cfg["depth"] - 1) * 11 + 1


# ----------------------------------------------------------------------------------------- oracle arm
def oracle_sample_seconds(cfg, rng_seed=0):
    """Time the oracle (as it stands) on a bounded sample of the step for ONE sequence and
    extrapolate to the full step of that sequence:
      t_attn  one layer of verify attention (60 nodes, 32 heads, 2048 prefix)
      t_proj  one target layer's projections for the 60 rows (row by row, fp64)
      t_lm    the LM head for 6 of the 60 rows over 1/8 of the vocabulary (scaled x80)
      t_acc   TOPK acceptance over the 60-node tree (V = 128256)
    step(seq) ~= 32 (t_attn + t_proj) + t_lm + t_acc + draft, with the draft estimated as
    51/60 of one layer's projections plus its own attention and 51/60 of the LM head."""
    import numpy as np

    import synth
    from oracle import accept as oacc
    from oracle import attention as oatt
    from oracle.llama import _rows, rmsnorm, silu
    c = cfg
    d, F, V, Hq, Hkv, D, N = c["d"], c["F"], c["V"], c["Hq"], c["Hkv"], c["D"], c["N"]
    r = synth.rng(rng_seed, 5)
    t = {}
    inp = synth.verify_attn_batch(rng_seed, 1, N, Hq, Hkv, D, [c["L0"]], S_max=c["L0"] + N)
    t0 = time.perf_counter()
    oatt.verify_attention(inp["q_f32"], inp["tree_k_f32"], inp["tree_v_f32"], inp["k_cache_f32"],
                          inp["v_cache_f32"], inp["parents"], inp["prefix_len"])
    t["attn"] = time.perf_counter() - t0
    x = r.standard_normal((N, d)).astype(np.float32)
    wq = (0.02 * r.standard_normal(((Hq + 2 * Hkv) * D, d))).astype(np.float32)
    wo = (0.02 * r.standard_normal((d, Hq * D))).astype(np.float32)
    wg = (0.02 * r.standard_normal((F, d))).astype(np.float32)
    wu = (0.02 * r.standard_normal((F, d))).astype(np.float32)
    wd = (0.02 * r.standard_normal((d, F))).astype(np.float32)
    t0 = time.perf_counter()
    h = rmsnorm(x, np.ones(d), 1e-5)
    _rows(wq, h)
    y = x + _rows(wo, h[:, : Hq * D])
    h2 = rmsnorm(y, np.ones(d), 1e-5)
    _rows(wd, silu(_rows(wg, h2)) * _rows(wu, h2))
    t["proj"] = time.perf_counter() - t0
    del wq, wo, wg, wu, wd
    lm = (0.02 * r.standard_normal((V // 8, d))).astype(np.float32)     # 1/8 of the vocabulary
    t0 = time.perf_counter()
    _rows(lm, h[:6])
    t["lm"] = (time.perf_counter() - t0) * (N / 6) * 8
    del lm
    zt, zd, parents = synth.accept_row(1, 0, N, V)
    tokens = synth.tokens_top_draft(zd, parents)
    t0 = time.perf_counter()
    oacc.accept_topk(tokens, parents, zt, 1.0, 2, 0, 0)
    t["acc"] = time.perf_counter() - t0
    rows_d = 1 + (c["depth"] - 1) * c["top_k"]
    draft = (rows_d / N) * (t["proj"] + t["lm"] + t["attn"])
    step = c["layers"] * (t["attn"] + t["proj"]) + t["lm"] + t["acc"] + draft
    return step, t


def host_threads():
    """Threads the host's NumPy BLAS may use (the oracle's matrix products)."""
    threads = torch.get_num_threads()
    try:
        import numpy as np  # noqa: F401
        from threadpoolctl import threadpool_info
        threads = max([i.get("num_threads", 1) for i in threadpool_info()] + [1])
    except Exception:
        pass
    return threads


def cpu_baseline(cfg):
    step, parts = oracle_sample_seconds(cfg)
    threads = host_threads()
    value = cfg["N"] / step          # verified tree tokens per second for one sequence on the host
    return {"value": round(value, 6), "unit": UNIT, "cores": threads, "kind": "oracle", "extrapolated": True,
            "scale_factors": {"layers": cfg["layers"], "lm_head_rows": cfg["N"] / 6, "lm_head_vocab": 8,
                              "draft_rows_per_verify_row": (1 + (cfg["depth"] - 1) * cfg["top_k"]) / cfg["N"],
                              "batch": cfg["B"]},
            "sample": ("one sequence: one layer of verify attention (60 nodes, 2048 prefix), one target "
                       "layer's projections and 6 LM-head rows (1/8 of the vocabulary) in fp64, TOPK acceptance at V=128256; "
                       "extrapolated to 32 layers + LM head + draft head; seconds per part: "
                       + ", ".join(f"{k}={v:.2f}" for k, v in parts.items()))}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    cfg = dict(CFG)
    # no warm-up steps are run: the oracle keeps no state between steps (no caches, no compiled
    # code, no device), so a warm-up would only lengthen the run; the line reports W as given
    total = 0.0
    per = []
    for i in range(args.steps):
        step, _ = oracle_sample_seconds(cfg, rng_seed=i)
        per.append(step)
        total += step * cfg["B"]        # the batch runs one sequence after another on the host
    ms = total / args.steps * 1e3
    value = cfg["B"] * cfg["N"] * args.steps / total
    cb = cpu_baseline(cfg)
    cb["value"] = round(value, 6)
    # n_gpus: the launch's GPU count (the oracle itself runs on the host cores, rank 0 only)
    line = {"metric": METRIC, "value": round(value, 6), "unit": UNIT, "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms, 2), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": "EAGLE-3 draft-and-verify step, Llama-3.1-8B-shaped target + EAGLE-3 head, "
                                   "B=64, N=60 (depth 6, top-k 10), prefix 2048, T=1, compaction on",
                       "global_batch": cfg["B"], "seq_len": cfg["L0"], "parallelism": "host cores"},
            "impl": "reference", "cpu_baseline": cb, "extrapolated": True,
            "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------------------- kernels
def _time_loop(fn, steps, warmup, flush=None):
    """Average device time per call with CUDA events on the launching stream.  Without a flush the
    calls run back to back between one pair of events (for inputs larger than L2), so the host's
    time to issue a call overlaps the previous call; with a flush, every call gets its own events
    after an L2 flush."""
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    if flush is None:
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(steps):
            fn()
        b.record()
        torch.cuda.synchronize()
        return a.elapsed_time(b) / steps
    total = 0.0
    for _ in range(steps):
        flush()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        fn()
        b.record()
        torch.cuda.synchronize()
        total += a.elapsed_time(b)
    return total / steps


def _raw_call(c_fn, args, ws):
    """A prepared C call on the current stream (argument struct built once): no Python marshalling
    inside the timed region."""
    import ctypes
    st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    wp = ctypes.c_void_p(ws.data_ptr()) if ws is not None else None
    wb = ctypes.c_size_t(ws.numel() if ws is not None else 0)
    status = c_fn(ctypes.byref(args), wp, wb, st)
    if status:
        raise RuntimeError(f"libeagle3 call failed with status {status}")
    return lambda: c_fn(ctypes.byref(args), wp, wb, st)


def run_generate(args):
    """The end-to-end run of the workload: every sequence generates `--generate` new tokens (each
    step emits accept_len + 1 >= 1 tokens per sequence, so that many steps always suffice); reports
    throughput and the measured acceptance length."""
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    import __graft_entry__
    __graft_entry__.build()
    stream = torch.cuda.Stream(device=dev)
    torch.cuda.set_stream(stream)
    cfg = dict(CFG)
    cfg["B"] = args.batch
    n_new = args.generate
    eng = Engine(cfg, n_new + 2, dev, timing=False, fused_rope=not args.rope_in_attention)
    eng.step()                                    # warm-up step (its tokens are not counted)
    eng.capture(1)
    gen = torch.zeros(cfg["B"], dtype=torch.int64, device=dev)
    steps_needed = torch.zeros((), dtype=torch.int64, device=dev)
    eng.replay(0)
    gen += eng.accept_len.to(torch.int64) + 1      # warm the bookkeeping ops too
    gen.zero_()
    torch.cuda.synchronize()
    clocks = ClockSampler(0)
    clocks.start()
    wall0 = time.time()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record()
    for _ in range(n_new):
        eng.replay(0)
        steps_needed += (gen < n_new).to(torch.int64).max()
        gen += eng.accept_len.to(torch.int64) + 1
    t1.record()
    torch.cuda.synchronize()
    wall1 = time.time()
    clocks.stop()
    ms = t0.elapsed_time(t1)
    g = gen.cpu()
    emitted = int(g.sum())
    line = {
        "mode": "generate", "new_tokens_per_sequence": n_new, "batch": cfg["B"], "steps": n_new,
        "steps_until_every_sequence_had_n_new": int(steps_needed.item()),
        "ms_total": round(ms, 2), "ms_per_step": round(ms / n_new, 4),
        "verified_tree_tokens_per_s": round(cfg["B"] * cfg["N"] * n_new / (ms / 1e3), 1),
        "emitted_tokens_per_s": round(emitted / (ms / 1e3), 1),
        "acceptance_length_mean": round(emitted / (cfg["B"] * n_new), 4),
        "emitted_per_sequence_min_max": [int(g.min()), int(g.max())],
        "final_prefix_len_mean": round(float(eng.prefix_len.float().mean()), 1),
        "dev_status": int(eng.dev_status.item()),
        "clocks": clocks.summary(wall0, wall1),
        "config": "B=64, N=60 (depth 6, top-k 10), prefix 2048, T=1, Philox seed 2, compaction on; "
                  "random-init weights, N(0,1) prefilled caches",
    }
    print(json.dumps(line), flush=True)


def run_kernel(args):
    """Single-kernel measurements of the rows of the path (not the headline line)."""
    import eagle_tree_speculative_spec_gb300 as e3
    import __graft_entry__
    __graft_entry__.build()
    dev = torch.device("cuda", 0)
    hbm, tf_burst, tf_sust, src = peaks()
    g = torch.Generator(device=dev)
    g.manual_seed(7)
    flush_buf = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    flush = lambda: flush_buf.zero_()
    out = {"kernel": args.kernel}
    if args.kernel == "verify_attn":
        B, L, N, Hq, Hkv, D = args.batch, args.prefix, 60, 32, 8, 128
        S = L + 64
        bf = torch.bfloat16
        q = torch.randn(B, N, Hq, D, generator=g, device=dev).to(bf)
        tk = torch.randn(B, N, Hkv, D, generator=g, device=dev).to(bf)
        tv = torch.randn(B, N, Hkv, D, generator=g, device=dev).to(bf)
        kc = torch.zeros(B, Hkv, S, D, device=dev, dtype=bf)
        vc = torch.zeros_like(kc)
        kc[:, :, :L].normal_(generator=g)
        vc[:, :, :L].normal_(generator=g)
        import synth
        r = synth.rng(3)
        parents = torch.as_tensor(synth.random_tree(r, N)).to(torch.int32).repeat(B, 1).to(dev)
        plen = torch.full((B,), L, dtype=torch.int32, device=dev)
        o = torch.empty(B, N, Hq, D, device=dev, dtype=bf)
        a = e3._lib.verify_attn_args(q, tk, tv, kc, vc, parents, plen, o, max_prefix_len=L)
        ws = torch.empty(max(16, e3._lib.eagle3_verify_attn_workspace_size(a)), dtype=torch.uint8, device=dev)
        # default: q and tree_k taken as already rotated (the fused RoPE projection's output, as in the
        # step); --rope-in-attention: the call rotates them (and writes the rotated tree keys back)
        qkr = not args.rope_in_attention
        a = e3._lib.verify_attn_args(q, tk, tv, kc, vc, parents, plen, o, max_prefix_len=L, qk_rotated=qkr)
        fn = _raw_call(e3._lib.lib().eagle3_verify_attn, a, ws)
        ms = _time_loop(fn, args.steps, args.warmup, flush if B * L * 4096 < 512e6 else None)
        nbytes = B * (4096 * L + 245760 + 983040 + (0 if qkr else 122880))
        out.update(batch=B, prefix=L, qk_rotated=qkr, ms=round(ms, 4), gbs=round(nbytes / ms / 1e6, 1),
                   frac_measured=round(nbytes / ms / 1e6 / hbm, 4), frac_8tbs=round(nbytes / ms / 1e6 / 8000, 4),
                   tflops=round(983040 * L * B / ms / 1e9, 1), bytes=nbytes)
    elif args.kernel == "accept":
        import synth
        B, N, V, W = args.batch, 60, 128256, 7
        mode = {"greedy": e3.GREEDY, "topk": e3.TOPK, "sampled": e3.SAMPLED}[args.mode]
        zt, zd, parents, tokens = synth.accept_batch(1, B, N, V, sampled=mode == e3.SAMPLED)
        zt_d = torch.as_tensor(zt, device=dev)
        zd_d = torch.as_tensor(zd, device=dev) if mode == e3.SAMPLED else None
        tok_d = torch.as_tensor(tokens, device=dev)
        par_d = torch.as_tensor(parents, device=dev)
        alen = torch.empty(B, dtype=torch.int32, device=dev)
        path = torch.empty(B, W, dtype=torch.int32, device=dev)
        emitted = torch.empty(B, W, dtype=torch.int32, device=dev)
        nroot = torch.empty(B, dtype=torch.int32, device=dev)
        ws = torch.empty(2 * B * V * 4 + 16, dtype=torch.uint8, device=dev)
        a = e3._lib.AcceptArgs(mode=int(mode), batch=B, n_nodes=N, vocab=V, max_path=W, temperature=1.0, seed=1,
                               step=0, target_logits=zt_d.data_ptr(),
                               draft_logits=zd_d.data_ptr() if zd_d is not None else None,
                               tokens=tok_d.data_ptr(), parents=par_d.data_ptr(), accept_len=alen.data_ptr(),
                               path=path.data_ptr(), emitted=emitted.data_ptr(), next_root=nroot.data_ptr(),
                               dev_status=None, step_counter=None)
        fn = _raw_call(e3._lib.lib().eagle3_accept, a, ws)
        ms = _time_loop(fn, args.steps, args.warmup, flush)   # the visited rows fit in L2: flush between calls
        visited = int((alen.to(torch.int64) + 1).sum().item())
        rows = visited * (2 if mode == e3.SAMPLED else 1)
        nbytes = rows * V * 4
        out.update(batch=B, mode=args.mode, ms=round(ms, 4), visited_rows=visited,
                   gbs_visited=round(nbytes / ms / 1e6, 1), us=round(ms * 1e3, 1))
    elif args.kernel == "draft":
        c = dict(CFG)
        c["B"] = args.batch
        eng = Engine(c, 4, dev, timing=False)
        so = eng.step_obj
        B = c["B"]
        tc1 = torch.ones(B, dtype=torch.int32, device=dev)
        dl0 = eng.draft_len.clone()
        # a reduced draft vocabulary: its own [Vd, d] head and the sorted target ids it covers
        Vd = args.draft_vocab if args.draft_vocab > 0 else c["V"]
        dw, d2t = so.draft_w, None
        if Vd != c["V"]:
            cpu_g = torch.Generator().manual_seed(7)
            dw = dict(so.draft_w)
            dw["lm_head"] = (torch.randn(Vd, c["d"], generator=cpu_g) * 0.02).to(torch.bfloat16).to(dev)
            d2t = torch.randperm(c["V"], generator=cpu_g)[:Vd].sort().values.to(torch.int32).to(dev)
        a = e3._lib.draft_tree_args(eng.aux_in, eng.next_tok, tc1, so.dk_cache, so.dv_cache, eng.draft_len,
                                    so.tokens, so.parents, so.depth, so.anc, so.score, n_heads=c["Hq"],
                                    ffn=c["F"], vocab=c["V"], depth=c["depth"], top_k=c["top_k"],
                                    max_draft_len=c["L0"], d2t=d2t)
        ws = torch.empty(e3._lib.eagle3_draft_tree_workspace_size(a), dtype=torch.uint8, device=dev)

        def fn():
            eng.draft_len.copy_(dl0)
            e3.eagle3_draft_tree(dw, eng.aux_in, eng.next_tok, tc1, so.dk_cache, so.dv_cache,
                                 eng.draft_len, so.tokens, so.parents, so.depth, so.anc, so.score,
                                 n_heads=c["Hq"], ffn=c["F"], vocab=c["V"], depth=c["depth"], top_k=c["top_k"],
                                 max_draft_len=c["L0"], d2t=d2t, workspace=ws)
        ms_eager = _time_loop(fn, args.steps, args.warmup)
        # the call as the step runs it: captured once into a CUDA graph and replayed (eager issue of
        # its ~70 launches from the host can take longer than the GPU work at small batches)
        cap = torch.cuda.Stream(device=dev)
        cap.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(cap):
            fn()
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=cap):
            fn()
        ms = _time_loop(graph.replay, args.steps, args.warmup)
        out.update(ms_eager=round(ms_eager, 4))
        d, F, V, qw = c["d"], c["F"], Vd, so.qkv_w
        layer = lambda m: 2 * m * (2 * d * qw + c["Hq"] * 128 * d + 2 * d * F + F * d)
        rows_c = B           # one real catch-up row per sequence (tc = 1); the launch pads to tc_max rows
        flops = 2 * rows_c * 3 * d * d + layer(rows_c) + 2 * B * d * V + 5 * (layer(10 * B) + 2 * 10 * B * d * V)
        wbytes = 2 * (3 * d * d + 2 * d * qw + c["Hq"] * 128 * d + 3 * d * F + d * V)
        out.update(batch=B, draft_vocab=Vd, ms=round(ms, 4), tflops=round(flops / ms / 1e9, 1),
                   frac_tensor=round(flops / ms / 1e9 / tf_sust, 4),
                   weight_gbs_6_passes=round(6 * wbytes / ms / 1e6, 1))
    elif args.kernel == "gemm":
        # one projection of the target layer at the step's shape (default: the SwiGLU gate + up
        # projection, M = B * N rows); x, w, w2 random bf16, output bf16
        M = args.m if args.m > 0 else args.batch * CFG["N"]
        N, K = args.n, args.k
        bf = torch.bfloat16
        x = (torch.randn(M, K, generator=g, device=dev) * 0.5).to(bf)
        w = (torch.randn(N, K, generator=g, device=dev) * 0.02).to(bf)
        epi = {"swiglu": e3.EPI_SWIGLU, "bf16": e3.EPI_BF16, "f32": e3.EPI_F32,
               "residual": e3.EPI_BF16_RESIDUAL}[args.epilogue]
        w2 = (torch.randn(N, K, generator=g, device=dev) * 0.02).to(bf) if epi == e3.EPI_SWIGLU else None
        res = torch.randn(M, N, generator=g, device=dev).to(bf) if epi == e3.EPI_BF16_RESIDUAL else None
        o = torch.empty(M, N, device=dev, dtype=torch.float32 if epi == e3.EPI_F32 else bf)
        ws = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
        a = e3._lib.LinearArgs(m=M, n=N, k=K, epilogue=epi, splits=0, ld_x=0, ld_w=0, ld_out=0, ld_res=0,
                               x=x.data_ptr(), w=w.data_ptr(), w2=None if w2 is None else w2.data_ptr(),
                               out=o.data_ptr(), residual=None if res is None else res.data_ptr(), dev_status=None,
                               rope_cols=0, rope_rows_per_seq=1, rope_theta=500000.0, rope_base=None,
                               rope_depth=None, row_max=None)
        fn = _raw_call(e3._lib.lib().eagle3_linear, a, ws)
        big = (x.numel() + w.numel() * (2 if w2 is not None else 1)) * 2 > 256e6   # inputs well beyond L2
        ms = _time_loop(fn, args.steps, args.warmup, None if big else flush)
        flops = 2.0 * M * N * K * (2 if w2 is not None else 1)
        out.update(m=M, n=N, k=K, epilogue=args.epilogue, ms=round(ms, 4), tflops=round(flops / ms / 1e9, 1),
                   frac_sustained=round(flops / ms / 1e9 / tf_sust, 4), frac_burst=round(flops / ms / 1e9 / tf_burst, 4))
    elif args.kernel == "next":
        # the NEXT rows, each on its prepared C call: the verify attention through block tables (paged
        # KV) beside the contiguous cache, the training-time-test attention, the chain rejection
        # sampler of a ragged batch and the batch's index bookkeeping
        import ctypes

        import numpy as np

        import synth
        L_ = e3._lib
        lib = L_.lib()
        stp = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
        bf, i32 = torch.bfloat16, torch.int32
        cpu_g = torch.Generator().manual_seed(11)
        B, N, Hq, Hkv, D = 64, 60, 32, 8, 128
        paged = {}
        for Lp in (2048, 4096):
            q = torch.randn(B, N, Hq, D, generator=g, device=dev).to(bf)
            tk = torch.randn(B, N, Hkv, D, generator=g, device=dev).to(bf)
            tv = torch.randn(B, N, Hkv, D, generator=g, device=dev).to(bf)
            parents = torch.as_tensor(synth.random_tree(synth.rng(3), N)).to(i32).repeat(B, 1).to(dev)
            plen = torch.full((B,), Lp, dtype=i32, device=dev)
            o = torch.empty(B, N, Hq, D, device=dev, dtype=bf)
            nbytes = B * (4096 * Lp + 245760 + 983040)     # as the contiguous call (the pool is read once too)
            row = {}
            for bs in (0, 64, 256):                         # 0: the contiguous cache
                if bs == 0:
                    kc = torch.randn(B, Hkv, Lp + 64, D, generator=g, device=dev).to(bf)
                    vc = torch.randn(B, Hkv, Lp + 64, D, generator=g, device=dev).to(bf)
                    a = L_.verify_attn_args(q, tk, tv, kc, vc, parents, plen, o, max_prefix_len=Lp, qk_rotated=True)
                else:
                    max_blocks = (Lp + bs - 1) // bs + 1
                    n_pages = B * max_blocks
                    bt = torch.randperm(n_pages, generator=cpu_g).view(B, max_blocks).to(i32).to(dev)
                    kc = torch.randn(n_pages * bs, Hkv, D, generator=g, device=dev).to(bf)
                    vc = torch.randn(n_pages * bs, Hkv, D, generator=g, device=dev).to(bf)
                    a = L_.verify_attn_args(q, tk, tv, kc, vc, parents, plen, o, max_prefix_len=Lp, qk_rotated=True,
                                            block_table=bt, block_size=bs)
                ws = torch.empty(max(16, L_.eagle3_verify_attn_workspace_size(a)), dtype=torch.uint8, device=dev)
                ms = _time_loop(_raw_call(lib.eagle3_verify_attn, a, ws), args.steps, args.warmup)
                row["contiguous" if bs == 0 else f"block_size_{bs}"] = {
                    "ms": round(ms, 4), "frac_hbm": round(nbytes / ms / 1e6 / hbm, 4)}
                del kc, vc
            paged[f"prefix_{Lp}"] = row
        out["paged_verify_attn"] = dict(paged, batch=B, nodes=N, bytes_per_call="B * (4096 L + 1.23 MB)")
        # training-time-test attention: 8 sequences of 2048 positions, the native step and 2 simulated
        Bt, T, S_ = 8, 2048, 3
        q = torch.randn(Bt, T, Hq, D, generator=g, device=dev).to(bf)
        k = torch.randn(S_, Bt, T, Hkv, D, generator=g, device=dev).to(bf)
        v = torch.randn(S_, Bt, T, Hkv, D, generator=g, device=dev).to(bf)
        o = torch.empty_like(q)
        a = L_.TttAttnArgs(batch=Bt, seq_len=T, n_heads=Hq, n_kv_heads=Hkv, head_dim=D, n_steps=S_, sm_scale=0.0,
                           q=q.data_ptr(), k=k.data_ptr(), v=v.data_ptr(), out=o.data_ptr(), dev_status=None)
        ws = torch.empty(max(16, lib.eagle3_ttt_attn_workspace_size(ctypes.byref(a))), dtype=torch.uint8, device=dev)
        ms = _time_loop(_raw_call(lib.eagle3_ttt_attn, a, ws), args.steps, args.warmup)
        flops = 4.0 * D * Bt * Hq * (T * (T + 1) / 2 + T * (S_ - 1))   # causal QK and PV, plus the diagonal keys
        out["ttt_attn"] = {"batch": Bt, "seq_len": T, "steps": S_, "heads": [Hq, Hkv], "ms": round(ms, 4),
                           "tflops": round(flops / ms / 1e9, 1), "frac_burst": round(flops / ms / 1e9 / tf_burst, 4)}
        del q, k, v, o
        # chain rejection sampler: 64 requests of 0..5 drafts over V = 128256 (logits N(0, 3^2)), and the
        # ragged batch's index bookkeeping
        R, K, V = 64, 5, 128256
        d, logits, drafts, greedy = synth.chain_batch(7, R, K, V)
        z = torch.as_tensor(logits, device=dev)
        dr = torch.as_tensor(drafts, dtype=i32, device=dev)
        cu = torch.as_tensor(np.cumsum(d).astype(np.int32), device=dev)
        gr = torch.as_tensor(greedy, dtype=i32, device=dev)
        oc = torch.empty(R, K + 1, dtype=i32, device=dev)
        nacc = torch.empty(R, dtype=i32, device=dev)
        a = L_.ChainVerifyArgs(n_requests=R, vocab=V, max_drafts=K, temperature=1.0, seed=2, step=0,
                               logits=z.data_ptr(), draft_tokens=dr.data_ptr(), cu_num_draft_tokens=cu.data_ptr(),
                               is_greedy=gr.data_ptr(), output_tokens=oc.data_ptr(), num_accepted=nacc.data_ptr(),
                               dev_status=None, step_counter=None)
        ms = _time_loop(lambda: lib.eagle3_chain_verify(ctypes.byref(a), stp), args.steps, args.warmup, flush)
        torch.cuda.synchronize()
        visited = int((nacc.to(torch.int64) + 1).sum())     # rows each request's walk reads
        out["chain_verify"] = {"requests": R, "max_drafts": K, "vocab": V, "rows": int(z.shape[0]),
                               "rows_visited": visited, "us": round(ms * 1e3, 1),
                               "gbs_two_passes_per_visited_row": round(2 * visited * V * 4 / ms / 1e6, 1)}
        nd = torch.as_tensor(d, device=dev)
        cu_sched = torch.as_tensor(np.cumsum(d + 1).astype(np.int32), device=dev)
        max_rows = int(d.sum()) + R
        li = torch.empty(max_rows, dtype=i32, device=dev)
        tli = torch.empty(max_rows, dtype=i32, device=dev)
        bli = torch.empty(R, dtype=i32, device=dev)
        nrows = torch.empty(1, dtype=i32, device=dev)
        a = L_.SpecDecodeMetadataArgs(n_requests=R, max_rows=max_rows, cu_num_scheduled_tokens=cu_sched.data_ptr(),
                                      num_draft_tokens=nd.data_ptr(), cu_num_draft_tokens=cu.data_ptr(),
                                      logits_indices=li.data_ptr(), target_logits_indices=tli.data_ptr(),
                                      bonus_logits_indices=bli.data_ptr(), num_rows=nrows.data_ptr(), dev_status=None)
        ms = _time_loop(lambda: lib.eagle3_spec_decode_metadata(ctypes.byref(a), stp), args.steps, args.warmup)
        out["spec_decode_metadata"] = {"requests": R, "us": round(ms * 1e3, 2)}
    elif args.kernel == "tiny":
        # the tiny lossless configuration (fp32, 4-layer d = 64 target and its EAGLE-3 head, 32-token
        # prompt): greedy speculative decoding with a K = 4 chain and vanilla greedy decoding, 64 new
        # tokens each, timed on the wall clock (the loop is host-driven: the accepted length is read
        # back every cycle); both must produce the same tokens
        import synth
        from eagle_tree_speculative_spec_gb300 import tiny
        cfg = synth.TINY
        tw = synth.llama_weights(0, **cfg)
        dw = synth.eagle3_weights(0, cfg["d"], cfg["n_heads"], cfg["n_kv_heads"], cfg["head_dim"], cfg["ffn"],
                                  cfg["vocab"], embed=tw["embed"], lm_head=tw["lm_head"])
        prompt, new = synth.tiny_prompt(0), 64
        make_t = lambda: tiny.TinyTarget(tw, cfg["n_layers"], cfg["n_heads"], cfg["n_kv_heads"], cfg["head_dim"],
                                         synth.TINY_AUX_LAYERS, 160, dev)
        make_d = lambda: tiny.TinyDraft(dw, cfg["n_heads"], cfg["n_kv_heads"], cfg["head_dim"], 160, dev)

        def timed(fn, reps):
            ts, res = [], None
            for _ in range(reps):
                objs = fn[1]()                       # weights uploaded outside the timed region
                torch.cuda.synchronize()
                t0 = time.perf_counter()
                res = fn[0](*objs)
                torch.cuda.synchronize()
                ts.append(time.perf_counter() - t0)
            return sorted(ts)[len(ts) // 2], res
        spec = (lambda t, d: tiny.speculative_greedy(t, d, prompt, new, k_draft=4), lambda: (make_t(), make_d()))
        van = (lambda t: tiny.vanilla_greedy(t, prompt, new), lambda: (make_t(),))
        timed(spec, 1)
        timed(van, 1)
        reps = max(3, args.steps)
        t_spec, (tok_spec, accepted) = timed(spec, reps)
        t_van, tok_van = timed(van, reps)
        out.update(new_tokens=new, speculative_ms_per_token=round(1e3 * t_spec / new, 4),
                   vanilla_ms_per_token=round(1e3 * t_van / new, 4), cycles=len(accepted),
                   accepted_per_cycle=round(sum(accepted) / len(accepted), 3),
                   speculative_equals_vanilla=tok_spec == tok_van, dtype="f32")
        if not args.no_cpu_baseline:
            # the oracle on the host: the same two decodes in fp64 NumPy, one run each
            from oracle import draft_tree as odt
            from oracle import llama as oll
            ot = oll.Llama(tw, cfg["n_layers"], cfg["n_heads"], cfg["n_kv_heads"], cfg["head_dim"],
                           aux_layers=synth.TINY_AUX_LAYERS)
            od = oll.Eagle3Draft(dw, cfg["n_heads"], cfg["n_kv_heads"], cfg["head_dim"])

            def chain(draft, d_cache, a_last, pending, L):
                r = odt.draft_tree_for_sequence(draft, d_cache, a_last, pending, L, 4, 1, 5)
                return r["tokens"].tolist(), r["parents"].tolist()
            t0 = time.perf_counter()
            ref_spec, _ = oll.speculative_greedy(ot, od, prompt, new, chain)
            t1 = time.perf_counter()
            ref_van = oll.vanilla_greedy(ot, prompt, new)
            t2 = time.perf_counter()
            out["cpu_baseline"] = {"kind": "oracle", "cores": host_threads(), "unit": "ms/token",
                                   "speculative_ms_per_token": round(1e3 * (t1 - t0) / new, 3),
                                   "vanilla_ms_per_token": round(1e3 * (t2 - t1) / new, 3),
                                   "sample": "the full 64-token runs, single process",
                                   "matches_gpu": ref_spec == tok_spec and ref_van == tok_van}
    print(json.dumps(out), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--batch", type=int, default=64)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--eager", action="store_true", help="issue every C call from the host instead of "
                                                          "replaying captured CUDA graphs")
    ap.add_argument("--generate", type=int, default=0,
                    help="run until every sequence has this many new tokens and report the acceptance length")
    ap.add_argument("--m", type=int, default=0, help="--kernel gemm: rows (default batch x tree nodes)")
    ap.add_argument("--n", type=int, default=CFG["F"], help="--kernel gemm: output features")
    ap.add_argument("--k", type=int, default=CFG["d"], help="--kernel gemm: input features")
    ap.add_argument("--epilogue", default="swiglu", choices=["swiglu", "bf16", "f32", "residual"])
    ap.add_argument("--draft-vocab", type=int, default=0,
                    help="--kernel draft: a reduced draft vocabulary of this many target ids (0 = all)")
    ap.add_argument("--kernel", choices=["verify_attn", "accept", "draft", "gemm", "tiny", "next"],
                    help="time one kernel of the path instead of the whole step")
    ap.add_argument("--prefix", type=int, default=4096)
    ap.add_argument("--mode", default="topk", choices=["greedy", "topk", "sampled"])
    ap.add_argument("--norm-kernels", action="store_true",
                    help="run every RMSNorm of the target as its own kernel instead of folding it into the "
                         "neighbouring projections")
    ap.add_argument("--rope-in-attention", action="store_true",
                    help="plain QKV projection, RoPE applied inside the verify attention (the unfused path)")
    args = ap.parse_args()
    if args.warmup < 3 and not args.kernel:
        args.warmup = 3
    if args.generate:
        run_generate(args)
    elif args.kernel:
        run_kernel(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
