"""The whole-step usage example of the package's documentation, run as written: a SpeculativeStep
at a small shape with random weights, one eager step, then a captured CUDA graph replayed eight
times; every step commits accept_len + 1 >= 1 tokens per sequence and reports no device error."""
import pytest
import torch

from tests._util import require_gpu

pytestmark = pytest.mark.gpu


def test_step_usage_example():
    require_gpu()
    import eagle_tree_speculative_spec_gb300 as e3
    from eagle_tree_speculative_spec_gb300.step import SpeculativeStep
    prev = torch.cuda.current_stream()
    try:
        dev, bf = "cuda", torch.bfloat16
        side = torch.cuda.Stream()
        torch.cuda.set_stream(side)   # the prepared calls launch on the stream that is current at prepare()
        cfg = dict(layers=4, d=256, Hq=4, Hkv=2, D=128, F=512, V=1000, taps=(1, 2, 3), B=8, N=12, depth=4,
                   top_k=4, W=5, mode=e3.TOPK, temperature=1.0, seed=1, rope_theta=500000.0, eps=1e-5)
        d, F, V, L = cfg["d"], cfg["F"], cfg["V"], cfg["layers"]
        qkv, hd = (cfg["Hq"] + 2 * cfg["Hkv"]) * cfg["D"], cfg["Hq"] * cfg["D"]
        rnd = lambda *shape: (0.02 * torch.randn(*shape, device=dev)).to(bf)
        ones = lambda: torch.ones(d, device=dev, dtype=bf)
        target = {"embed": rnd(V, d), "lm_head": rnd(V, d), "final_norm": ones(),
                  "wqkv": [rnd(qkv, d) for _ in range(L)], "wo": [rnd(d, hd) for _ in range(L)],
                  "wg": [rnd(F, d) for _ in range(L)], "wu": [rnd(F, d) for _ in range(L)],
                  "wd": [rnd(d, F) for _ in range(L)], "norm1": [ones() for _ in range(L)],
                  "norm2": [ones() for _ in range(L)]}
        draft = {"w_fc": rnd(d, 3 * d), "embed": target["embed"], "input_norm": ones(), "hidden_norm": ones(),
                 "w_qkv": rnd(qkv, 2 * d), "w_o": rnd(d, hd), "post_norm": ones(), "w_gate": rnd(F, d),
                 "w_up": rnd(F, d), "w_down": rnd(d, F), "final_norm": ones(), "lm_head": rnd(V, d)}
        step = SpeculativeStep(cfg, target, draft, 512, 400, dev, fold_norms=True)
        # the state after a 100-token prompt: rotated K/V in the caches, the last position's aux states and token
        P = 100
        step.k_cache[..., :P, :].normal_(); step.v_cache[..., :P, :].normal_()
        step.dk_cache[..., :P - 1, :].normal_(); step.dv_cache[..., :P - 1, :].normal_()
        step.prefix_len.fill_(P); step.draft_len.fill_(P - 1); step.tc.fill_(1)
        step.aux_in[:, 0].normal_(); step.next_tok[:, 0] = torch.randint(0, V, (cfg["B"],), device=dev)
        step.prepare()
        step.run()                                   # one eager step
        graph = torch.cuda.CUDAGraph()               # then capture one step and replay it
        with torch.cuda.graph(graph, stream=side):
            step.run()
        for _ in range(8):
            graph.replay()
        torch.cuda.synchronize()
        assert int(step.dev_status) == 0             # no device-detected error
        advanced = (step.prefix_len - P).cpu()
        assert bool((advanced >= 9).all()) and bool((advanced <= 9 * (cfg["depth"] + 1)).all()), advanced
    finally:
        torch.cuda.set_stream(prev)
