"""eagle3_verify_attn_noalloc: the verify attention for callers that cannot allocate device memory.

Some callers cannot hand the library a workspace: their device memory is owned by a pool that
was sized before the first step, or they must not allocate while a step is captured into a CUDA
graph.  This entry point keeps its split-KV partials in a fixed static scratch array instead.
It must give the same results as eagle3_verify_attn (the entry point with a workspace), on
consecutive calls (the scratch is shared and keeps the previous call's contents), and reject a
split plan that does not fit the scratch.

The file is named to be collected last, so a run that stops at the first failure has already run
every other test.
"""
import numpy as np
import pytest
import torch

import synth
from tests._util import close, require_gpu

pytestmark = pytest.mark.gpu
ATOL, RTOL = 2e-2, 1e-2


def _inputs(seed, B, L):
    return synth.verify_attn_batch(seed, B, 60, 32, 8, 128, [L] * B, S_max=L + 64)


def _run(fn_name, inp, L, dev, **kw):
    import eagle_tree_speculative_spec_gb300._lib as lib
    tk = inp["tree_k"].to(dev).clone()            # the call rotates the tree keys in place
    out = torch.full(inp["q"].shape, float("nan"), dtype=torch.bfloat16, device=dev)
    lse = torch.full(inp["q"].shape[:3], float("nan"), dtype=torch.float32, device=dev)
    getattr(lib, fn_name)(inp["q"].to(dev), tk, inp["tree_v"].to(dev), inp["k_cache"].to(dev),
                          inp["v_cache"].to(dev), torch.as_tensor(inp["parents"], device=dev),
                          torch.as_tensor(inp["prefix_len"], device=dev), out, lse=lse, max_prefix_len=L, **kw)
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), lse.cpu().numpy(), tk.float().cpu().numpy()


@pytest.mark.parametrize("B,L", [(1, 4096), (2, 2048)])
def test_noalloc_matches_workspace_entry_on_consecutive_calls(B, L):
    dev = require_gpu()
    first, second = _inputs(41, B, L), _inputs(42, B, L)
    for inp in (first, second):                   # two calls in a row, different inputs
        ref = _run("eagle3_verify_attn", inp, L, dev)
        got = _run("eagle3_verify_attn_noalloc", inp, L, dev)
        for g, r in zip(got, ref):
            ok, err = close(g, r, ATOL, RTOL)
            assert ok, err


def test_noalloc_uses_split_scratch():
    """The cases above split the prefix across CTAs, so the static scratch is really used."""
    dev = require_gpu()
    import eagle_tree_speculative_spec_gb300._lib as lib
    inp = _inputs(43, 1, 4096)
    args = lib.verify_attn_args(inp["q"].to(dev), inp["tree_k"].to(dev), inp["tree_v"].to(dev),
                                inp["k_cache"].to(dev), inp["v_cache"].to(dev),
                                torch.as_tensor(inp["parents"], device=dev),
                                torch.as_tensor(inp["prefix_len"], device=dev),
                                torch.empty(inp["q"].shape, dtype=torch.bfloat16, device=dev), max_prefix_len=4096)
    assert lib.eagle3_verify_attn_workspace_size(args) > 0


def test_noalloc_rejects_plans_beyond_the_scratch():
    dev = require_gpu()
    import eagle_tree_speculative_spec_gb300._lib as lib
    inp = _inputs(44, 64, 1024)
    with pytest.raises(lib.Eagle3Error) as e:
        # 64 sequences x 60 nodes x 32 heads x 8 splits x 520 bytes = 511 MB > 32 MiB
        _run("eagle3_verify_attn_noalloc", inp, 1024, dev, num_splits=8)
    assert e.value.status == 6
