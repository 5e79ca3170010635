"""The timeout path of a bounded wait, on the GPU, without a fault or a hang.

Every wait inside the kernels gives up after a limit, sets EAGLE3_DEV_TIMEOUT, drains its copies,
frees its tensor memory and returns (include/eagle3.h).  The test hook eagle3_test_verify_attn_timeout
(include/eagle3_testing.h) runs the verify attention with one K tile never loaded and a short limit
(about a millisecond), so the wait for that tile runs out in every CTA.  Checked: the call returns,
the status word carries EAGLE3_DEV_TIMEOUT, and the same context then runs ordinary calls that
still match the oracle.
"""
import pytest
import torch

import synth
from oracle import attention as oatt
from tests._util import close, require_gpu

pytestmark = pytest.mark.gpu
ATOL, RTOL = 2e-2, 1e-2


@pytest.mark.parametrize("qk_rotated", [False, True])
def test_verify_attn_wait_runs_out_and_context_survives(qk_rotated):
    import eagle_tree_speculative_spec_gb300._lib as lib
    dev = require_gpu()
    B, N, Hq, Hkv, D, L = 3, 12, 32, 8, 128, 512
    inp = synth.verify_attn_batch(41, B, N, Hq, Hkv, D, [L, L - 100, 300], S_max=L + 64)

    def args():
        return (inp["q"].to(dev), inp["tree_k"].to(dev).clone(), inp["tree_v"].to(dev), inp["k_cache"].to(dev),
                inp["v_cache"].to(dev), torch.as_tensor(inp["parents"], device=dev),
                torch.as_tensor(inp["prefix_len"], device=dev),
                torch.zeros(B, N, Hq, D, dtype=torch.bfloat16, device=dev))

    st = torch.zeros(1, dtype=torch.int32, device=dev)
    a = args()
    lib.eagle3_test_verify_attn_timeout(*a, max_prefix_len=L, stall_tile=1, wait_limit_cycles=2_000_000,
                                        num_splits=1, dev_status=st, qk_rotated=qk_rotated)
    torch.cuda.synchronize()                        # the call returned: no hang
    assert int(st.item()) & lib.DEV_TIMEOUT
    # the context is still usable: an ordinary call on fresh inputs matches the oracle
    for _ in range(2):
        st2 = torch.zeros(1, dtype=torch.int32, device=dev)
        q, tk, tv, kc, vc, par, plen, out = args()
        lib.eagle3_verify_attn(q, tk, tv, kc, vc, par, plen, out, max_prefix_len=L, dev_status=st2)
        torch.cuda.synchronize()
        assert int(st2.item()) == 0
        ref_o, _, _ = oatt.verify_attention(inp["q_f32"], inp["tree_k_f32"], inp["tree_v_f32"], inp["k_cache_f32"],
                                            inp["v_cache_f32"], inp["parents"], inp["prefix_len"])
        ok, err = close(out.float().cpu().numpy(), ref_o, ATOL, RTOL)
        assert ok, err


def test_timeout_hook_rejects_bad_limits():
    import eagle_tree_speculative_spec_gb300._lib as lib
    dev = require_gpu()
    inp = synth.verify_attn_batch(42, 1, 4, 32, 8, 128, [64], S_max=128)
    q, tk, tv = inp["q"].to(dev), inp["tree_k"].to(dev), inp["tree_v"].to(dev)
    kc, vc = inp["k_cache"].to(dev), inp["v_cache"].to(dev)
    par = torch.as_tensor(inp["parents"], device=dev)
    plen = torch.as_tensor(inp["prefix_len"], device=dev)
    out = torch.zeros(1, 4, 32, 128, dtype=torch.bfloat16, device=dev)
    for stall, limit in ((-1, 10_000), (0, 10), (0, 10**10)):
        with pytest.raises(lib.Eagle3Error):
            lib.eagle3_test_verify_attn_timeout(q, tk, tv, kc, vc, par, plen, out, max_prefix_len=64,
                                                stall_tile=stall, wait_limit_cycles=limit)
