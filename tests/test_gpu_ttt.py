"""GPU parity of eagle3_ttt_attn (training-time-test attention) against oracle.attention.ttt_attention
("EAGLE-3: Engineering Implementation of LLM Inference Acceleration", sections VII.5 and VIII.2: causal
over the native step, the diagonal of every simulated step), bf16 tolerance 2e-2 abs + 1e-2 rel."""
import math

import numpy as np
import pytest
import torch

import synth
from oracle import attention as oatt
from tests._util import close, require_gpu

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("Bt,T,Hq,Hkv,S", [(2, 128, 32, 8, 3), (1, 256, 32, 8, 1), (2, 192, 16, 2, 2),
                                          (1, 64, 8, 8, 4)])
def test_ttt_attention_matches_oracle(Bt, T, Hq, Hkv, S):
    from eagle_tree_speculative_spec_gb300 import eagle3_ttt_attn
    dev = require_gpu()
    D = 128
    inp = synth.ttt_batch(T + S, Bt, T, Hq, Hkv, D, S)
    out = torch.full((Bt, T, Hq, D), float("nan"), dtype=torch.bfloat16, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    eagle3_ttt_attn(inp["q"].to(dev), inp["k"].to(dev), inp["v"].to(dev), out, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    got = out.float().cpu().numpy()
    for b in range(Bt):
        ref = oatt.ttt_attention(inp["q_f32"][b], [inp["k_f32"][s, b] for s in range(S)],
                                 [inp["v_f32"][s, b] for s in range(S)], 1.0 / math.sqrt(D))
        ok, err = close(got[b], ref, 2e-2, 1e-2)
        assert ok, (b, err)


def test_ttt_rejects_unsupported_lengths():
    from eagle_tree_speculative_spec_gb300 import Eagle3Error, eagle3_ttt_attn
    dev = require_gpu()
    q = torch.zeros(1, 96, 32, 128, dtype=torch.bfloat16, device=dev)
    k = torch.zeros(2, 1, 96, 8, 128, dtype=torch.bfloat16, device=dev)
    with pytest.raises(Eagle3Error):
        eagle3_ttt_attn(q, k, k.clone(), q.clone())
