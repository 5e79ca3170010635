"""The tiny lossless configuration on the GPU (fp32): a 4-layer d = 64 Llama-style target and its
EAGLE-3 head, chain draft of K = 4, greedy, 64 new tokens.  Speculative decoding on the GPU must
reproduce vanilla greedy decoding on the GPU token for token, and both must equal the oracle's
vanilla greedy output; the prompt pass's logits agree with the oracle within 1e-4."""
import numpy as np
import pytest
import torch

import synth
from oracle import llama
from tests._util import agreeing_proposer, require_gpu

pytestmark = pytest.mark.gpu


def _weights():
    cfg = synth.TINY
    tw = synth.llama_weights(0, **cfg)
    dw = synth.eagle3_weights(0, cfg["d"], cfg["n_heads"], cfg["n_kv_heads"], cfg["head_dim"], cfg["ffn"],
                              cfg["vocab"], embed=tw["embed"], lm_head=tw["lm_head"])
    return cfg, tw, dw


def _target(cfg, tw, dev, s_max=160):
    from eagle_tree_speculative_spec_gb300 import tiny
    return tiny.TinyTarget(tw, cfg["n_layers"], cfg["n_heads"], cfg["n_kv_heads"], cfg["head_dim"],
                           synth.TINY_AUX_LAYERS, s_max, dev)


def test_tiny_prompt_logits_match_oracle():
    from eagle_tree_speculative_spec_gb300 import tiny
    dev = require_gpu()
    cfg, tw, _ = _weights()
    prompt = synth.tiny_prompt(0)
    P = len(prompt)
    t = _target(cfg, tw, dev)
    logits, aux, _, _ = t.forward(prompt, list(range(P)), tiny.chain_visible(P), 0)
    torch.cuda.synchronize()
    ot = llama.Llama(tw, cfg["n_layers"], cfg["n_heads"], cfg["n_kv_heads"], cfg["head_dim"],
                     aux_layers=synth.TINY_AUX_LAYERS)
    ref, ref_aux, _, _ = ot.forward(prompt, np.arange(P), ot.new_cache(), llama.chain_visible(P))
    assert np.abs(logits.cpu().numpy() - ref).max() <= 1e-4
    assert np.abs(aux.cpu().numpy() - ref_aux).max() <= 1e-4


@pytest.mark.parametrize("prompt_seed", [0, 1])
def test_tiny_speculative_equals_vanilla_and_oracle(prompt_seed):
    from eagle_tree_speculative_spec_gb300 import tiny
    dev = require_gpu()
    cfg, tw, dw = _weights()
    prompt = synth.tiny_prompt(prompt_seed)
    vanilla = tiny.vanilla_greedy(_target(cfg, tw, dev), prompt, 64)
    draft = tiny.TinyDraft(dw, cfg["n_heads"], cfg["n_kv_heads"], cfg["head_dim"], 160, dev)
    spec, accepted = tiny.speculative_greedy(_target(cfg, tw, dev), draft, prompt, 64, k_draft=4)
    assert spec == vanilla
    assert len(spec) == 64 and all(0 <= a <= 4 for a in accepted)
    ot = llama.Llama(tw, cfg["n_layers"], cfg["n_heads"], cfg["n_kv_heads"], cfg["head_dim"],
                     aux_layers=synth.TINY_AUX_LAYERS)
    assert vanilla == llama.vanilla_greedy(ot, prompt, 64)


def test_tiny_speculative_with_accepted_drafts():
    """The same losslessness check with drafts that are accepted: a proposer that follows vanilla
    greedy (with a planted mismatch every third cycle) drives full acceptance of all 4 drafts and
    partial acceptance, so the GPU path runs multi-row commits, catch-ups of several rows and the
    draft-cache rollback after an accepted chain; the output still equals vanilla greedy."""
    from eagle_tree_speculative_spec_gb300 import tiny
    dev = require_gpu()
    cfg, tw, dw = _weights()
    prompt = synth.tiny_prompt(0)
    vanilla = tiny.vanilla_greedy(_target(cfg, tw, dev), prompt, 64)
    ot = llama.Llama(tw, cfg["n_layers"], cfg["n_heads"], cfg["n_kv_heads"], cfg["head_dim"],
                     aux_layers=synth.TINY_AUX_LAYERS)
    assert vanilla == llama.vanilla_greedy(ot, prompt, 64)
    propose = agreeing_proposer(vanilla, len(prompt), 4, cfg["vocab"])
    draft = tiny.TinyDraft(dw, cfg["n_heads"], cfg["n_kv_heads"], cfg["head_dim"], 160, dev)
    spec, accepted = tiny.speculative_greedy(_target(cfg, tw, dev), draft, prompt, 64, k_draft=4, propose=propose)
    assert spec == vanilla
    assert 4 in accepted and any(1 <= a <= 3 for a in accepted), accepted
