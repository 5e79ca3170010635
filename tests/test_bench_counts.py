"""bench.py's algorithmic counts, which are the numerators of its roofline fractions, against
closed forms written from the model's shapes (host logic; no GPU)."""
import bench
from eagle_tree_speculative_spec_gb300.step import SpeculativeStep


def _engine(fused_rope=True):
    e = bench.Engine.__new__(bench.Engine)        # the count methods read only these fields
    e.cfg = dict(bench.CFG)
    c = e.cfg
    e.qkv_w = (c["Hq"] + 2 * c["Hkv"]) * c["D"]
    e.fused_rope = fused_rope
    so = SpeculativeStep.__new__(SpeculativeStep)   # flops() reads only these fields
    so.cfg, so.qkv_w, so.d2t = c, e.qkv_w, None
    e.step_obj = so
    return e


def test_target_flops_are_two_flops_per_weight_per_row():
    e = _engine()
    target, draft = e.flops_per_step()
    # Llama-3.1-8B-shaped layer: q/k/v 4096 x 6144, o 4096 x 4096, gate/up 2 x 4096 x 14336,
    # down 14336 x 4096; 32 layers plus the 4096 x 128256 LM head; 64 x 60 tree rows
    weights = 32 * (4096 * 6144 + 4096 * 4096 + 2 * 4096 * 14336 + 14336 * 4096) + 4096 * 128256
    assert weights == 7_504_658_432
    assert target == 2 * 3840 * weights
    # draft: fc on the real catch-up rows (one per sequence when nothing was accepted; the launch
    # pads to 7 per sequence, which is not counted), the layer (q/k/v read 2d inputs) on those rows
    # and on 5 x 640 frontier rows, the LM head on 64 root rows and on 5 x 640 frontier rows
    layer = 2 * 4096 * 6144 + 4096 * 4096 + 2 * 4096 * 14336 + 14336 * 4096
    want = 2 * (64 * 3 * 4096 * 4096 + 64 * layer + 64 * 4096 * 128256 + 5 * 640 * (layer + 4096 * 128256))
    assert draft == want
    # with accepted drafts the committed rows count: 2 rows for each of the 64 sequences
    _, draft2 = e.flops_per_step(128)
    assert draft2 - draft == 2 * 64 * (3 * 4096 * 4096 + layer)


def test_verify_attention_bytes_per_launch():
    L = 2048
    per_seq = 2 * 8 * L * 128 * 2 + 2 * 60 * 8 * 128 * 2 + 2 * 60 * 32 * 128 * 2   # prefix K+V, tree K+V, Q+O
    assert per_seq == 4096 * L + 245_760 + 983_040
    assert _engine(True).attn_bytes_per_launch(L) == 64 * per_seq
    # the call that rotates the tree keys itself also writes them back
    assert _engine(False).attn_bytes_per_launch(L) == 64 * (per_seq + 122_880)
