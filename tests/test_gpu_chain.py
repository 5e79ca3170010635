"""GPU parity of the ragged chain entry points (include/eagle3_chain.h) against the oracle.

* eagle3_spec_decode_metadata: the worked example of "Speculative Decoding (EAGLE3) in the vLLM
  Neuron Framework", section "SpecDecodeMetadata: Index Bookkeeping" (tests/golden), and random
  ragged batches against oracle.ragged, bit-exact; capacity and inconsistent counts are flagged.
* eagle3_chain_verify: every output token and acceptance count bit-exact against
  oracle.chain_sampler.chain_verify_specified on the same logits, at the full vocabulary
  (128256), greedy and random requests mixed, on consecutive Philox steps.
"""
import os

import numpy as np
import pytest
import torch

import synth
from oracle import chain_sampler as ocs
from oracle import ragged as oragged
from tests._util import require_gpu

pytestmark = pytest.mark.gpu


def _meta_gpu(cu_sched, d, max_rows):
    from eagle_tree_speculative_spec_gb300 import eagle3_spec_decode_metadata
    dev = require_gpu()
    R = len(d)
    i32 = dict(dtype=torch.int32, device=dev)
    out = dict(cu=torch.full((R,), -7, **i32), li=torch.full((max_rows,), -7, **i32),
               ti=torch.full((max_rows,), -7, **i32), bi=torch.full((R,), -7, **i32), n=torch.zeros(1, **i32),
               st=torch.zeros(1, **i32))
    eagle3_spec_decode_metadata(torch.as_tensor(cu_sched, **i32), torch.as_tensor(d, **i32), out["cu"], out["li"],
                                out["ti"], out["bi"], out["n"], dev_status=out["st"])
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in out.items()}


def test_metadata_worked_example(golden_dir):
    rows = {}
    for line in open(os.path.join(golden_dir, "spec_decode_metadata_5req.txt")):
        if line.strip() and not line.startswith("#"):
            k, v = line.split(":")
            rows[k.strip()] = [int(x) for x in v.split()]
    g = _meta_gpu(rows["cu_num_scheduled_tokens"], rows["num_draft_tokens"], 16)
    n = int(g["n"][0])
    assert g["st"][0] == 0 and n == len(rows["logits_indices"])
    assert g["cu"].tolist() == rows["cu_num_draft_tokens"]
    assert g["li"][:n].tolist() == rows["logits_indices"]
    nt = len(rows["target_logits_indices"])
    assert g["ti"][:nt].tolist() == rows["target_logits_indices"]
    assert g["bi"].tolist() == rows["bonus_logits_indices"]


@pytest.mark.parametrize("R", [1, 37, 3000])
def test_metadata_random_batches(R):
    r = np.random.default_rng(R)
    d = r.integers(0, 8, R)
    sched = d + 1 + r.integers(0, 50, R)
    cu = np.cumsum(sched)
    ref = oragged.spec_decode_metadata(cu, d)
    g = _meta_gpu(cu, d, int(d.sum()) + R)
    n = int(g["n"][0])
    assert g["st"][0] == 0 and n == len(ref["logits_indices"])
    assert np.array_equal(g["cu"], ref["cu_num_draft_tokens"])
    assert np.array_equal(g["li"][:n], ref["logits_indices"])
    assert np.array_equal(g["ti"][: int(d.sum())], ref["target_logits_indices"])
    assert np.array_equal(g["bi"], ref["bonus_logits_indices"])


def test_metadata_flags():
    from eagle_tree_speculative_spec_gb300._lib import DEV_BAD_COUNTS, DEV_CAPACITY
    g = _meta_gpu([4, 104, 107], [3, 0, 2], 5)          # (3 + 1) + (0 + 1) + (2 + 1) = 8 rows, 5 available
    assert g["st"][0] & DEV_CAPACITY and int(g["n"][0]) == 8
    g = _meta_gpu([4, 5, 9], [3, 1, 0], 16)            # request 1 schedules 1 token for 1 draft
    assert g["st"][0] & DEV_BAD_COUNTS


def _chain_gpu(logits, d, drafts, greedy, K, T, seed, steps, step_counter=True, bad=None):
    from eagle_tree_speculative_spec_gb300 import eagle3_chain_verify
    dev = require_gpu()
    R = len(d)
    i32 = dict(dtype=torch.int32, device=dev)
    z = torch.as_tensor(logits, device=dev)
    dr = torch.as_tensor(drafts if len(drafts) else np.zeros(1, np.int32), **i32)
    cu = torch.as_tensor(np.cumsum(d).astype(np.int32), **i32)
    gr = torch.as_tensor(greedy, **i32)
    ctr = torch.zeros(1, dtype=torch.int64, device=dev) if step_counter else None
    outs = []
    for s in range(steps):
        out = torch.full((R, K + 1), -7, **i32)
        nacc = torch.full((R,), -7, **i32)
        st = torch.zeros(1, **i32)
        eagle3_chain_verify(z, dr, cu, out, is_greedy=gr, num_accepted=nacc, temperature=T, seed=seed,
                            step=0 if step_counter else s, dev_status=st, step_counter=ctr)
        torch.cuda.synchronize()
        outs.append((out.cpu().numpy(), nacc.cpu().numpy(), int(st.item())))
    return outs


def _chain_ref(logits, d, drafts, greedy, K, T, seed, step, r):
    row0 = int(d[:r].sum()) + r
    start = int(d[:r].sum())
    out, n = ocs.chain_verify_specified(logits[row0: row0 + d[r] + 1], drafts[start: start + d[r]], bool(greedy[r]),
                                        T, seed, step, r)
    return out + [-1] * (K + 1 - len(out)), n


@pytest.mark.parametrize("R,K,V,T", [(64, 5, 128256, 1.0), (9, 3, 1001, 0.7),
                                     (6, 2, 5, 1.0)])   # V = 5: most CTAs of a cluster get an empty slice
def test_chain_verify_matches_oracle(R, K, V, T):
    d, logits, drafts, greedy = synth.chain_batch(R + V, R, K, V)
    seed = 2
    res = _chain_gpu(logits, d, drafts, greedy, K, T, seed, steps=2)
    kept = 0
    for step, (out, nacc, st) in enumerate(res):
        assert st == 0
        for r in range(R):
            ref, n = _chain_ref(logits, d, drafts, greedy, K, T, seed, step, r)
            assert nacc[r] == n, (step, r)
            assert out[r].tolist() == ref, (step, r, out[r], ref)
            kept += n
    assert kept > 0                                    # some drafts are accepted


def test_chain_verify_skips_bad_requests():
    from eagle_tree_speculative_spec_gb300._lib import DEV_BAD_TOKEN
    V, K = 500, 2
    d = np.array([1, 2, 0], np.int32)
    logits = np.random.default_rng(3).standard_normal((int(d.sum()) + 3, V)).astype(np.float32)
    drafts = np.array([3, 4, V + 9], np.int32)         # request 1's second draft is out of range
    out, nacc, st = _chain_gpu(logits, d, drafts, np.zeros(3, np.int32), K, 1.0, 0, steps=1)[0]
    assert st & DEV_BAD_TOKEN
    assert nacc[1] == -1 and (out[1] == -1).all()
    for r in (0, 2):
        ref, n = _chain_ref(logits, d, drafts, np.zeros(3, np.int32), K, 1.0, 0, 0, r)
        assert out[r].tolist() == ref and nacc[r] == n
