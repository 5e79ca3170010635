"""Helpers shared by the tests (no method arithmetic here)."""
import os
import re

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", h) for h in sorted(os.listdir(os.path.join(ROOT, "include"))) if h.endswith(".h")]


def header_functions():
    """Names of the functions include/eagle3.h declares."""
    text = "".join(open(h).read() for h in HEADERS)
    return sorted(set(re.findall(r"^\s*(?:const\s+char\s*\*|eagle3_status_t|size_t|int)\s*(eagle3_\w+)\s*\(",
                                 text, flags=re.M)))


def built_lib():
    from eagle_tree_speculative_spec_gb300 import build
    build.build()
    from eagle_tree_speculative_spec_gb300 import _lib
    return _lib.lib()


def require_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    built_lib()
    return torch.device("cuda:0")


def close(got, want, atol, rtol):
    """Elementwise |got - want| <= atol + rtol * |want|; returns (ok, max_abs_err)."""
    import numpy as np
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    err = np.abs(got - want)
    return bool((err <= atol + rtol * np.abs(want)).all()), float(err.max()) if err.size else 0.0


def agreeing_proposer(ref, prompt_len, k, vocab, corrupt_every=3):
    """A stand-in draft that proposes the vanilla greedy continuation ``ref`` (so drafts are
    accepted), with one position corrupted in every ``corrupt_every``-th cycle (cycles 1, 4, 7, ...
    corrupt positions 0, 1, 2, ... in turn), so accept lengths cover k and values below it."""
    cycle = [0]

    def propose(n, root, kk):
        i = n - prompt_len                   # root is generated token i
        assert root == ref[i]
        nxt = [ref[i + 1 + j] if i + 1 + j < len(ref) else 0 for j in range(kk)]
        c = cycle[0]
        cycle[0] += 1
        if c % corrupt_every == 1:
            pos = (c // corrupt_every) % kk
            nxt[pos] = (nxt[pos] + 1) % vocab
        return nxt
    return propose
