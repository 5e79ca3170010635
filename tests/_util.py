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
