"""Philox4x32-10, the counter-based generator the acceptance stage draws from.

Definition: J. Salmon, M. Moraes, R. Dror, D. Shaw, "Parallel Random Numbers:
As Easy as 1, 2, 3", SC'11, section 3 (Philox-4x32 with 10 rounds).  The pages
on EAGLE-3 call for random draws (``torch.rand`` / ``multinomial`` in "EAGLE-3:
Engineering Implementation of LLM Inference Acceleration", section X) but name
no generator; a counter-based one lets the CPU and the GPU draw the same
numbers for the same (seed, step, sequence, node, slot).

Pinned by the published known-answer vectors (tests/golden/philox4x32_10_kat.txt).

Counter layout used by the acceptance stage (both sides implement it):
    c0 = slot + 256 * node      slot in [0, 256), node in [0, 2**24)
    c1 = b                      sequence index in the batch
    c2 = step & 0xffffffff      draft-and-verify cycle counter
    c3 = step >> 32
    key = (seed & 0xffffffff, seed >> 32)
    U32 = x0                    uniform 32-bit word
    R64 = (x1 << 32) | x2       uniform 64-bit word
Slots: s in [0, 64) the accept test of the s-th child (children in ascending
node index), 64 the residual / bonus draw at the node, 128 + s the draw of the
s-th child when children are sampled from the draft.
"""
import numpy as np

_M0 = 0xD2511F53
_M1 = 0xCD9E8D57
_W0 = 0x9E3779B9
_W1 = 0xBB67AE85
_MASK = 0xFFFFFFFF

SLOT_RESIDUAL = 64
SLOT_DRAW = 128


def philox4x32_10(ctr, key):
    """One Philox4x32-10 block: 4 counter words and 2 key words -> 4 words."""
    c0, c1, c2, c3 = (int(v) & _MASK for v in ctr)
    k0, k1 = (int(v) & _MASK for v in key)
    for rnd in range(10):
        if rnd:
            k0 = (k0 + _W0) & _MASK
            k1 = (k1 + _W1) & _MASK
        p0 = _M0 * c0
        p1 = _M1 * c2
        hi0, lo0 = p0 >> 32, p0 & _MASK
        hi1, lo1 = p1 >> 32, p1 & _MASK
        c0, c1, c2, c3 = hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0
    return c0, c1, c2, c3


def philox4x32_10_np(c0, c1, c2, c3, k0, k1):
    """Vectorised Philox4x32-10 over numpy arrays (uint32-valued, broadcastable)."""
    c0, c1, c2, c3 = (np.asarray(v, dtype=np.uint64) & _MASK for v in (c0, c1, c2, c3))
    k0 = np.asarray(k0, dtype=np.uint64) & _MASK
    k1 = np.asarray(k1, dtype=np.uint64) & _MASK
    m0, m1 = np.uint64(_M0), np.uint64(_M1)
    mask, sh = np.uint64(_MASK), np.uint64(32)
    for rnd in range(10):
        if rnd:
            k0 = (k0 + np.uint64(_W0)) & mask
            k1 = (k1 + np.uint64(_W1)) & mask
        p0 = m0 * c0
        p1 = m1 * c2
        c0, c1, c2, c3 = (p1 >> sh) ^ c1 ^ k0, p1 & mask, (p0 >> sh) ^ c3 ^ k1, p0 & mask
    return c0, c1, c2, c3


def counter(slot, node, b, step):
    return (slot + 256 * node, b, step & _MASK, (step >> 32) & _MASK)


def seed_key(seed):
    return (seed & _MASK, (seed >> 32) & _MASK)


def draw(seed, step, b, node, slot):
    """(U32, R64) for one acceptance decision."""
    x0, x1, x2, _ = philox4x32_10(counter(slot, node, b, step), seed_key(seed))
    return x0, (x1 << 32) | x2
