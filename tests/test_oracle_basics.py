"""Pins of the oracle's Philox, DSM, tree and compaction functions (CPU only)."""
import math
import os

import numpy as np
import pytest

import synth
from oracle import compact, dsm, philox, tree


def _read_rows(path):
    rows = []
    for line in open(path):
        line = line.strip()
        if line and not line.startswith("#"):
            rows.append(line)
    return rows


# ----------------------------------------------------------------------------- Philox
def test_philox_known_answers(golden_dir):
    rows = _read_rows(os.path.join(golden_dir, "philox4x32_10_kat.txt"))
    assert len(rows) == 3
    for row in rows:
        v = [int(x, 16) for x in row.split()]
        assert philox.philox4x32_10(v[0:4], v[4:6]) == tuple(v[6:10])


def test_philox_vectorised_matches_scalar():
    r = np.random.default_rng(5)
    c = r.integers(0, 2**32, size=(4, 257), dtype=np.uint64)
    k = r.integers(0, 2**32, size=(2, 257), dtype=np.uint64)
    out = philox.philox4x32_10_np(c[0], c[1], c[2], c[3], k[0], k[1])
    for i in range(257):
        ref = philox.philox4x32_10([int(x) for x in c[:, i]], [int(x) for x in k[:, i]])
        assert tuple(int(o[i]) for o in out) == ref


def test_philox_uniformity():
    # 2**16 words of the stream: mean and bit balance of a uniform 32-bit source
    n = 1 << 16
    out = philox.philox4x32_10_np(np.arange(n), 0, 0, 0, 123, 456)
    u = out[0].astype(np.float64) / 2**32
    assert abs(u.mean() - 0.5) < 4 * math.sqrt(1 / 12 / n)
    bits = np.unpackbits(out[1].astype(">u4").view(np.uint8))
    assert abs(bits.mean() - 0.5) < 4 * 0.5 / math.sqrt(bits.size)


# ----------------------------------------------------------------------------- DSM
def test_exp_matches_exp_within_ulps():
    t = np.concatenate([-np.random.default_rng(0).random(100000) * 64,
                        [0.0, -1e-30, -0.5, -1.0, -math.log(2.0), -63.999]]).astype(np.float32)
    e = dsm.exp_f32(t).astype(np.float64)
    ref = np.exp(t.astype(np.float64))
    rel = np.abs(e - ref) / ref
    assert rel.max() < 4 * 2.0 ** -24
    assert dsm.exp_f32(np.float32([0.0]))[0] == 1.0


def test_exp_underflow_and_monotone():
    assert dsm.exp_f32(np.float32([-64.5, -100.0, -np.inf])).tolist() == [0.0, 0.0, 0.0]
    t = np.sort(-np.random.default_rng(1).random(20000).astype(np.float32) * 30)
    e = dsm.exp_f32(t)
    assert np.all(np.diff(e.astype(np.float64)) >= 0)


@pytest.mark.parametrize("S", [2**31, 2**31 + 1, 3 * 2**31, 7 * 2**31 + 12345, 128256 * 2**31 - 1,
                               2**52 + 2**40 + 17, 2**31 * 1000003])
def test_log31_matches_log(S):
    got = float(dsm.log31(S))
    ref = math.log(S / 2**31)
    assert abs(got - ref) <= 4e-7 * max(1.0, abs(ref))


def test_weights_match_softmax():
    r = np.random.default_rng(2)
    for V, T in ((8, 1.0), (1000, 1.0), (128256, 1.0), (5000, 0.7), (5000, 2.5)):
        z = (3 * r.standard_normal(V)).astype(np.float32)
        W, S = dsm.weights(z, dsm.inv_temperature(T))
        assert W.max() == 2**31 and S == int(W.sum())
        p = W / S
        x = z.astype(np.float64) / T
        sm = np.exp(x - x.max())
        sm /= sm.sum()
        # truncation to 2**-31 per entry plus fp32 rounding of t_i
        assert np.abs(p - sm).max() <= V * 2.0**-31 + 2e-6 * sm.max()
        lq = dsm.logq(z) if T == 1.0 else None
        if lq is not None:
            big = sm > 1e-6
            assert np.abs(lq[big] - np.log(sm[big])).max() < 1e-5


def _logq_excess(fn, z, T):
    """Largest |fn(z) - log softmax(z / T)| over the row, divided by its error bound.

    The bound follows the arithmetic: t_i = fp32(fp32(z_i - m) * fp32(1/T)) is within 3 ulp-units
    (2**-24 relative each) of x_i = (z_i - m) / T; EXP is within 4 * 2**-24 relative; the weights
    are truncated to 2**-31 each against a sum of at least 1 (the maximum weighs 1), so S loses at
    most V * 2**-31 relative; LOG31 is within 4e-7 of ln(S * 2**-31) (max(1, |.|) relative); the
    final fp32 subtraction rounds by half an ulp of the result."""
    x = (z.astype(np.float64) - float(z.max())) / T
    lse = math.log(np.exp(x).sum())
    ref = x - lse
    got = fn(z, dsm.inv_temperature(T)).astype(np.float64)
    bound = (2.0**-22 * (np.abs(x) + np.abs(x).max() + 1.0) + len(z) * 2.0**-31
             + 4e-7 * max(1.0, lse) + 2.0**-23 * np.abs(ref))
    return float((np.abs(got - ref) / bound).max())


def _logq_sign_slip(z, inv_t):
    t = dsm.scaled(z, inv_t)
    return (t + dsm.log31(dsm.weights(z, inv_t)[1])).astype(np.float32)


def _logq_raw_logit(z, inv_t):
    t = (np.asarray(z, np.float32) * np.float32(inv_t)).astype(np.float32)
    return (t - dsm.log31(dsm.weights(z, inv_t)[1])).astype(np.float32)


def _logq_no_temperature(z, inv_t):
    return dsm.logq(z, np.float32(1.0))


def _logq_fix_bits_off_by_one(z, inv_t):
    t = dsm.scaled(z, inv_t)
    return (t - (dsm.log31(dsm.weights(z, inv_t)[1]) - np.float32(math.log(2.0)))).astype(np.float32)


@pytest.mark.parametrize("V", [8, 1000, 128256])
@pytest.mark.parametrize("T", [1.0, 0.7])
def test_logq_is_log_softmax(V, T):
    """logq = the log of the tempered softmax ("EAGLE-3: Engineering Implementation of LLM
    Inference Acceleration", section X, probs = softmax(z / T)), over whole N(0, 3^2) rows, within
    the bound of its fixed-point arithmetic; planted mistakes (sign of the normaliser, the row
    maximum not subtracted, the temperature dropped, the fixed point off by one bit) all fail."""
    r = np.random.default_rng(V + int(10 * T))
    z = (3 * r.standard_normal(V)).astype(np.float32) + np.float32(5.0)   # the maximum is not 0
    assert _logq_excess(dsm.logq, z, T) <= 1.0
    planted = [_logq_sign_slip, _logq_raw_logit, _logq_fix_bits_off_by_one]
    if T != 1.0:
        planted.append(_logq_no_temperature)
    for bad in planted:
        assert _logq_excess(bad, z, T) > 1.0, bad.__name__


def test_logq_of_certain_token_is_zero():
    z = np.full(16, -1000.0, np.float32)
    z[3] = 0.0
    lq = dsm.logq(z)
    assert lq[3] == 0.0


# ----------------------------------------------------------------------------- tree
def test_tree_mask_golden(golden_dir):
    rows = _read_rows(os.path.join(golden_dir, "tree_mask_6.txt"))
    parents = [int(x) for x in rows[0].split(":")[1].split()]
    want = np.array([[int(x) for x in r.split()] for r in rows[1:]], dtype=bool)
    assert (tree.mask_matrix(parents) == want).all()
    bits = tree.anc_bits(parents)
    for i in range(6):
        assert [(int(bits[i]) >> j) & 1 for j in range(6)] == want[i].astype(int).tolist()
    assert tree.depths(parents).tolist() == [0, 1, 1, 2, 2, 2]
    assert tree.positions(parents, 10).tolist() == [10, 11, 11, 12, 12, 12]


def test_bitmask_matches_brute_force_on_random_trees():
    r = np.random.default_rng(3)
    for n in (1, 2, 7, 60, 64):
        for _ in range(5):
            parents = synth.random_tree(r, n, max_depth=min(63, n), max_children=10)
            m = tree.mask_matrix(parents)
            bits = tree.anc_bits(parents)
            for i in range(n):
                row = np.array([(int(bits[i]) >> j) & 1 for j in range(n)], dtype=bool)
                assert (row == m[i]).all()
            # depth = number of strict ancestors
            assert (tree.depths(parents) == m.sum(1) - 1).all()


def test_random_tree_shape():
    r = np.random.default_rng(4)
    for _ in range(20):
        p = synth.random_tree(r, 60)
        tree.validate(p)
        d = tree.depths(p)
        assert d.max() <= 6
        counts = np.bincount(p[1:], minlength=60)
        assert counts.max() <= 10


@pytest.mark.parametrize("bad", [[0], [-1, 1], [-1, 0, 3, 1], [-1, -1], list(range(-1, 64))])
def test_tree_validate_rejects(bad):
    with pytest.raises(ValueError):
        tree.validate(bad)


# ----------------------------------------------------------------------------- compaction
def test_compaction_equals_sequential_append():
    r = np.random.default_rng(6)
    layers, B, Hkv, S_max, D, N, width = 3, 4, 2, 40, 8, 12, 7
    kc = r.standard_normal((layers, B, Hkv, S_max, D)).astype(np.float32)
    vc = r.standard_normal((layers, B, Hkv, S_max, D)).astype(np.float32)
    tk = r.standard_normal((layers, B, N, Hkv, D)).astype(np.float32)
    tv = r.standard_normal((layers, B, N, Hkv, D)).astype(np.float32)
    aux = r.standard_normal((B, N, 6)).astype(np.float32)
    L = np.array([0, 5, 20, 33])
    paths, alen = np.full((B, width), -1), np.zeros(B, int)
    for b in range(B):
        parents = synth.random_tree(r, N, max_depth=6, max_children=3)
        leaf = int(r.integers(0, N))
        p = tree.path_to(parents, leaf)[: S_max - L[b]]
        paths[b, : len(p)] = p
        alen[b] = len(p) - 1
    k2, v2, slot, newL, aux_out = compact.compact_kv(kc, vc, tk, tv, paths, alen, L, width, aux)
    for b in range(B):
        # sequential append: one position at a time, like a cache.update per accepted token
        ks = [kc[:, b, :, j] for j in range(L[b])]
        for j in range(alen[b] + 1):
            ks.append(tk[:, b, paths[b, j]])
        seq = np.stack(ks, 2) if ks else None
        assert (k2[:, b, :, : L[b] + alen[b] + 1] == seq).all()
        assert (k2[:, b, :, L[b] + alen[b] + 1:] == kc[:, b, :, L[b] + alen[b] + 1:]).all()
        assert newL[b] == L[b] + alen[b] + 1
        assert slot[b, : alen[b] + 1].tolist() == list(range(L[b], L[b] + alen[b] + 1))
        assert (slot[b, alen[b] + 1:] == -1).all()
        assert (aux_out[b, : alen[b] + 1] == aux[b, paths[b, : alen[b] + 1]]).all()
        assert (v2[:, b, :, L[b]: L[b] + alen[b] + 1] == np.moveaxis(tv[:, b, paths[b, : alen[b] + 1]], 1, 2)).all()


@pytest.mark.parametrize("branching,n_draft", [([2, 2, 1, 1], 14), ([3, 3, 2], 30)])
def test_static_tree_node_counts(branching, n_draft):
    """"Advanced speculative decoding: tree drafts and EAGLE", "Exercises", exercise 1 and its
    answer: 2 + 4 + 4 + 4 = 14 and 3 + 9 + 18 = 30 draft nodes besides the root."""
    parents = tree.static_tree(branching)
    tree.validate(parents)
    assert len(parents) - 1 == n_draft
    d = tree.depths(parents)
    width = 1
    for t, b in enumerate(branching, start=1):
        width *= b
        assert int((d == t).sum()) == width
        assert all(int((parents[d == t] == p).sum()) == b for p in np.flatnonzero(d == t - 1))


def test_spec_decode_metadata_worked_example(golden_dir):
    from oracle import ragged
    fields = {}
    for line in open(os.path.join(golden_dir, "spec_decode_metadata_5req.txt")):
        if line.startswith("#") or not line.strip():
            continue
        k, v = line.split(":")
        fields[k.strip()] = [int(x) for x in v.split()]
    got = ragged.spec_decode_metadata(fields["cu_num_scheduled_tokens"], fields["num_draft_tokens"])
    for k in ("cu_num_draft_tokens", "logits_indices", "target_logits_indices", "bonus_logits_indices"):
        assert got[k].tolist() == fields[k], k


def test_spec_decode_metadata_invariants():
    from oracle import ragged
    r = np.random.default_rng(5)
    d = r.integers(0, 8, 40)
    sched = d + 1 + r.integers(0, 50, 40)
    got = ragged.spec_decode_metadata(np.cumsum(sched), d)
    n_rows = int((d + 1).sum())
    assert len(got["logits_indices"]) == n_rows
    rows = np.sort(np.concatenate([got["target_logits_indices"], got["bonus_logits_indices"]]))
    assert rows.tolist() == list(range(n_rows))          # every logits row is a target or a bonus row
    assert (np.diff(got["logits_indices"]) > 0).all()
    with pytest.raises(ValueError):
        ragged.spec_decode_metadata([2, 3], [2, 0])       # 2 scheduled tokens cannot carry 2 drafts + 1


# ----------------------------------------------------------------------------- paged cache addressing
def test_slot_mapping_invariants():
    from oracle import ragged
    r = np.random.default_rng(12)
    bs, n_pages, B, blocks = 64, 97, 5, 7
    pages = r.permutation(n_pages)[: B * blocks].reshape(B, blocks)      # disjoint pages per sequence
    seen = set()
    for b in range(B):
        L = int(r.integers(1, blocks * bs + 1))
        slots = ragged.slot_mapping(pages[b], bs, np.arange(L))
        # every position lands in one of the sequence's own pages, at its offset within the page
        assert np.isin(slots // bs, pages[b]).all()
        assert (slots % bs == np.arange(L) % bs).all()
        # consecutive positions of a page are consecutive slots; a new page starts at a page boundary
        for p in range(1, L):
            if p % bs:
                assert slots[p] == slots[p - 1] + 1
            else:
                assert slots[p] % bs == 0
        # distinct positions never share a slot, within or across sequences
        assert len(set(slots.tolist()) & seen) == 0 and len(set(slots.tolist())) == L
        seen |= set(slots.tolist())
        # a pool written position by position reads back as the contiguous cache
        cache = r.standard_normal((L, 3))
        pool = np.zeros((n_pages * bs, 3))
        for p in range(L):
            pool[ragged.slot_mapping(pages[b], bs, [p])[0]] = cache[p]
        assert np.array_equal(ragged.paged_view(pool, pages[b], bs, L), cache)
