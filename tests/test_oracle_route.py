"""Pins for the oracle's router, top-k, combine weights and union (CPU only)."""
import itertools
from fractions import Fraction

import numpy as np
import scipy.special

import oracle


def _exact_logit(x_row, w_row, b=None):
    s = sum((Fraction(float(a)) * Fraction(float(c)) for a, c in zip(x_row, w_row)), Fraction(0))
    if b is not None:
        s += Fraction(float(b))
    return float(s)  # Fraction -> float rounds correctly


def test_logits_are_correctly_rounded_exact_sums():
    rng = np.random.default_rng(0)
    for trial in range(6):
        T, E, H = 3, 5, 64
        x = rng.standard_normal((T, H)).astype(np.float32).astype(np.float64)
        w = (rng.standard_normal((E, H)) * 0.02).astype(np.float32)
        if trial % 2:
            # adversarial cancellation: huge terms that cancel exactly
            x[:, 0] = 2.0 ** 60
            x[:, 1] = -(2.0 ** 60)
            w[:, 1] = w[:, 0]
        b = rng.standard_normal(E).astype(np.float32) if trial >= 3 else None
        l = oracle.router_logits(x, w, b)
        for t in range(T):
            for e in range(E):
                assert l[t, e] == _exact_logit(x[t], w[e], None if b is None else b[e])


def test_topk_brute_force():
    rng = np.random.default_rng(1)
    for (E, k) in ((16, 2), (10, 3), (7, 7)):
        logits = rng.standard_normal((20, E))
        idx = oracle.topk_select(logits, k)
        for t in range(20):
            best = max(itertools.combinations(range(E), k),
                       key=lambda s: sum(logits[t, list(s)]))
            assert set(idx[t].tolist()) == set(best)
            vals = logits[t, idx[t]]
            assert np.all(np.diff(vals) <= 0)


def test_topk_ties_go_to_lower_id():
    l = np.array([[1.0, 3.0, 3.0, 2.0],
                  [0.0, 0.0, 0.0, 0.0],
                  [5.0, 1.0, 5.0, 5.0]])
    idx = oracle.topk_select(l, 2)
    assert idx.tolist() == [[1, 2], [0, 1], [0, 2]]


def test_combine_weights_sum_to_one_and_renormalise_softmax():
    rng = np.random.default_rng(2)
    logits = rng.standard_normal((50, 16)) * 3
    idx = oracle.topk_select(logits, 4)
    w = oracle.combine_weights(logits, idx)
    assert np.all(np.abs(w.sum(axis=1) - 1.0) <= 4 * 2.0 ** -52)
    full = scipy.special.softmax(logits, axis=1)
    sel = np.take_along_axis(full, idx.astype(np.int64), axis=1)
    assert np.allclose(w, sel / sel.sum(axis=1, keepdims=True), rtol=1e-13, atol=0)
    # selection on logits or on softmax probabilities is the same
    assert np.array_equal(idx, oracle.topk_select(np.log(full), 4))


def test_route_zero_input():
    x = np.zeros((2, 32))
    w = np.ones((6, 32), dtype=np.float32)
    idx, wts, _ = oracle.route(x, w, None, 3)
    assert idx.tolist() == [[0, 1, 2], [0, 1, 2]]
    assert np.all(wts == 1.0 / 3)


def test_plan_brute_force():
    rng = np.random.default_rng(3)
    for (T, E, k) in ((1, 8, 2), (4, 16, 3), (13, 9, 4)):
        idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
        w = rng.random((T, k))
        p = oracle.plan_union(idx, w, E)
        assert p["counts"].sum() == T * k
        assert p["offsets"][0] == 0 and p["offsets"][-1] == T * k
        assert p["uniq"].tolist() == sorted(set(idx.ravel().tolist()))
        for e in range(E):
            lo, hi = p["offsets"][e], p["offsets"][e + 1]
            toks = [t for t in range(T) if e in idx[t].tolist()]
            assert p["perm_tok"][lo:hi].tolist() == toks
            for q in range(lo, hi):
                t, j = p["perm_tok"][q], p["perm_rank"][q]
                assert idx[t, j] == e and p["perm_w"][q] == w[t, j]
                assert p["inv"][t * k + j] == q
        assert sorted(p["inv"].tolist()) == list(range(T * k))


def test_union_reduction_arithmetic(golden_dir):
    # Nanite §5.3 prints 5,600 assignments -> 3,670 unique uses (34.5% removed);
    # the union size is the number of distinct experts, so the reduction is
    # 1 - |U| / (T*k).
    import os
    vals = {}
    for line in open(os.path.join(golden_dir, "page_numbers.txt")):
        if not line.startswith("#") and line.strip():
            a, b = line.split()[:2]
            vals[a] = float(b)
    red = 100 * (1 - vals["nanite_unique"] / vals["nanite_assignments"])
    assert round(red, 1) == vals["nanite_reduction_pct"]
    # a window where 5 positions pick the same 8 experts collapses to 8 uses
    idx = np.tile(np.arange(8, dtype=np.int32), (5, 1))
    p = oracle.plan_union(idx, np.ones((5, 8)), 256)
    assert len(p["uniq"]) == 8 and p["counts"][:8].tolist() == [5] * 8
