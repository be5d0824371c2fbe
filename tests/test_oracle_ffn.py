"""Pins for the oracle's SwiGLU expert FFN, shared expert and combine (CPU only).

The expected values come from closed forms: with permutation matrices as
weights, the FFN reduces to index shuffles and scalar silu values known in
closed form, so a transposed operand, a wrong index, a dropped term or a
swapped gate/up fails.
"""
import math

import numpy as np

import oracle


def test_silu_closed_forms():
    z = np.array([0.0, math.log(3.0), -math.log(3.0), 1000.0, -1000.0])
    s = oracle.silu(z)
    assert s[0] == 0.0
    assert math.isclose(s[1], 0.75 * math.log(3.0), rel_tol=1e-15)
    assert math.isclose(s[2], -0.25 * math.log(3.0), rel_tol=1e-15)
    assert s[3] == 1000.0 and s[4] == 0.0


def _perm(n, shift):
    P = np.zeros((n, n))
    for r in range(n):
        P[r, (r * 5 + shift) % n] = 1.0  # 5 is coprime with the sizes used
    return P


def _perm_expert(n, a, b, c, sg, su, sd):
    """gate = sg*P_a, up = su*P_b, down = sd*P_c (square, hidden == inter)."""
    return (sg * _perm(n, a), su * _perm(n, b), sd * _perm(n, c))


def test_expert_ffn_permutation_closed_form():
    n = 16
    rng = np.random.default_rng(0)
    x = rng.standard_normal((3, n))
    mats = _perm_expert(n, 1, 2, 3, 2.0, -0.5, 4.0)
    y = oracle.expert_ffn(mats, x)
    for t in range(3):
        for o in range(n):
            # y[o] = 4 * h[(5o+3)%n];  h[r] = silu(2 x[(5r+1)%n]) * (-0.5 x[(5r+2)%n])
            r = (5 * o + 3) % n
            g = 2.0 * x[t, (5 * r + 1) % n]
            u = -0.5 * x[t, (5 * r + 2) % n]
            want = 4.0 * (g / (1.0 + math.exp(-g))) * u
            assert math.isclose(y[t, o], want, rel_tol=1e-14, abs_tol=1e-300)


def test_expert_ffn_rectangular_orientation():
    # hidden 4, inter 2: Wg/Wu are [I, H], Wd is [H, I]
    wg = np.array([[1.0, 0, 0, 0], [0, 0, 1.0, 0]])
    wu = np.array([[0, 1.0, 0, 0], [0, 0, 0, 1.0]])
    wd = np.array([[1.0, 0], [0, 0], [0, 1.0], [2.0, 3.0]])
    x = np.array([[math.log(3.0), 2.0, 0.0, 5.0]])
    y = oracle.expert_ffn((wg, wu, wd), x)
    h0 = 0.75 * math.log(3.0) * 2.0
    h1 = 0.0
    assert np.allclose(y, [[h0, 0.0, h1, 2 * h0 + 3 * h1]], rtol=1e-15, atol=0)


def test_moe_layer_combine_and_shared():
    n = 8
    rng = np.random.default_rng(1)
    x = rng.standard_normal((3, n))
    experts = {e: _perm_expert(n, e, e + 1, e + 2, 1.0, 1.0, float(e + 1)) for e in range(4)}
    shared = _perm_expert(n, 7, 6, 5, 1.0, 2.0, 1.0)
    idx = np.array([[2, 0], [1, 3], [0, 2]])
    w = np.array([[0.25, 0.75], [0.5, 0.5], [1.0, 0.0]])
    y = oracle.moe_layer(x, idx, w, lambda e: experts[e], shared)
    for t in range(3):
        want = oracle.expert_ffn(shared, x[t:t + 1])[0]
        for j in range(2):
            want = want + w[t, j] * oracle.expert_ffn(experts[idx[t, j]], x[t:t + 1])[0]
        assert np.allclose(y[t], want, rtol=1e-14, atol=1e-14)
    # zero routed weights -> shared expert only; zero input -> zero output
    y0 = oracle.moe_layer(x, idx, np.zeros_like(w), lambda e: experts[e], shared)
    assert np.array_equal(y0, oracle.expert_ffn(shared, x))
    assert np.all(oracle.moe_layer(np.zeros((2, n)), idx[:2], w[:2], lambda e: experts[e], shared) == 0)


def test_moe_layer_from_quantised_payload():
    # a Q8_0 expert whose quants are permutation patterns with power-of-two
    # scales dequantises to c * P exactly, so the layer output is the closed form
    H = I = 32
    parts = []
    for m, (shift, code, dbits) in enumerate(((1, 1, 0x3C00), (2, 2, 0x3800), (3, 1, 0x4000))):
        q = np.zeros((32, 32), dtype=np.int8)
        for r in range(32):
            q[r, (5 * r + shift) % 32] = code
        parts.append(q.view(np.uint8).ravel())
        parts.append(np.full(32, dbits, dtype="<u2").view(np.uint8))
    p = np.concatenate(parts)
    mats = oracle.expert_matrices(p, H, I, oracle.Q8_0)
    assert np.array_equal(mats[0], _perm(32, 1)) and np.array_equal(mats[1], _perm(32, 2))
    assert np.array_equal(mats[2], 2.0 * _perm(32, 3))
    x = np.random.default_rng(2).standard_normal((1, 32))
    y = oracle.moe_layer(x, np.array([[0]]), np.array([[1.0]]), lambda e: mats, None)
    for o in range(32):
        r = (5 * o + 3) % 32
        g = x[0, (5 * r + 1) % 32]
        u = x[0, (5 * r + 2) % 32]
        assert math.isclose(y[0, o], 2.0 * g / (1 + math.exp(-g)) * u, rel_tol=1e-14, abs_tol=1e-300)
