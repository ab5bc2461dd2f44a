"""Pins for the Stieltjes attention oracle (no GPU).

FlashStieltjes page: weights p_j = (lambda - s_j)^-q with the pole lambda placed
so that they add up to 1 ("Why touch softmax"), found by Newton-Raphson from 1.1
after subtracting the row max ("The challenge").  Pinned here by the page's
printed weight table, an independent root finder, closed forms and the
pure-Python brute force.
"""
import math
import os

import numpy as np
import pytest

import oracle
from oracle.brute import brute_stj_fwd

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand(shape, seed, lo=-1.0, hi=1.0):
    return np.random.default_rng(seed).uniform(lo, hi, size=shape)


def _gap_example():
    """64 keys, scores 0, -0.25, ..., -15.75 against one query; V = identity so
    O's row is the weight row (the page's figure)."""
    N = D = 64
    q = np.zeros((1, 1, N, D))
    q[0, 0, 0, 0] = 1.0
    k = np.zeros((1, 1, N, D))
    k[0, 0, :, 0] = -0.25 * np.arange(N)
    v = np.eye(N).reshape(1, 1, N, D)
    return q, k, v


def _bisect_pole(t, order):
    """Root of sum (l - t_j)^-q = 1 for l > 0 by bisection (independent of Newton)."""
    lo, hi = 1e-12, 1.0
    f = lambda l: math.fsum((l - x) ** (-order) for x in t) - 1.0
    while f(hi) > 0:
        hi *= 2.0
    for _ in range(200):
        mid = 0.5 * (lo + hi)
        if f(mid) > 0:
            lo = mid
        else:
            hi = mid
    return 0.5 * (lo + hi)


def test_printed_weight_table_q4():
    """The page's table (q = 4): each printed weight to half a unit of its last
    printed digit, with the kernel's default three Newton steps."""
    q, k, v = _gap_example()
    o, pole = oracle.stj_fwd_rows(q, k, v, False, 1.0, 4, 3, rows=[0])
    w = o[0]
    with open(os.path.join(GOLDEN, "stieltjes_gap_table.txt")) as f:
        rows = [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]
    assert len(rows) == 7
    for gap_s, printed in rows:
        j = int(round(float(gap_s) / 0.25))
        mant = printed.split("e")[0]
        digits = len(mant.split(".")[1]) if "." in mant else 0
        exp = int(printed.split("e")[1]) if "e" in printed else 0
        half_ulp = 0.5 * 10.0 ** (exp - digits)
        assert abs(w[j] - float(printed)) <= half_ulp, (gap_s, w[j], printed)


def test_newton_three_steps_reach_the_root_on_the_example():
    """"Single-precision accuracy in 2-3 steps for q <= 4" on the page's example:
    three steps from 1.1 land within 2e-6 of a bisection root, and solving to
    convergence lands on it."""
    q, k, v = _gap_example()
    t = [-0.25 * j for j in range(64)]
    for order in (2, 4):
        root = _bisect_pole(t, order)
        _, p3 = oracle.stj_fwd_rows(q, k, v, False, 1.0, order, 3, rows=[0])
        _, pc = oracle.stj_fwd_rows(q, k, v, False, 1.0, order, 0, rows=[0])
        assert abs(pc[0] - root) <= 1e-12, (order, pc[0], root)
        if order == 4:
            assert abs(p3[0] - root) <= 2e-6, (p3[0], root)


def test_weights_sum_to_one_at_convergence():
    B, Hq, Hkv, N, D = 1, 2, 1, 37, 8
    q, k = _rand((B, Hq, N, D), 1), _rand((B, Hkv, N, D), 2)
    ones = np.ones((B, Hkv, N, D))
    for causal in (False, True):
        for order in (2, 4):
            o, _ = oracle.stj_fwd(q, k, ones, causal, 0.7, order, 0)
            np.testing.assert_allclose(o, 1.0, rtol=0, atol=1e-12)


def test_single_key_and_uniform_scores():
    """One key: pole = s + 1 and O = v.  Equal scores (Q = 0): pole = n^(1/q)
    over the n allowed keys, O = their mean (the causal prefix mean)."""
    rng = np.random.default_rng(3)
    q1, k1, v1 = rng.normal(size=(1, 1, 1, 4)), rng.normal(size=(1, 1, 1, 4)), rng.normal(size=(1, 1, 1, 4))
    o, pole = oracle.stj_fwd(q1, k1, v1, False, 0.5, 4, 0)
    s = 0.5 * float((q1 * k1).sum())
    np.testing.assert_allclose(o, v1, rtol=0, atol=1e-12)
    assert abs(pole[0, 0, 0] - (s + 1.0)) <= 1e-12
    N, D = 50, 6
    q0 = np.zeros((1, 1, N, D))
    k0, v0 = rng.normal(size=(1, 1, N, D)), rng.normal(size=(1, 1, N, D))
    for order in (2, 4):
        o, pole = oracle.stj_fwd(q0, k0, v0, True, 0.3, order, 0)
        csum = np.cumsum(v0[0, 0], axis=0) / np.arange(1, N + 1)[:, None]
        np.testing.assert_allclose(o[0, 0], csum, rtol=0, atol=1e-12)
        np.testing.assert_allclose(pole[0, 0], np.arange(1, N + 1) ** (1.0 / order),
                                   rtol=0, atol=1e-12)


def test_dominant_key_power_law_tail():
    """A key 50 above the rest takes nearly all the weight, but the power law
    leaves each other key about 51^-q of it (softmax would leave e^-50)."""
    N, D = 20, 4
    q = np.zeros((1, 1, N, D))
    q[0, 0, :, 0] = 1.0
    k = np.zeros((1, 1, N, D))
    k[0, 0, 7, 0] = 50.0
    v = np.random.default_rng(5).normal(size=(1, 1, N, D))
    o, _ = oracle.stj_fwd(q, k, v, False, 1.0, 4, 0)
    w_other = 51.0 ** -4
    expect = v[0, 0, 7] * (1 - 19 * w_other) + w_other * (v[0, 0].sum(0) - v[0, 0, 7])
    np.testing.assert_allclose(o[0, 0, 0], expect, rtol=0, atol=1e-6)


@pytest.mark.parametrize("B,Hq,Hkv,N,D,causal,scale,order,steps", [
    (1, 2, 1, 5, 4, True, 0.5, 4, 3),
    (2, 2, 2, 7, 3, False, 0.37, 2, 3),
    (1, 4, 2, 6, 5, True, 1.3, 4, 5),
])
def test_stieltjes_matches_brute_force(B, Hq, Hkv, N, D, causal, scale, order, steps):
    q, k, v = _rand((B, Hq, N, D), 11), _rand((B, Hkv, N, D), 12), _rand((B, Hkv, N, D), 13)
    o, pole = oracle.stj_fwd(q, k, v, causal, scale, order, steps)
    bo, bpole = brute_stj_fwd(q.ravel().tolist(), k.ravel().tolist(), v.ravel().tolist(),
                              B, Hq, Hkv, N, D, causal, scale, order, steps)
    np.testing.assert_allclose(o.ravel(), bo, rtol=0, atol=1e-11)
    np.testing.assert_allclose(pole.ravel(), bpole, rtol=0, atol=1e-12)
