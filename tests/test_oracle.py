"""Pins for the fp64 CPU oracle (no GPU).

Each test pins the oracle to something other than itself: the pure-Python
brute force (a separate code path), the worked example printed on the
FlashStieltjes page, closed forms, invariants, finite differences and the
GQA -> MHA reduction.
"""
import math
import os

import numpy as np
import pytest

import oracle
from oracle.brute import brute_bwd, brute_fwd
from flash_exact_attention_gb300.synth import bf16_bits_to_f32, make_inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand(shape, seed, lo=-1.0, hi=1.0):
    return np.random.default_rng(seed).uniform(lo, hi, size=shape)


# ---------------------------------------------------------------- brute force
@pytest.mark.parametrize("B,Hq,Hkv,N,D,causal,scale", [
    (1, 2, 1, 5, 4, True, 0.5),
    (2, 2, 2, 7, 3, False, 0.37),
    (1, 4, 2, 6, 5, True, 1.3),
    (1, 1, 1, 1, 2, False, 0.7),
])
def test_fwd_matches_brute_force(B, Hq, Hkv, N, D, causal, scale):
    q = _rand((B, Hq, N, D), 1)
    k = _rand((B, Hkv, N, D), 2)
    v = _rand((B, Hkv, N, D), 3)
    o, lse = oracle.fwd(q, k, v, causal, scale)
    bo, blse = brute_fwd(q.ravel().tolist(), k.ravel().tolist(), v.ravel().tolist(),
                         B, Hq, Hkv, N, D, causal, scale)
    np.testing.assert_allclose(o.ravel(), bo, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse.ravel(), blse, rtol=0, atol=1e-12)


@pytest.mark.parametrize("B,Hq,Hkv,N,D,causal,scale", [
    (1, 2, 1, 5, 4, True, 0.5),
    (2, 2, 2, 6, 3, False, 0.37),
    (1, 4, 2, 4, 3, False, 1.1),
])
def test_bwd_matches_brute_force(B, Hq, Hkv, N, D, causal, scale):
    q = _rand((B, Hq, N, D), 4)
    k = _rand((B, Hkv, N, D), 5)
    v = _rand((B, Hkv, N, D), 6)
    do = _rand((B, Hq, N, D), 7)
    dq, dk, dv = oracle.bwd(q, k, v, do, causal, scale)
    bq, bk, bv = brute_bwd(q.ravel().tolist(), k.ravel().tolist(), v.ravel().tolist(),
                           do.ravel().tolist(), B, Hq, Hkv, N, D, causal, scale)
    np.testing.assert_allclose(dq.ravel(), bq, rtol=0, atol=1e-12)
    np.testing.assert_allclose(dk.ravel(), bk, rtol=0, atol=1e-12)
    np.testing.assert_allclose(dv.ravel(), bv, rtol=0, atol=1e-12)


@pytest.mark.parametrize("B,Hq,Hkv,N,D,causal,scale", [
    (1, 2, 1, 5, 4, True, 0.5),
    (2, 2, 2, 6, 3, False, 0.37),
    (1, 4, 2, 4, 3, True, 1.1),
])
def test_bwd_dq_rows_match_brute_force(B, Hq, Hkv, N, D, causal, scale):
    """The row-wise dQ (for problems too large for the whole backward) against
    the pure-Python brute force, every row and a shuffled subset."""
    q = _rand((B, Hq, N, D), 14)
    k = _rand((B, Hkv, N, D), 15)
    v = _rand((B, Hkv, N, D), 16)
    do = _rand((B, Hq, N, D), 17)
    bq, _, _ = brute_bwd(q.ravel().tolist(), k.ravel().tolist(), v.ravel().tolist(),
                         do.ravel().tolist(), B, Hq, Hkv, N, D, causal, scale)
    bq = np.asarray(bq).reshape(-1, D)
    rows = np.arange(B * Hq * N)
    np.testing.assert_allclose(oracle.bwd_dq_rows(q, k, v, do, causal, scale, rows), bq,
                               rtol=0, atol=1e-12)
    some = np.random.default_rng(0).permutation(rows)[: max(1, rows.size // 3)]
    np.testing.assert_allclose(oracle.bwd_dq_rows(q, k, v, do, causal, scale, some), bq[some],
                               rtol=0, atol=1e-12)
    with pytest.raises(ValueError):
        oracle.bwd_dq_rows(q, k, v, do, causal, scale, [B * Hq * N])


# --------------------------------------------------------- printed worked example
def _read_gap_table():
    rows = []
    with open(os.path.join(GOLDEN, "softmax_gap_table.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            gap, val = line.split()
            rows.append((float(gap), val))
    return rows


def _half_unit_of_last_digit(text):
    mant, _, exp = text.lower().partition("e")
    decimals = len(mant.split(".")[1]) if "." in mant else 0
    return 0.5 * 10.0 ** (-decimals) * 10.0 ** (int(exp) if exp else 0)


def test_printed_softmax_gap_table():
    """64 scores 0, -0.25, ..., -15.75 in one row; V one-hot so O row = P row."""
    N = D = 64
    q = np.zeros((1, 1, N, D))
    k = np.zeros((1, 1, N, D))
    v = np.eye(N).reshape(1, 1, N, D)
    q[0, 0, 0, 0] = 1.0
    k[0, 0, :, 0] = -0.25 * np.arange(N)   # exact in bf16 (<= 6 significant bits)
    o, lse = oracle.fwd(q, k, v, causal=False, scale=1.0)
    p = o[0, 0, 0]
    rows = _read_gap_table()
    assert len(rows) == 7
    for gap, text in rows:
        j = int(round(gap / 0.25))
        assert abs(p[j] - float(text)) <= _half_unit_of_last_digit(text), (gap, p[j], text)
    # The weights form a geometric series with ratio e^-0.25 over 64 terms.
    top = (1 - math.exp(-0.25)) / (1 - math.exp(-16.0))
    assert p[0] == pytest.approx(top, rel=1e-13)
    assert lse[0, 0, 0] == pytest.approx(-math.log(top), rel=1e-13)


# ------------------------------------------------------------------ closed forms
@pytest.mark.parametrize("causal", [False, True])
def test_zero_query_gives_mean_of_values(causal):
    B, Hq, Hkv, N, D = 1, 2, 1, 9, 4
    q = np.zeros((B, Hq, N, D))
    k = _rand((B, Hkv, N, D), 8)
    v = _rand((B, Hkv, N, D), 9)
    o, lse = oracle.fwd(q, k, v, causal, 0.9)
    for i in range(N):
        n = i + 1 if causal else N
        for h in range(Hq):
            np.testing.assert_allclose(o[0, h, i], v[0, 0, :n].mean(axis=0), atol=1e-14)
            assert lse[0, h, i] == pytest.approx(math.log(n), abs=1e-14)


def test_dominant_key_returns_its_value():
    N, D = 12, 4
    q = np.zeros((1, 1, N, D))
    k = _rand((1, 1, N, D), 10, -0.1, 0.1)
    v = _rand((1, 1, N, D), 11)
    q[..., 0] = 1.0
    star = 7
    k[0, 0, star, 0] = 100.0        # score >= ~99 above every other key
    o, _ = oracle.fwd(q, k, v, False, 1.0)
    for i in range(N):
        np.testing.assert_allclose(o[0, 0, i], v[0, 0, star], atol=1e-12)


def test_probability_rows_sum_to_one_and_lse_identity():
    """V = identity makes O's rows the probability rows."""
    N = D = 16
    q = _rand((1, 1, N, D), 12, -2, 2)
    k = _rand((1, 1, N, D), 13, -2, 2)
    v = np.eye(N).reshape(1, 1, N, D)
    for causal in (False, True):
        o, lse = oracle.fwd(q, k, v, causal, 0.6)
        P = o[0, 0]
        np.testing.assert_allclose(P.sum(axis=1), 1.0, atol=1e-14)
        if causal:
            assert np.all(np.triu(P, 1) == 0.0)
        # each probability equals exp(s - LSE) for its own score, computed by hand
        for i in range(N):
            for j in range(i + 1 if causal else N):
                s = 0.6 * sum(q[0, 0, i, d] * k[0, 0, j, d] for d in range(D))
                assert P[i, j] == pytest.approx(math.exp(s - lse[0, 0, i]), rel=1e-12)


def test_shift_invariance():
    """A constant added to every score of a row leaves O unchanged, shifts LSE."""
    N, D = 10, 5
    q = _rand((1, 1, N, D), 14)
    k = _rand((1, 1, N, D), 15)
    v = _rand((1, 1, N, D), 16)
    k[..., D - 1] = 1.0              # every key has a constant last feature
    q2 = q.copy()
    shift = np.linspace(-3, 3, N)
    q2[0, 0, :, D - 1] += shift      # adds scale*shift_i to every score in row i
    for causal in (False, True):
        o1, l1 = oracle.fwd(q, k, v, causal, 0.8)
        o2, l2 = oracle.fwd(q2, k, v, causal, 0.8)
        np.testing.assert_allclose(o2, o1, atol=1e-13)
        np.testing.assert_allclose(l2[0, 0] - l1[0, 0], 0.8 * shift, atol=1e-13)


def test_single_key():
    q = _rand((2, 3, 1, 6), 17)
    k = _rand((2, 3, 1, 6), 18)
    v = _rand((2, 3, 1, 6), 19)
    for causal in (False, True):
        o, lse = oracle.fwd(q, k, v, causal, 0.4)
        np.testing.assert_allclose(o, v, atol=1e-15)
        np.testing.assert_allclose(lse, 0.4 * (q * k).sum(-1), atol=1e-15)


def test_selected_rows_match_full():
    d = make_inputs(2, 4, 2, 37, 8, seed=3)
    q, k, v = (bf16_bits_to_f32(d[n]) for n in ("q", "k", "v"))
    o, lse = oracle.fwd(q, k, v, True, 0.35)
    rows = np.array([0, 5, 36, 37, 100, 2 * 4 * 37 - 1])
    os_, ls_ = oracle.fwd_rows(q, k, v, True, 0.35, rows)
    np.testing.assert_array_equal(os_, o.reshape(-1, 8)[rows])
    np.testing.assert_array_equal(ls_, lse.reshape(-1)[rows])


def test_bad_rows_rejected():
    q = np.zeros((1, 1, 4, 2))
    with pytest.raises(ValueError):
        oracle.fwd_rows(q, q, q, False, 1.0, rows=[4])


# ------------------------------------------------------------------ GQA == MHA
def test_gqa_equals_mha_after_repeat_interleave():
    B, Hq, Hkv, N, D = 2, 6, 2, 11, 4
    G = Hq // Hkv
    q = _rand((B, Hq, N, D), 20)
    k = _rand((B, Hkv, N, D), 21)
    v = _rand((B, Hkv, N, D), 22)
    do = _rand((B, Hq, N, D), 23)
    kr, vr = np.repeat(k, G, axis=1), np.repeat(v, G, axis=1)
    for causal in (False, True):
        o1, l1 = oracle.fwd(q, k, v, causal, 0.5)
        o2, l2 = oracle.fwd(q, kr, vr, causal, 0.5)
        np.testing.assert_allclose(o1, o2, atol=1e-15)
        np.testing.assert_allclose(l1, l2, atol=1e-15)
        dq1, dk1, dv1 = oracle.bwd(q, k, v, do, causal, 0.5)
        dq2, dk2, dv2 = oracle.bwd(q, kr, vr, do, causal, 0.5)
        np.testing.assert_allclose(dq1, dq2, atol=1e-14)
        np.testing.assert_allclose(dk1, dk2.reshape(B, Hkv, G, N, D).sum(2), atol=1e-14)
        np.testing.assert_allclose(dv1, dv2.reshape(B, Hkv, G, N, D).sum(2), atol=1e-14)


# ------------------------------------------------------------------- backward
@pytest.mark.parametrize("causal", [False, True])
def test_bwd_central_finite_differences(causal):
    """dX of L = sum(dO * O) against central differences of the fp64 forward."""
    B, Hq, Hkv, N, D, scale = 1, 4, 2, 6, 3, 0.7
    q = _rand((B, Hq, N, D), 24)
    k = _rand((B, Hkv, N, D), 25)
    v = _rand((B, Hkv, N, D), 26)
    do = _rand((B, Hq, N, D), 27)
    dq, dk, dv = oracle.bwd(q, k, v, do, causal, scale)
    h = 1e-6

    def loss(q_, k_, v_):
        o, _ = oracle.fwd(q_, k_, v_, causal, scale)
        return float((o * do).sum())

    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        fd = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            args_p = {"q": q, "k": k, "v": v}
            args_m = dict(args_p)
            args_p[name], args_m[name] = xp, xm
            fd[idx] = (loss(**{a + "_": b for a, b in args_p.items()})
                       - loss(**{a + "_": b for a, b in args_m.items()})) / (2 * h)
        np.testing.assert_allclose(g, fd, atol=1e-8, rtol=1e-6, err_msg=name)


@pytest.mark.parametrize("causal", [False, True])
def test_bwd_invariants(causal):
    B, Hq, Hkv, N, D = 2, 4, 2, 13, 5
    G = Hq // Hkv
    q = _rand((B, Hq, N, D), 28)
    k = _rand((B, Hkv, N, D), 29)
    v = _rand((B, Hkv, N, D), 30)
    do = _rand((B, Hq, N, D), 31)
    dq, dk, dv = oracle.bwd(q, k, v, do, causal, 0.45)
    # sum_j dS_ij = 0 for every row, so dK sums to zero over keys
    np.testing.assert_allclose(dk.sum(axis=2), 0.0, atol=1e-13)
    # rows of P sum to one, so dV summed over keys is dO summed over rows and group
    np.testing.assert_allclose(dv.sum(axis=2),
                               do.reshape(B, Hkv, G, N, D).sum(axis=(2, 3)), atol=1e-12)
    # Q = 0 makes every score 0, so dK = scale * sum_i dS_ij q_i = 0
    _, dk0, _ = oracle.bwd(np.zeros_like(q), k, v, do, causal, 0.45)
    assert np.abs(dk0).max() == 0.0


def test_threads_reported():
    assert oracle.num_threads() >= 1
