"""Pins for the Nystrom attention oracle (no GPU).

FlashNystrom page, "Scope": O = softmax(Q Kt^T) pinv(softmax(Qt Kt^T))
softmax(Qt K^T) V with segment-mean landmarks and a Newton-Schulz
pseudo-inverse; "Configuration": the Tikhonov ridge (kappa*) and the number of
iterations.  Pinned here by results the mathematics fixes independently of the
oracle's code: the pseudo-inverse library routine, a closed form for diagonal
matrices, the squaring of the Newton-Schulz residual, exact attention when
every key is its own landmark, a constant V, one landmark, and the
pure-Python brute force.
"""
import numpy as np
import pytest

import oracle
from oracle.brute import brute_nys_fwd


def _rand(shape, seed, scale=1.0):
    return scale * np.random.default_rng(seed).standard_normal(shape)


def _stochastic(m, seed, temp=1.0):
    """A row-stochastic m x m matrix with positive entries (a softmax)."""
    s = _rand((m, m), seed, temp)
    e = np.exp(s - s.max(axis=1, keepdims=True))
    return e / e.sum(axis=1, keepdims=True)


@pytest.mark.parametrize("m", [1, 3, 8, 32])
def test_ns_converges_to_library_pinv(m):
    """Without the ridge, enough Newton-Schulz steps give numpy's pseudo-inverse."""
    a = _stochastic(m, m)
    got = oracle.ns_pinv(a, 80, 0.0)
    want = np.linalg.pinv(a)
    assert np.abs(got - want).max() <= 1e-8 * max(1.0, np.abs(want).max())


def test_ns_rank_deficient_converges_to_moore_penrose():
    """A singular matrix: the iteration from A^T/(|A|_1|A|_inf) reaches the
    Moore-Penrose inverse (not an inverse, which does not exist).  Round-off
    that lands in the null space doubles every step, so the step count is
    chosen where the range part has converged and that growth is still
    below 1e-12."""
    u, _ = np.linalg.qr(_rand((6, 3), 1))
    a = u @ np.diag([1.0, 1.5, 2.0]) @ u.T  # rank 3, symmetric
    got = oracle.ns_pinv(a, 14, 0.0)
    assert np.abs(got - np.linalg.pinv(a)).max() <= 1e-10


@pytest.mark.parametrize("kappa", [5.0, 1.0, 20.0])
def test_ridge_converges_to_regularised_solve(kappa):
    """With the ridge the result tends to (A^T A + lambda I)^-1 A^T,
    lambda = |A|_1 |A|_inf / kappa (max column sum times max row sum)."""
    a = _stochastic(16, 3, 2.0)
    lam = np.abs(a).sum(axis=0).max() * np.abs(a).sum(axis=1).max() / kappa
    want = np.linalg.solve(a.T @ a + lam * np.eye(16), a.T)
    got = oracle.ns_pinv(a, 200, kappa)
    assert np.abs(got - want).max() <= 1e-9


def test_ns_diagonal_closed_form():
    """For A = diag(a) the iteration acts entry by entry: with c = max|a|^2 the
    start is a/c, and 1 - a x_t = (1 - a^2/c)^(2^t), so
    x_t = (1 - (1 - a^2/c)^(2^t)) / a."""
    a = np.array([2.0, 0.5, 1.0, 0.1])
    c = a.max() ** 2
    for t in range(0, 7):
        got = oracle.ns_pinv(np.diag(a), t, 0.0)
        want = (1.0 - (1.0 - a * a / c) ** (2 ** t)) / a
        assert np.abs(np.diag(got) - want).max() <= 1e-13
        assert np.abs(got - np.diag(np.diag(got))).max() == 0.0


def test_ns_residual_squares():
    """Newton-Schulz squares the residual: I - A X_{t+1} = (I - A X_t)^2 for
    iterates started at a multiple of A^T (then A X_t is symmetric)."""
    a = _stochastic(12, 5)
    for t in range(0, 5):
        r0 = np.eye(12) - a @ oracle.ns_pinv(a, t, 0.0)
        r1 = np.eye(12) - a @ oracle.ns_pinv(a, t + 1, 0.0)
        assert np.abs(r1 - r0 @ r0).max() <= 1e-12


def test_ns_one_by_one_ridge_fixed_point():
    """1 x 1: A = a, M = a^2 + lambda with lambda = a^2 / kappa; the start
    M / M^2 = 1/M is already the inverse, so pinv = a / M for any step count."""
    a, kappa = 0.7, 4.0
    M = a * a * (1.0 + 1.0 / kappa)
    for t in (0, 1, 6):
        assert abs(oracle.ns_pinv(np.array([[a]]), t, kappa)[0, 0] - a / M) <= 1e-15


def test_landmarks_are_segment_means():
    """Landmark i is the mean of rows floor(iN/m) .. floor((i+1)N/m) - 1; m = N
    gives Q itself and m = 1 the mean of all rows."""
    B, H, N, D = 1, 2, 23, 5
    q, k, v = _rand((B, H, N, D), 1), _rand((B, H, N, D), 2), _rand((B, H, N, D), 3)
    for m in (1, 4, 7, 23):
        _, it = oracle.nys_fwd(q, k, v, m, 3, 5.0, 0.3, intermediates=True)
        for i in range(m):
            lo, hi = i * N // m, (i + 1) * N // m
            assert hi > lo
            np.testing.assert_allclose(it["qt"][0, :, i], q[0, :, lo:hi].mean(axis=1), atol=1e-14)
            np.testing.assert_allclose(it["kt"][0, :, i], k[0, :, lo:hi].mean(axis=1), atol=1e-14)
    _, it = oracle.nys_fwd(q, k, v, N, 3, 5.0, 0.3, intermediates=True)
    assert np.array_equal(it["qt"], q) and np.array_equal(it["kt"], k)


@pytest.mark.parametrize("causal_shape", [(1, 2, 2, 7, 6), (2, 4, 2, 5, 8)])
def test_every_key_a_landmark_is_exact_attention(causal_shape):
    """m = N, no ridge, converged pseudo-inverse: Qt = Q, Kt = K, so the middle
    factor inverts the first and the result is exact softmax attention (the
    softmax oracle, pinned separately)."""
    B, Hq, Hkv, N, D = causal_shape
    q, k, v = _rand((B, Hq, N, D), 4, 0.5), _rand((B, Hkv, N, D), 5, 0.5), _rand((B, Hkv, N, D), 6)
    scale = D ** -0.5
    got = oracle.nys_fwd(q, k, v, N, 100, 0.0, scale)
    want, _ = oracle.fwd(q, k, v, False, scale)
    assert np.abs(got - want).max() <= 1e-9


def test_constant_values_pass_through():
    """Every value row equal to u: softmax(Qt K^T) V = 1 u^T, and a converged
    inverse of the row-stochastic landmark softmax maps 1 to 1, so O = 1 u^T."""
    B, H, N, D, m = 1, 2, 40, 6, 5
    q, k = _rand((B, H, N, D), 7, 0.5), _rand((B, H, N, D), 8, 0.5)
    u = _rand((D,), 9)
    v = np.broadcast_to(u, (B, H, N, D)).copy()
    got = oracle.nys_fwd(q, k, v, m, 100, 0.0, 0.4)
    assert np.abs(got - u).max() <= 1e-9


def test_one_landmark_closed_form():
    """m = 1: the landmark softmaxes are 1 x 1 ones, so every output row is the
    attention of the mean query over all keys, times kappa / (kappa + 1) with
    the ridge (lambda = 1 / kappa for A = [1])."""
    B, H, N, D = 1, 3, 17, 4
    q, k, v = _rand((B, H, N, D), 10), _rand((B, H, N, D), 11), _rand((B, H, N, D), 12)
    scale = 0.6
    qbar = q.mean(axis=2)
    s = scale * np.einsum("bhd,bhnd->bhn", qbar, k)
    p = np.exp(s - s.max(axis=-1, keepdims=True))
    p /= p.sum(axis=-1, keepdims=True)
    att = np.einsum("bhn,bhnd->bhd", p, v)
    got0 = oracle.nys_fwd(q, k, v, 1, 6, 0.0, scale)
    assert np.abs(got0 - att[:, :, None, :]).max() <= 1e-13
    kappa = 5.0
    got = oracle.nys_fwd(q, k, v, 1, 6, kappa, scale)
    assert np.abs(got - kappa / (kappa + 1.0) * att[:, :, None, :]).max() <= 1e-13


@pytest.mark.parametrize("cfg", [
    (1, 1, 1, 6, 3, 3, 2, 0.0),
    (1, 2, 1, 7, 4, 3, 6, 5.0),
    (2, 2, 2, 5, 2, 5, 1, 2.0),
])
def test_matches_brute_force(cfg):
    """The C oracle and the pure-Python statement agree on tiny shapes
    (uneven segments, GQA, with and without the ridge)."""
    B, Hq, Hkv, N, D, m, iters, kappa = cfg
    q, k, v = _rand((B, Hq, N, D), 13), _rand((B, Hkv, N, D), 14), _rand((B, Hkv, N, D), 15)
    scale = 0.7
    got = oracle.nys_fwd(q, k, v, m, iters, kappa, scale)
    want = np.array(brute_nys_fwd(q.ravel().tolist(), k.ravel().tolist(), v.ravel().tolist(),
                                  B, Hq, Hkv, N, D, m, iters, kappa, scale)).reshape(got.shape)
    assert np.abs(got - want).max() <= 1e-11 * max(1.0, np.abs(want).max())


def test_gqa_equals_repeated_heads():
    """Hkv < Hq equals MHA on key/value heads repeated over each group."""
    B, Hq, Hkv, N, D, m = 1, 4, 2, 12, 4, 3
    q, k, v = _rand((B, Hq, N, D), 16), _rand((B, Hkv, N, D), 17), _rand((B, Hkv, N, D), 18)
    a = oracle.nys_fwd(q, k, v, m, 4, 5.0, 0.5)
    b = oracle.nys_fwd(q, np.repeat(k, 2, axis=1), np.repeat(v, 2, axis=1), m, 4, 5.0, 0.5)
    assert np.array_equal(a, b)


def test_rejects_bad_sizes():
    q = np.zeros((1, 1, 4, 2))
    with pytest.raises(ValueError):
        oracle.nys_fwd(q, q, q, 5, 3, 5.0, 1.0)  # N < m
    with pytest.raises(ValueError):
        oracle.nys_fwd(q, q, q, 2, -1, 5.0, 1.0)
