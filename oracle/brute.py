"""Pure-Python brute-force attention for tiny inputs (test infrastructure only).

A second, independent statement of the same definitions as ``attn_oracle.c``,
written with Python floats and ``math.fsum`` so that it shares no code path,
compiler or summation order with the C oracle.  It exists to pin the C oracle
on shapes small enough for nested Python loops (N, D of a few dozen at most).

Definitions (FlashNystrom page, "Scope"; FlashAttention for Tesla P100 page,
"What it supports" and "Documentation"):
  s_ij = scale * q_i . k_j over allowed keys (j <= i when causal),
  P_i  = softmax(s_i), O_i = sum_j P_ij v_j, LSE_i = ln sum_j exp(s_ij),
  dS_ij = P_ij (dO_i . v_j - dO_i . O_i), dQ_i = scale sum_j dS_ij k_j,
  dK_j = scale sum_i dS_ij q_i, dV_j = sum_i P_ij dO_i  (summed over the
  query heads that share a key/value head).

Only tests/ may import this module.
"""
import math


def _idx(shape, b, h, n):
    _, H, N, D = shape
    return ((b * H + h) * N + n) * D


def _row(flat, shape, b, h, n):
    D = shape[3]
    o = _idx(shape, b, h, n)
    return flat[o:o + D]


def brute_fwd(q, k, v, B, Hq, Hkv, N, D, causal, scale):
    """q, k, v are flat Python lists of floats. Returns (o, lse) as lists."""
    G = Hq // Hkv
    qs, ks = (B, Hq, N, D), (B, Hkv, N, D)
    o = [0.0] * (B * Hq * N * D)
    lse = [0.0] * (B * Hq * N)
    for b in range(B):
        for h in range(Hq):
            hk = h // G
            for i in range(N):
                qi = _row(q, qs, b, h, i)
                keys = range(i + 1) if causal else range(N)
                s = [scale * math.fsum(a * c for a, c in zip(qi, _row(k, ks, b, hk, j)))
                     for j in keys]
                m = max(s)
                tot = math.fsum(math.exp(x - m) for x in s)
                ell = m + math.log(tot)
                p = [math.exp(x - ell) for x in s]
                lse[(b * Hq + h) * N + i] = ell
                base = _idx(qs, b, h, i)
                for d in range(D):
                    o[base + d] = math.fsum(p[t] * _row(v, ks, b, hk, j)[d]
                                            for t, j in enumerate(keys))
    return o, lse


def brute_bwd(q, k, v, do, B, Hq, Hkv, N, D, causal, scale):
    """Returns (dq, dk, dv) flat lists, from the chain rule written out."""
    G = Hq // Hkv
    qs, ks = (B, Hq, N, D), (B, Hkv, N, D)
    o, _ = brute_fwd(q, k, v, B, Hq, Hkv, N, D, causal, scale)
    dq = [0.0] * len(q)
    dk_terms = [[] for _ in range(len(k))]
    dv_terms = [[] for _ in range(len(v))]
    for b in range(B):
        for h in range(Hq):
            hk = h // G
            for i in range(N):
                qi = _row(q, qs, b, h, i)
                doi = _row(do, qs, b, h, i)
                oi = _row(o, qs, b, h, i)
                keys = list(range(i + 1) if causal else range(N))
                s = [scale * math.fsum(a * c for a, c in zip(qi, _row(k, ks, b, hk, j)))
                     for j in keys]
                m = max(s)
                tot = math.fsum(math.exp(x - m) for x in s)
                p = [math.exp(x - m) / tot for x in s]
                delta = math.fsum(a * c for a, c in zip(doi, oi))
                ds = []
                for t, j in enumerate(keys):
                    dp = math.fsum(a * c for a, c in zip(doi, _row(v, ks, b, hk, j)))
                    ds.append(p[t] * (dp - delta))
                qbase = _idx(qs, b, h, i)
                for d in range(D):
                    dq[qbase + d] = scale * math.fsum(
                        ds[t] * _row(k, ks, b, hk, j)[d] for t, j in enumerate(keys))
                for t, j in enumerate(keys):
                    kbase = _idx(ks, b, hk, j)
                    for d in range(D):
                        dk_terms[kbase + d].append(scale * ds[t] * qi[d])
                        dv_terms[kbase + d].append(p[t] * doi[d])
    dk = [math.fsum(t) for t in dk_terms]
    dv = [math.fsum(t) for t in dv_terms]
    return dq, dk, dv


def brute_stj_fwd(q, k, v, B, Hq, Hkv, N, D, causal, scale, order, steps):
    """Stieltjes attention (FlashStieltjes page, "Why touch softmax" and "The
    challenge"): per row, m = max score, Newton from 1.1 on
    sum (l - (s - m))^-q = 1 for `steps` steps, weights (m + l - s)^-q.
    Returns (o, pole) as flat lists; pole = m + l."""
    G = Hq // Hkv
    qs, ks = (B, Hq, N, D), (B, Hkv, N, D)
    o = [0.0] * (B * Hq * N * D)
    pole = [0.0] * (B * Hq * N)
    for b in range(B):
        for h in range(Hq):
            hk = h // G
            for i in range(N):
                qi = _row(q, qs, b, h, i)
                keys = range(i + 1) if causal else range(N)
                s = [scale * math.fsum(a * c for a, c in zip(qi, _row(k, ks, b, hk, j)))
                     for j in keys]
                m = max(s)
                lam = 1.1
                for _ in range(steps):
                    f = math.fsum((lam - (x - m)) ** (-order) for x in s) - 1.0
                    fp = -order * math.fsum((lam - (x - m)) ** (-order - 1) for x in s)
                    lam -= f / fp
                pole[(b * Hq + h) * N + i] = m + lam
                w = [(m + lam - x) ** (-order) for x in s]
                base = _idx(qs, b, h, i)
                for d in range(D):
                    o[base + d] = math.fsum(w[t] * _row(v, ks, b, hk, j)[d]
                                            for t, j in enumerate(keys))
    return o, pole


def _matmul(a, b):
    """Product of two matrices held as lists of rows (math.fsum per entry)."""
    cols = list(zip(*b))
    return [[math.fsum(x * y for x, y in zip(r, c)) for c in cols] for r in a]


def _softmax(row):
    mx = max(row)
    e = [math.exp(x - mx) for x in row]
    t = math.fsum(e)
    return [x / t for x in e]


def brute_nys_fwd(q, k, v, B, Hq, Hkv, N, D, m, iters, kappa, scale):
    """Nystrom attention (FlashNystrom page, "Scope" and "Configuration"):
    landmarks are the means of the m segments floor(iN/m)..floor((i+1)N/m)-1,
    O = softmax(s Q Kt^T) pinv(softmax(s Qt Kt^T)) softmax(s Qt K^T) V with
    pinv from `iters` Newton-Schulz steps X <- 2X - X A X started at
    A^T / (|A|_1 |A|_inf), on A^T A + lambda I (lambda = |A|_1 |A|_inf / kappa)
    followed by a product with A^T when kappa > 0.  Returns o as a flat list."""
    G = Hq // Hkv
    qs, ks = (B, Hq, N, D), (B, Hkv, N, D)
    o = [0.0] * (B * Hq * N * D)

    def pool(flat, shape, b, h):
        out = []
        for i in range(m):
            lo, hi = i * N // m, (i + 1) * N // m
            rows = [_row(flat, shape, b, h, r) for r in range(lo, hi)]
            out.append([math.fsum(r[d] for r in rows) / (hi - lo) for d in range(D)])
        return out

    def norms(a):
        n1 = max(math.fsum(abs(a[r][c]) for r in range(len(a))) for c in range(len(a)))
        ninf = max(math.fsum(abs(x) for x in r) for r in a)
        return n1 * ninf

    for b in range(B):
        for h in range(Hq):
            hk = h // G
            Q = [_row(q, qs, b, h, i) for i in range(N)]
            K = [_row(k, ks, b, hk, j) for j in range(N)]
            V = [_row(v, ks, b, hk, j) for j in range(N)]
            Qt, Kt = pool(q, qs, b, h), pool(k, ks, b, hk)
            scores = lambda X, Y: [[scale * math.fsum(a * c for a, c in zip(x, y)) for y in Y]
                                   for x in X]
            A1 = [_softmax(r) for r in scores(Q, Kt)]
            A2 = [_softmax(r) for r in scores(Qt, Kt)]
            A3 = [_softmax(r) for r in scores(Qt, K)]
            A2T = [list(c) for c in zip(*A2)]
            if kappa > 0:
                lam = norms(A2) / kappa
                M = _matmul(A2T, A2)
                for i in range(m):
                    M[i][i] += lam
            else:
                M = A2
            c0 = norms(M)
            X = [[x / c0 for x in c] for c in zip(*M)]
            for _ in range(iters):
                XAX = _matmul(X, _matmul(M, X))
                X = [[2.0 * x - y for x, y in zip(rx, ry)] for rx, ry in zip(X, XAX)]
            P = _matmul(X, A2T) if kappa > 0 else X
            Y = _matmul(P, _matmul(A3, V))
            Oh = _matmul(A1, Y)
            for i in range(N):
                base = _idx(qs, b, h, i)
                o[base:base + D] = Oh[i]
    return o
