"""fp64 CPU oracle for exact attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg (and its ``--impl reference`` arm) may import this package.  The CUDA
library never calls it and shares no code with it.

``attn_oracle.c`` holds the arithmetic (plain definition, fp64, OpenMP) of
softmax attention, of Stieltjes attention and of Nystrom attention;
this module compiles it with gcc and calls it through ctypes.  Inputs may be
any array-likes of bf16-representable values: they are widened to fp64
exactly before the call.  Every function here follows the definitions cited
in ``attn_oracle.c``.
"""
import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force=False):
    """Compile attn_oracle.c into oracle/_build/liboracle.so (gcc, OpenMP)."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + ".tmp%d" % os.getpid()
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
           _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def bind(lib):
    """Sets the ctypes signatures of a loaded oracle library; returns it."""
    d = ctypes.POINTER(ctypes.c_double)
    i = ctypes.c_int
    lib.oracle_fwd_rows.argtypes = [d, d, d, i, i, i, i, i, i, ctypes.c_double,
                                    ctypes.POINTER(ctypes.c_int64), ctypes.c_int64, d, d]
    lib.oracle_fwd_rows.restype = i
    lib.oracle_bwd.argtypes = [d, d, d, d, i, i, i, i, i, i, ctypes.c_double, d, d, d]
    lib.oracle_bwd.restype = i
    lib.oracle_bwd_dq_rows.argtypes = [d, d, d, d, i, i, i, i, i, i, ctypes.c_double,
                                       ctypes.POINTER(ctypes.c_int64), ctypes.c_int64, d]
    lib.oracle_bwd_dq_rows.restype = i
    lib.oracle_stj_fwd_rows.argtypes = [d, d, d, i, i, i, i, i, i, ctypes.c_double, i, i,
                                        ctypes.POINTER(ctypes.c_int64), ctypes.c_int64, d, d]
    lib.oracle_stj_fwd_rows.restype = i
    lib.oracle_ns_pinv.argtypes = [d, i, i, ctypes.c_double, d]
    lib.oracle_ns_pinv.restype = i
    lib.oracle_nys_fwd.argtypes = [d, d, d, i, i, i, i, i, i, i, ctypes.c_double,
                                   ctypes.c_double, d, d, d, d, d]
    lib.oracle_nys_fwd.restype = i
    lib.oracle_num_threads.restype = i
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = bind(ctypes.CDLL(build()))
    return _lib


def _f64(x):
    """Exact widening of any float tensor/array to a C-contiguous fp64 array."""
    if hasattr(x, "detach"):  # torch tensor (CPU); bf16 -> fp32 -> fp64 is exact
        x = x.detach().to("cpu").float().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def num_threads():
    """OpenMP threads the oracle runs with (OMP_NUM_THREADS or all cores)."""
    return _load().oracle_num_threads()


def fwd_rows(q, k, v, causal, scale, rows=None):
    """O and LSE for selected rows.

    q: [B,Hq,N,D]; k, v: [B,Hkv,N,D].  rows: flat ids (b*Hq + h)*N + i, or
    None for all rows.  Returns (o [len(rows), D], lse [len(rows)]) in fp64.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, Hq, N, D = q.shape
    Hkv = k.shape[1]
    if rows is None:
        nrows = B * Hq * N
        rptr = None
    else:
        rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        nrows = rows.size
        rptr = rows.ctypes.data_as(ctypes.POINTER(ctypes.c_int64))
    o = np.empty((nrows, D), dtype=np.float64)
    lse = np.empty((nrows,), dtype=np.float64)
    rc = _load().oracle_fwd_rows(_ptr(q), _ptr(k), _ptr(v), B, Hq, Hkv, N, D,
                                 int(bool(causal)), float(scale), rptr, nrows,
                                 _ptr(o), _ptr(lse))
    if rc != 0:
        raise ValueError("oracle_fwd_rows rejected its arguments")
    return o, lse


def fwd(q, k, v, causal, scale):
    """Full forward: returns (o [B,Hq,N,D], lse [B,Hq,N]) in fp64."""
    B, Hq, N, D = tuple(q.shape)
    o, lse = fwd_rows(q, k, v, causal, scale)
    return o.reshape(B, Hq, N, D), lse.reshape(B, Hq, N)


def bwd(q, k, v, do, causal, scale):
    """Gradients of sum(dO * O): returns (dq, dk, dv) in fp64."""
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    B, Hq, N, D = q.shape
    Hkv = k.shape[1]
    dq = np.empty_like(q)
    dk = np.empty_like(k)
    dv = np.empty_like(v)
    rc = _load().oracle_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(do), B, Hq, Hkv, N, D,
                            int(bool(causal)), float(scale), _ptr(dq), _ptr(dk), _ptr(dv))
    if rc != 0:
        raise ValueError("oracle_bwd rejected its arguments")
    return dq, dk, dv


def bwd_dq_rows(q, k, v, do, causal, scale, rows):
    """dQ of selected rows (flat ids (b*Hq + h)*N + i), each from its own row
    of scores: the dQ of ``bwd`` without the N x N work of the whole backward.
    Returns dq [len(rows), D] in fp64."""
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    B, Hq, N, D = q.shape
    Hkv = k.shape[1]
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    dq = np.empty((rows.size, D), dtype=np.float64)
    rc = _load().oracle_bwd_dq_rows(_ptr(q), _ptr(k), _ptr(v), _ptr(do), B, Hq, Hkv, N, D,
                                    int(bool(causal)), float(scale),
                                    rows.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
                                    rows.size, _ptr(dq))
    if rc != 0:
        raise ValueError("oracle_bwd_dq_rows rejected its arguments")
    return dq


def stj_fwd_rows(q, k, v, causal, scale, order, steps, rows=None):
    """Stieltjes attention for selected rows: (o [len(rows), D], pole [len(rows)]).

    The pole is returned in score units (row max + Newton's lambda); steps <= 0
    solves for the exact pole instead of running `steps` Newton steps."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, Hq, N, D = q.shape
    Hkv = k.shape[1]
    if rows is None:
        nrows = B * Hq * N
        rptr = None
    else:
        rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        nrows = rows.size
        rptr = rows.ctypes.data_as(ctypes.POINTER(ctypes.c_int64))
    o = np.empty((nrows, D), dtype=np.float64)
    pole = np.empty((nrows,), dtype=np.float64)
    rc = _load().oracle_stj_fwd_rows(_ptr(q), _ptr(k), _ptr(v), B, Hq, Hkv, N, D,
                                     int(bool(causal)), float(scale), int(order), int(steps),
                                     rptr, nrows, _ptr(o), _ptr(pole))
    if rc != 0:
        raise ValueError("oracle_stj_fwd_rows rejected its arguments")
    return o, pole


def stj_fwd(q, k, v, causal, scale, order, steps):
    """Full Stieltjes forward: (o [B,Hq,N,D], pole [B,Hq,N]) in fp64."""
    B, Hq, N, D = tuple(q.shape)
    o, pole = stj_fwd_rows(q, k, v, causal, scale, order, steps)
    return o.reshape(B, Hq, N, D), pole.reshape(B, Hq, N)


def ns_pinv(a, iters, kappa):
    """Newton-Schulz pseudo-inverse of a square matrix after `iters` steps
    (Tikhonov ridge when kappa > 0), as the Nystrom forward takes it."""
    a = _f64(a)
    m = a.shape[0]
    if a.shape != (m, m):
        raise ValueError("ns_pinv wants a square matrix")
    out = np.empty((m, m), dtype=np.float64)
    if _load().oracle_ns_pinv(_ptr(a), m, int(iters), float(kappa), _ptr(out)) != 0:
        raise ValueError("oracle_ns_pinv rejected its arguments")
    return out


def nys_fwd(q, k, v, m, iters, kappa, scale, intermediates=False):
    """Nystrom attention forward: o [B,Hq,N,D] in fp64.

    With intermediates=True returns (o, dict(qt, kt, pinv, w)): the landmarks
    Qt [B,Hq,m,D] and Kt [B,Hkv,m,D], the pseudo-inverse of the landmark
    softmax [B,Hq,m,m] and W = softmax(scale Qt K^T) V [B,Hq,m,D]."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, Hq, N, D = q.shape
    Hkv = k.shape[1]
    o = np.empty_like(q)
    qt = np.empty((B, Hq, m, D)) if intermediates else None
    kt = np.empty((B, Hkv, m, D)) if intermediates else None
    pinv = np.empty((B, Hq, m, m)) if intermediates else None
    w = np.empty((B, Hq, m, D)) if intermediates else None
    opt = lambda a: _ptr(a) if a is not None else None
    rc = _load().oracle_nys_fwd(_ptr(q), _ptr(k), _ptr(v), B, Hq, Hkv, N, D, int(m),
                                int(iters), float(kappa), float(scale), _ptr(o),
                                opt(qt), opt(kt), opt(pinv), opt(w))
    if rc != 0:
        raise ValueError("oracle_nys_fwd rejected its arguments")
    if intermediates:
        return o, dict(qt=qt, kt=kt, pinv=pinv, w=w)
    return o
