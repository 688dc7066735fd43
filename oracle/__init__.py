"""fp64 CPU oracle for the diagonal metaplastic scan and the Moebius scan.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package.  The CUDA library and its Python binding never import it, and it
imports nothing from them.

The arithmetic lives in ``kdn_oracle.c`` (plain token-by-token loops in fp64;
see the header there for the equations and the page passages they follow).
This module compiles it with gcc, loads it with ctypes and converts arrays.
``diag_scan_py`` / ``mobius_scan_py`` are the same definitions written as pure
Python loops, for tiny inputs only.  Both transcriptions are pinned by the same
closed forms and invariants (``tests/oracle_pins.py``) and checked against each
other on the smallest scan workload (``tests/test_oracle_pins.py``).
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kdn_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False, src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile ``src`` into the shared library ``out`` (OpenMP if available).

    No fast-math: the oracle keeps IEEE fp64 semantics.
    """
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    os.makedirs(os.path.dirname(out), exist_ok=True)
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
            "-ffp-contract=off", src, "-o", out + ".tmp", "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       capture_output=True, text=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True, text=True)
    os.replace(out + ".tmp", out)
    return out


def load(path: str | None = None):
    """Load (building first if needed) and return the ctypes library."""
    global _lib
    if path is not None:
        return _declare(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            build()
            _lib = _declare(ctypes.CDLL(_LIB_PATH))
    return _lib


def _declare(lib):
    dp = ctypes.POINTER(ctypes.c_double)
    L = ctypes.c_long
    lib.oracle_diag_scan.restype = ctypes.c_int
    lib.oracle_diag_scan.argtypes = [dp, dp, dp, dp, dp, dp, ctypes.c_double, dp, dp,
                                     dp, dp, dp, L, L, L, L, L]
    lib.oracle_mobius_scan.restype = ctypes.c_int
    lib.oracle_mobius_scan.argtypes = [dp, dp, dp, dp, dp, dp, L, L]
    lib.oracle_diag_scan_bwd.restype = ctypes.c_int
    lib.oracle_diag_scan_bwd.argtypes = [dp, dp, dp, dp, dp, dp, ctypes.c_double, dp, dp,
                                         dp, dp, dp, dp, dp, dp, dp, dp, dp, dp, dp,
                                         L, L, L, L, L]
    lib.oracle_lin_scan.restype = ctypes.c_int
    lib.oracle_lin_scan.argtypes = [dp, dp, dp, dp, dp, dp, ctypes.c_double, dp, dp, dp,
                                    L, L, L, L, L]
    lib.oracle_max_threads.restype = ctypes.c_int
    lib.oracle_set_threads.argtypes = [ctypes.c_int]
    return lib


def _f64(x):
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor: upcast the exact stored values
        x = x.detach().cpu().double().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def max_threads() -> int:
    return int(load().oracle_max_threads())


def set_threads(n: int) -> None:
    load().oracle_set_threads(int(n))


def diag_scan(q, k, v, beta, d, A, I_prior, I0=None, mu0=None, lib=None):
    """Oracle of the diagonal metaplastic scan.

    Shapes: q, k [B,H,T,dk]; v, beta [B,H,T,dv]; d [B,H,T]; A [H];
    I0, mu0 [B,H,dv,dk] or None.  Returns (out [B,H,T,dv], mu_T, I_T) as
    fp64 numpy arrays.
    """
    lib = lib or load()
    q, k, v, beta, d, A = (_f64(x) for x in (q, k, v, beta, d, A))
    I0, mu0 = _f64(I0), _f64(mu0)
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    assert k.shape == (B, H, T, dk) and beta.shape == v.shape == (B, H, T, dv)
    assert d.shape == (B, H, T) and A.shape == (H,)
    if I0 is not None:
        assert I0.shape == (B, H, dv, dk)
    if mu0 is not None:
        assert mu0.shape == (B, H, dv, dk)
    out = np.empty((B, H, T, dv))
    mu_T = np.empty((B, H, dv, dk))
    I_T = np.empty((B, H, dv, dk))
    rc = lib.oracle_diag_scan(_ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(d), _ptr(A),
                              float(I_prior), _ptr(I0), _ptr(mu0), _ptr(out), _ptr(mu_T),
                              _ptr(I_T), B, H, T, dk, dv)
    if rc != 0:
        raise RuntimeError(f"oracle_diag_scan failed ({rc})")
    return out, mu_T, I_T


def lin_scan(q, k, v, beta, d, A, I_prior, mu0=None, lib=None):
    """Oracle of the non-metaplastic limit (importance held at I_prior).

    Shapes as ``diag_scan``; mu0 [B,H,dv,dk] or None.  Returns (out
    [B,H,T,dv], mu_T [B,H,dv,dk]) as fp64 numpy arrays.
    """
    lib = lib or load()
    q, k, v, beta, d, A = (_f64(x) for x in (q, k, v, beta, d, A))
    mu0 = _f64(mu0)
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    assert k.shape == (B, H, T, dk) and beta.shape == v.shape == (B, H, T, dv)
    assert d.shape == (B, H, T) and A.shape == (H,)
    assert mu0 is None or mu0.shape == (B, H, dv, dk)
    out = np.empty((B, H, T, dv))
    mu_T = np.empty((B, H, dv, dk))
    rc = lib.oracle_lin_scan(_ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(d), _ptr(A),
                             float(I_prior), _ptr(mu0), _ptr(out), _ptr(mu_T), B, H, T, dk, dv)
    if rc != 0:
        raise RuntimeError(f"oracle_lin_scan failed ({rc})")
    return out, mu_T


def diag_scan_bwd(q, k, v, beta, d, A, I_prior, I0=None, mu0=None, dout=None,
                  dmu_T=None, dI_T=None, lib=None):
    """Oracle of the backward pass: reverse-mode derivative of ``diag_scan``
    for L = sum(dout * out) + sum(dmu_T * mu_T) + sum(dI_T * I_T).

    ``dout`` [B,H,T,dv] is required; ``dmu_T``, ``dI_T`` [B,H,dv,dk] may be
    None (zero).  Returns a dict of fp64 arrays: dq, dk [B,H,T,dk]; dv, dbeta
    [B,H,T,dv]; dd [B,H,T]; dA [H] (summed over the batch); dI0, dmu0
    [B,H,dv,dk].  Keeps every state of a head: (T+1)*dv*dk*16 bytes per head
    being processed.
    """
    lib = lib or load()
    q, k, v, beta, d, A = (_f64(x) for x in (q, k, v, beta, d, A))
    I0, mu0, dout, dmu_T, dI_T = (_f64(x) for x in (I0, mu0, dout, dmu_T, dI_T))
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    assert dout is not None and dout.shape == (B, H, T, dv)
    for x in (I0, mu0, dmu_T, dI_T):
        assert x is None or x.shape == (B, H, dv, dk)
    g = dict(dq=np.empty((B, H, T, dk)), dk=np.empty((B, H, T, dk)), dv=np.empty((B, H, T, dv)),
             dbeta=np.empty((B, H, T, dv)), dd=np.empty((B, H, T)), dA_bh=np.empty((B, H)),
             dI0=np.empty((B, H, dv, dk)), dmu0=np.empty((B, H, dv, dk)))
    rc = lib.oracle_diag_scan_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(d), _ptr(A),
                                  float(I_prior), _ptr(I0), _ptr(mu0), _ptr(dout), _ptr(dmu_T),
                                  _ptr(dI_T), _ptr(g["dq"]), _ptr(g["dk"]), _ptr(g["dv"]),
                                  _ptr(g["dbeta"]), _ptr(g["dd"]), _ptr(g["dA_bh"]),
                                  _ptr(g["dI0"]), _ptr(g["dmu0"]), B, H, T, dk, dv)
    if rc != 0:
        raise RuntimeError(f"oracle_diag_scan_bwd failed ({rc})")
    g["dA"] = g.pop("dA_bh").sum(axis=0)
    return g


def mobius_scan(a, b, c, d, lambda0, lib=None):
    """Oracle of the Moebius precision recursion: a,b,c,d [N,T], lambda0 [N]
    -> lambda_1..lambda_T as [N,T] fp64."""
    lib = lib or load()
    a, b, c, d, lambda0 = (_f64(x) for x in (a, b, c, d, lambda0))
    N, T = a.shape
    assert b.shape == c.shape == d.shape == (N, T) and lambda0.shape == (N,)
    out = np.empty((N, T))
    rc = lib.oracle_mobius_scan(_ptr(a), _ptr(b), _ptr(c), _ptr(d), _ptr(lambda0),
                                _ptr(out), N, T)
    if rc != 0:
        raise RuntimeError(f"oracle_mobius_scan failed ({rc})")
    return out


def diag_scan_py(q, k, v, beta, d, A, I_prior, I0=None, mu0=None):
    """The diagonal update as pure Python loops (tiny inputs only)."""
    q, k, v, beta, d, A = (_f64(x).tolist() for x in (q, k, v, beta, d, A))
    B, H, T, dk = len(q), len(q[0]), len(q[0][0]), len(q[0][0][0])
    dv = len(v[0][0][0])
    I0 = _f64(I0).tolist() if I0 is not None else None
    mu0 = _f64(mu0).tolist() if mu0 is not None else None
    out = [[[[0.0] * dv for _ in range(T)] for _ in range(H)] for _ in range(B)]
    muT = [[None] * H for _ in range(B)]
    IT = [[None] * H for _ in range(B)]
    for b_ in range(B):
        for h in range(H):
            I = [[I0[b_][h][i][j] if I0 else I_prior for j in range(dk)] for i in range(dv)]
            mu = [[mu0[b_][h][i][j] if mu0 else 0.0 for j in range(dk)] for i in range(dv)]
            for t in range(T):
                alpha = math.exp(-A[h] * d[b_][h][t])
                kt, vt, bt, qt = k[b_][h][t], v[b_][h][t], beta[b_][h][t], q[b_][h][t]
                for i in range(dv):
                    for j in range(dk):
                        In = alpha * I[i][j] + (1 - alpha) * I_prior + bt[i] * kt[j] ** 2
                        mu[i][j] = alpha * I[i][j] / In * mu[i][j] + bt[i] * vt[i] * kt[j] / In
                        I[i][j] = In
                for i in range(dv):
                    out[b_][h][t][i] = sum(mu[i][j] * qt[j] for j in range(dk))
            muT[b_][h], IT[b_][h] = mu, I
    return np.array(out), np.array(muT), np.array(IT)


def mobius_scan_py(a, b, c, d, lambda0):
    """The Moebius recursion as pure Python loops (tiny inputs only)."""
    a, b, c, d, lambda0 = (_f64(x).tolist() for x in (a, b, c, d, lambda0))
    out = []
    for n in range(len(a)):
        lam, row = lambda0[n], []
        for t in range(len(a[n])):
            lam = (a[n][t] * lam + b[n][t]) / (c[n][t] * lam + d[n][t])
            row.append(lam)
        out.append(row)
    return np.array(out)
