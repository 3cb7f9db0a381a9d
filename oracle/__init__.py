"""fp64 CPU oracle for the batched KKT path -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product (``trajectory_optimization_kkt_gb300``)
never imports, loads or calls it, and the two share no code.

The arithmetic lives in ``gato_oracle.c`` (plain C, double precision), which
is compiled with gcc into ``oracle/_build/libgato_oracle.so`` on first use.
This module only marshals numpy arrays: fp32 workload data is upcast to fp64,
and every batch function loops over solves calling the C routines one solve
at a time.  See ``gato_oracle.c`` for the equations and the readings of the
GATO paper that each routine follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Dict, Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gato_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "libgato_oracle.so")
_lock = threading.Lock()
_lib = None

_D = ctypes.POINTER(ctypes.c_double)


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no-op when the library is up to date)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", _SRC,
                           "-o", tmp, "-lm"])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i, d = ctypes.c_int, ctypes.c_double
            pi = ctypes.POINTER(ctypes.c_int)
            lq = [i, i, i, _D, _D, _D, _D, _D, _D, _D, _D]
            lib.oracle_kkt_dense.argtypes = lq + [i, _D, _D, _D]
            lib.oracle_schur.argtypes = lq + [_D, _D, _D]
            lib.oracle_stair.argtypes = [i, i, _D, _D, _D, _D]
            lib.oracle_bt_dense.argtypes = [i, i, _D, _D, _D]
            lib.oracle_bt_dense.restype = None
            lib.oracle_pcg.argtypes = [i, i, _D, _D, _D, _D, _D, _D, d, i, i, _D, pi]
            lib.oracle_block_cholesky.argtypes = [i, i, _D, _D, _D, _D]
            lib.oracle_recover.argtypes = [i, i, i, _D, _D, _D, _D, _D, _D, _D, _D, _D]
            lib.oracle_merit.argtypes = lq + [_D, _D, d, d, _D, _D]
            lib.oracle_merit.restype = d
            lib.oracle_linesearch.argtypes = lq + [_D, _D, i, d, d, _D]
            lib.oracle_solve_kkt.argtypes = lq + [d, i, i, i, d, d, _D, _D, _D, pi, _D, pi]
            lib.oracle_sqp_linear.argtypes = lq + [i, d, d, d, d, i, d, d, _D, _D, _D, _D, pi, _D]
            _lib = lib
    return _lib


def _p(a: Optional[np.ndarray]):
    if a is None:
        return None
    assert a.dtype == np.float64 and a.flags.c_contiguous
    return a.ctypes.data_as(_D)


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float64)


_KEYS = ("Q", "R", "q", "r", "A", "B", "e", "s0")


def _one(prob: Dict[str, np.ndarray], j: Optional[int]):
    """fp64 copies of solve j's arrays (j=None: prob is already one solve)."""
    return [_f64(prob[k] if j is None else prob[k][j]) for k in _KEYS]


def _dims(prob, batched=True):
    Q, R = prob["Q"], prob["R"]
    off = 1 if batched else 0
    N, n = Q.shape[off], Q.shape[off + 1]
    m = R.shape[off + 1] if R.shape[off] > 0 else (prob["B"].shape[-1])
    return N, n, m


# ----------------------------------------------------------------------------
# single-solve routines (prob holds one solve: Q [N][n][n] ...)
# ----------------------------------------------------------------------------

def kkt_dense(prob, method: str = "ldlt"):
    """Dense KKT solve (eq. (2)); method 'ldlt' (no pivoting) or 'lu'."""
    L = _load()
    N, n, m = _dims(prob, batched=False)
    arr = _one(prob, None)
    dX, dU, lam = np.zeros((N, n)), np.zeros((max(N - 1, 0), m)), np.zeros((N, n))
    rc = L.oracle_kkt_dense(N, n, m, *[_p(a) for a in arr], 0 if method == "ldlt" else 1,
                            _p(dX), _p(dU), _p(lam))
    if rc:
        raise np.linalg.LinAlgError(f"dense KKT {method} failed ({rc})")
    return dX, dU, lam


def schur(prob):
    """S's blocks (D [N][n][n], O [N-1][n][n]) and gamma [N][n] (eqs. (4)-(6))."""
    L = _load()
    N, n, m = _dims(prob, batched=False)
    arr = _one(prob, None)
    D, O, g = np.zeros((N, n, n)), np.zeros((max(N - 1, 0), n, n)), np.zeros((N, n))
    rc = L.oracle_schur(N, n, m, *[_p(a) for a in arr], _p(D), _p(O), _p(g))
    return D, O, g, rc


def stair(D, O):
    """Phi^-1's blocks (Pd [N][n][n], Po [N-1][n][n]) from S's blocks."""
    L = _load()
    N, n = D.shape[0], D.shape[1]
    D, O = _f64(D), _f64(O)
    Pd, Po = np.zeros_like(D), np.zeros_like(O)
    rc = L.oracle_stair(N, n, _p(D), _p(O), _p(Pd), _p(Po))
    return Pd, Po, rc


def bt_dense(D, O):
    """Dense (N n) x (N n) matrix from block-tridiagonal blocks."""
    L = _load()
    N, n = D.shape[0], D.shape[1]
    D, O = _f64(D), _f64(O)
    M = np.zeros((N * n, N * n))
    L.oracle_bt_dense(N, n, _p(D), _p(O), _p(M))
    return M


def pcg(D, O, Pd, Po, gamma, eps, max_iters, lambda0=None, stop_rule=0):
    """PCG on S lambda = gamma; returns (lambda [N][n], iterations, converged).

    stop_rule 0: ||r|| <= eps ||gamma||;  1: r^T Phi^-1 r <= eps^2 eta0;
    2: r^T D^-1 r <= eps^2 gamma^T D^-1 gamma (D = blockdiag(S))."""
    L = _load()
    N, n = D.shape[0], D.shape[1]
    args = [_f64(x) for x in (D, O, Pd, Po, gamma)]
    lam = np.zeros((N, n))
    it = ctypes.c_int(0)
    rc = L.oracle_pcg(N, n, *[_p(a) for a in args],
                      _p(_f64(lambda0)) if lambda0 is not None else None,
                      float(eps), int(max_iters), int(stop_rule), _p(lam), ctypes.byref(it))
    return lam, it.value, rc == 0


def block_cholesky(D, O, gamma):
    """Direct fp64 solve of S lambda = gamma by block-tridiagonal Cholesky."""
    L = _load()
    N, n = D.shape[0], D.shape[1]
    D, O, gamma = _f64(D), _f64(O), _f64(gamma)
    lam = np.zeros((N, n))
    if L.oracle_block_cholesky(N, n, _p(D), _p(O), _p(gamma), _p(lam)):
        raise np.linalg.LinAlgError("S is not positive definite")
    return lam


def recover(prob, lam):
    """dz from lambda (eq. (4)); returns (dX [N][n], dU [N-1][m])."""
    L = _load()
    N, n, m = _dims(prob, batched=False)
    Q, R, q, r, A, B, _, _ = _one(prob, None)
    dX, dU = np.zeros((N, n)), np.zeros((max(N - 1, 0), m))
    L.oracle_recover(N, n, m, _p(Q), _p(R), _p(q), _p(r), _p(A), _p(B), _p(_f64(lam)),
                     _p(dX), _p(dU))
    return dX, dU


def merit(prob, dX, dU, alpha, mu):
    """L1 merit at step alpha: (merit, J, ||c||_1)."""
    L = _load()
    N, n, m = _dims(prob, batched=False)
    arr = _one(prob, None)
    J, v = ctypes.c_double(0), ctypes.c_double(0)
    val = L.oracle_merit(N, n, m, *[_p(a) for a in arr], _p(_f64(dX)), _p(_f64(dU)),
                         float(alpha), float(mu), ctypes.byref(J), ctypes.byref(v))
    return val, J.value, v.value


def linesearch(prob, dX, dU, n_alpha=8, beta=2.0, mu=10.0):
    """Exhaustive line search: (merit [n_alpha+1], best)."""
    L = _load()
    N, n, m = _dims(prob, batched=False)
    arr = _one(prob, None)
    out = np.zeros(n_alpha + 1)
    best = L.oracle_linesearch(N, n, m, *[_p(a) for a in arr], _p(_f64(dX)), _p(_f64(dU)),
                               int(n_alpha), float(beta), float(mu), _p(out))
    return out, best


def direct_solve(prob):
    """Reference fp64 solution through Schur + block Cholesky: (dX, dU, lambda)."""
    D, O, g, rc = schur(prob)
    if rc:
        raise np.linalg.LinAlgError("Q or R not positive definite")
    lam = block_cholesky(D, O, g)
    dX, dU = recover(prob, lam)
    return dX, dU, lam


def solve_kkt(prob, eps=1e-6, max_iters=200, n_alpha=8, beta=2.0, mu=10.0, stop_rule=0):
    """Whole path for one solve (Schur, stair, PCG, recovery, line search)."""
    L = _load()
    N, n, m = _dims(prob, batched=False)
    arr = _one(prob, None)
    dX, dU, lam = np.zeros((N, n)), np.zeros((max(N - 1, 0), m)), np.zeros((N, n))
    merit_out = np.zeros(n_alpha + 1)
    it, best = ctypes.c_int(0), ctypes.c_int(0)
    status = L.oracle_solve_kkt(N, n, m, *[_p(a) for a in arr], float(eps), int(max_iters),
                                int(stop_rule), int(n_alpha), float(beta), float(mu), _p(dX), _p(dU),
                                _p(lam), ctypes.byref(it), _p(merit_out), ctypes.byref(best))
    return dict(dX=dX, dU=dU, lam=lam, iters=it.value, merit=merit_out, best=best.value,
                status=status)


# ----------------------------------------------------------------------------
# batch helpers (prob holds M solves stacked on axis 0)
# ----------------------------------------------------------------------------

def solve_one(prob, j: int) -> Dict[str, np.ndarray]:
    """Solve j of a batch as a single-solve dict."""
    return {k: prob[k][j] for k in _KEYS}


def batch_direct(prob, solves=None):
    M = prob["Q"].shape[0]
    solves = range(M) if solves is None else solves
    out = [direct_solve(solve_one(prob, j)) for j in solves]
    return [np.stack([o[i] for o in out]) for i in range(3)]


def batch_solve_kkt(prob, solves=None, **kw):
    M = prob["Q"].shape[0]
    solves = range(M) if solves is None else solves
    return [solve_kkt(solve_one(prob, j), **kw) for j in solves]


# ----------------------------------------------------------------------------
# SQP on the linear model (x_{k+1} = A_k x_k + B_k u_k + c_k, x_0 = xs)
# ----------------------------------------------------------------------------

_MODEL_KEYS = ("Q", "R", "q", "r", "A", "B", "c", "xs")


def sqp_linear(model, iters, rho, rho_factor=10.0, rho_min=1e-8, rho_max=10.0, n_alpha=8,
               beta=2.0, mu=10.0, X0=None, U0=None):
    """fp64 SQP loop on one linear-model problem (model holds Q, R, q, r, A,
    B, c, xs of one solve); starts from (X0, U0), zero by default.  Returns
    dict(X, U, lam, merit_hist [iters+1], best_hist [iters], rho_hist
    [iters+1], status)."""
    L = _load()
    N, n, m = _dims(model, batched=False)
    arr = [_f64(model[k]) for k in _MODEL_KEYS]
    X = np.zeros((N, n)) if X0 is None else _f64(X0).copy()
    U = np.zeros((max(N - 1, 0), m)) if U0 is None else _f64(U0).copy()
    lam = np.zeros((N, n))
    hist, rhos = np.zeros(iters + 1), np.zeros(iters + 1)
    best = np.zeros(iters, dtype=np.int32)
    status = L.oracle_sqp_linear(N, n, m, *[_p(a) for a in arr], int(iters), float(rho),
                                 float(rho_factor), float(rho_min), float(rho_max),
                                 int(n_alpha), float(beta), float(mu), _p(X), _p(U), _p(lam),
                                 _p(hist), best.ctypes.data_as(ctypes.POINTER(ctypes.c_int)),
                                 _p(rhos))
    return dict(X=X, U=U, lam=lam, merit_hist=hist, best_hist=best, rho_hist=rhos,
                status=status)


def model_one(model, j: int) -> Dict[str, np.ndarray]:
    """Problem j of a batch of linear models as a single-problem dict."""
    return {k: model[k][j] for k in _MODEL_KEYS}
