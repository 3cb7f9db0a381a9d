"""Pins for the fp64 oracle: checks against things other than the oracle itself.

Each test ties an oracle routine to a fact fixed by the GATO paper's
equations or by the mathematics (hand-worked values, an independent
condensed-QP solve, a library CG, spectral bounds, closed forms), chosen so
that a dropped term, a wrong sign or a transposed block fails at least one.
"""
import json
import os

import numpy as np
import pytest
import scipy.sparse.linalg as spla

import oracle
from trajectory_optimization_kkt_gb300.workloads import WORKLOADS, make_batch, random_lq

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")

TINY = [(1, 2, 1), (2, 1, 1), (3, 3, 2), (4, 4, 2), (5, 3, 3)]


def tiny_problem(N, n, m, seed=7, **kw):
    return oracle.solve_one(random_lq(1, N, n, m, seed, **kw), 0)


def f64(p):
    return {k: np.asarray(v, dtype=np.float64) for k, v in p.items()}


def rel(a, b):
    a, b = np.ravel(a), np.ravel(b)
    return np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300)


# --------------------------------------------------------------------------
# hand-worked instance (golden fixture, derivation inside the file)
# --------------------------------------------------------------------------

def load_scalar():
    with open(os.path.join(GOLDEN, "scalar_N2.json")) as f:
        g = json.load(f)
    prob = {k: np.array(g[k], dtype=np.float64) for k in ("Q", "R", "q", "r", "A", "B", "e", "s0")}
    return prob, g


def test_hand_worked_instance_all_routines():
    prob, g = load_scalar()
    for method in ("ldlt", "lu"):
        dX, dU, lam = oracle.kkt_dense(prob, method)
        np.testing.assert_allclose(dX, g["dX"], atol=1e-14)
        np.testing.assert_allclose(dU, g["dU"], atol=1e-14)
        np.testing.assert_allclose(lam, g["lambda"], atol=1e-14)
    D, O, gam, rc = oracle.schur(prob)
    assert rc == 0
    np.testing.assert_allclose(D, g["S_diag"], atol=1e-14)
    np.testing.assert_allclose(O, g["S_off"], atol=1e-14)
    np.testing.assert_allclose(gam, g["gamma"], atol=1e-14)
    dX, dU, lam = oracle.direct_solve(prob)
    np.testing.assert_allclose(lam, g["lambda"], atol=1e-14)
    Pd, Po, _ = oracle.stair(D, O)
    lam_p, it, ok = oracle.pcg(D, O, Pd, Po, gam, 1e-12, 10)
    assert ok and it <= 2
    np.testing.assert_allclose(lam_p, g["lambda"], atol=1e-12)
    for a, v in zip(g["merit_alpha"], g["merit_value"]):
        val, _, _ = oracle.merit(prob, np.array(g["dX"]), np.array(g["dU"]), a, g["mu"])
        assert val == pytest.approx(v, abs=1e-13)
    merit, best = oracle.linesearch(prob, np.array(g["dX"]), np.array(g["dU"]), 8, 2.0, g["mu"])
    assert best == g["best"]
    assert merit[0] == pytest.approx(3.0, abs=1e-14)


# --------------------------------------------------------------------------
# P1: Schur path == dense KKT (LDL^T and LU), the definition of eq. (2)
# --------------------------------------------------------------------------

def _schur_cases():
    cases = [(f"tiny{N}_{n}_{m}", tiny_problem(N, n, m), 1e-10) for N, n, m in TINY]
    b0 = make_batch(WORKLOADS[0])
    cases.append(("cfg0", oracle.solve_one(b0, 0), 1e-10))
    b1 = make_batch(WORKLOADS[1], M=2)
    cases += [(f"cfg1_{j}", oracle.solve_one(b1, j), 1e-10) for j in range(2)]
    b3 = make_batch(WORKLOADS[3], M=2)
    # the log-scaled blocks have cond ~1e6; 1e-16 * cond bounds the agreement
    cases += [(f"cfg3_{j}", oracle.solve_one(b3, j), 1e-8) for j in range(2)]
    return cases


@pytest.mark.parametrize("name,prob,tol", _schur_cases(), ids=lambda x: x if isinstance(x, str) else "")
def test_schur_equals_dense_kkt(name, prob, tol):
    dX, dU, lam = oracle.direct_solve(prob)
    for method in ("ldlt", "lu"):
        kX, kU, kl = oracle.kkt_dense(prob, method)
        assert rel(dX, kX) < tol, (method, rel(dX, kX))
        assert rel(dU, kU) < tol, (method, rel(dU, kU))
        assert rel(lam, kl) < tol, (method, rel(lam, kl))


# --------------------------------------------------------------------------
# P2: KKT residuals, written per knot from the QP's optimality conditions
# --------------------------------------------------------------------------

def kkt_residuals(p, dX, dU, lam):
    """max-norm of stationarity and feasibility of eq. (1) at (dz, lambda)."""
    Q, R, q, r, A, B, e, s0 = (p[k] for k in ("Q", "R", "q", "r", "A", "B", "e", "s0"))
    N = Q.shape[0]
    res = [np.abs(dX[0] - s0).max()]
    for k in range(N):
        st = Q[k] @ dX[k] + q[k] - lam[k]
        if k < N - 1:
            st += A[k].T @ lam[k + 1]
            res.append(np.abs(R[k] @ dU[k] + r[k] + B[k].T @ lam[k + 1]).max())
            res.append(np.abs(A[k] @ dX[k] + B[k] @ dU[k] + e[k] - dX[k + 1]).max())
        res.append(np.abs(st).max())
    return max(res)


@pytest.mark.parametrize("N,n,m", TINY + [(16, 14, 7)])
def test_kkt_residuals_vanish(N, n, m):
    p = f64(tiny_problem(N, n, m, seed=11))
    for solver in ("direct", "ldlt", "lu"):
        if solver == "direct":
            dX, dU, lam = oracle.direct_solve(p)
        else:
            dX, dU, lam = oracle.kkt_dense(p, solver)
        scale = max(np.abs(lam).max(), 1.0)
        assert kkt_residuals(p, dX, dU, lam) < 1e-10 * scale


def condensed_qp(p):
    """Independent primal solve: eliminate the states by forward simulation
    (x_0 = s0, x_{k+1} = A x + B u + e), then minimise the cost over U with a
    dense normal-equation solve.  Shares nothing with the KKT/Schur code."""
    Q, R, q, r, A, B, e, s0 = (p[k] for k in ("Q", "R", "q", "r", "A", "B", "e", "s0"))
    N, n, m = Q.shape[0], Q.shape[1], B.shape[-1]
    nu = (N - 1) * m
    # x_k = c_k + T_k U  (affine in the stacked controls U)
    c = [s0.copy()]
    T = [np.zeros((n, nu))]
    for k in range(N - 1):
        Tk = A[k] @ T[k]
        Tk[:, k * m:(k + 1) * m] += B[k]
        T.append(Tk)
        c.append(A[k] @ c[k] + e[k])
    H = np.zeros((nu, nu))
    h = np.zeros(nu)
    for k in range(N):
        H += T[k].T @ Q[k] @ T[k]
        h += T[k].T @ (Q[k] @ c[k] + q[k])
    for k in range(N - 1):
        sl = slice(k * m, (k + 1) * m)
        H[sl, sl] += R[k]
        h[sl] += r[k]
    U = np.linalg.solve(H, -h) if nu else np.zeros(0)
    X = np.stack([c[k] + T[k] @ U for k in range(N)])
    return X, U.reshape(N - 1, m)


@pytest.mark.parametrize("N,n,m", TINY + [(16, 14, 7), (8, 6, 3)])
def test_primal_equals_condensed_qp(N, n, m):
    p = f64(tiny_problem(N, n, m, seed=3))
    X, U = condensed_qp(p)
    dX, dU, _ = oracle.direct_solve(p)
    assert rel(dX, X) < 1e-9
    if N > 1:
        assert rel(dU, U) < 1e-9


# --------------------------------------------------------------------------
# P3/P4: S symmetric positive definite; stair preconditioner spectrum
# --------------------------------------------------------------------------

@pytest.mark.parametrize("N,n,m", TINY + [(16, 14, 7), (6, 5, 2)])
def test_S_spd_and_stair_spectrum(N, n, m):
    p = tiny_problem(N, n, m, seed=5, a_sigma=0.3)
    D, O, gam, rc = oracle.schur(p)
    assert rc == 0
    S = oracle.bt_dense(D, O)
    for j in range(N):
        np.testing.assert_allclose(D[j], D[j].T, atol=1e-12 * np.abs(D[j]).max())
    assert np.linalg.eigvalsh(0.5 * (S + S.T)).min() > 0
    np.linalg.cholesky(S)
    Pd, Po, rc = oracle.stair(D, O)
    assert rc == 0
    P = oracle.bt_dense(Pd, Po)
    assert np.linalg.eigvalsh(0.5 * (P + P.T)).min() > 0
    ev = np.linalg.eigvals(P @ S)
    assert np.abs(ev.imag).max() < 1e-8
    assert ev.real.min() > 0
    assert ev.real.max() <= 1.0 + 1e-9


def test_stair_inverts_block_diagonal_when_A_is_zero():
    """A = 0 decouples the knots: S is block diagonal, Phi^-1 = S^-1 and PCG
    stops after one iteration."""
    p = tiny_problem(6, 4, 2, seed=9, a_sigma=0.0)
    p = dict(p)
    p["A"] = np.zeros_like(p["A"])
    D, O, gam, _ = oracle.schur(p)
    assert np.abs(O).max() == 0.0
    Pd, Po, _ = oracle.stair(D, O)
    S, P = oracle.bt_dense(D, O), oracle.bt_dense(Pd, Po)
    np.testing.assert_allclose(P @ S, np.eye(S.shape[0]), atol=1e-10)
    lam, it, ok = oracle.pcg(D, O, Pd, Po, gam, 1e-10, 50)
    assert ok and it == 1


# --------------------------------------------------------------------------
# PCG: iterates equal a library PCG's; converges to the direct solution
# --------------------------------------------------------------------------

@pytest.mark.parametrize("k", [1, 2, 5, 9])
def test_pcg_iterates_match_scipy(k):
    p = tiny_problem(8, 4, 2, seed=21, a_sigma=0.2)
    D, O, gam, _ = oracle.schur(p)
    Pd, Po, _ = oracle.stair(D, O)
    S, P = oracle.bt_dense(D, O), oracle.bt_dense(Pd, Po)
    lam, it, _ = oracle.pcg(D, O, Pd, Po, gam, 0.0, k)
    assert it == k
    Mop = spla.LinearOperator(S.shape, matvec=lambda x: P @ x)
    ref, _ = spla.cg(S, gam.ravel(), rtol=1e-300, atol=0.0, maxiter=k, M=Mop)
    assert rel(lam, ref) < 1e-9


@pytest.mark.parametrize("stop_rule", [0, 1, 2])
@pytest.mark.parametrize("w", [0, 1, 2, 4])
def test_pcg_tight_tolerance_reaches_direct(w, stop_rule):
    prob = oracle.solve_one(make_batch(WORKLOADS[w], M=1, N=min(WORKLOADS[w].N, 32)), 0)
    D, O, gam, _ = oracle.schur(prob)
    Pd, Po, _ = oracle.stair(D, O)
    lam, it, ok = oracle.pcg(D, O, Pd, Po, gam, 1e-12, 5000, stop_rule=stop_rule)
    assert ok
    assert rel(lam, oracle.block_cholesky(D, O, gam)) < 1e-8


def test_pcg_finite_termination_and_warm_start():
    p = tiny_problem(3, 2, 1, seed=4)
    D, O, gam, _ = oracle.schur(p)
    Pd, Po, _ = oracle.stair(D, O)
    exact = oracle.block_cholesky(D, O, gam)
    # dimension 6: CG terminates in at most 6 steps in exact arithmetic
    lam, it, ok = oracle.pcg(D, O, Pd, Po, gam, 1e-11, 6)
    assert ok and rel(lam, exact) < 1e-9
    # warm start at the solution: converged before the first iteration
    lam, it, ok = oracle.pcg(D, O, Pd, Po, gam, 1e-6, 50, lambda0=exact)
    assert ok and it == 0
    # zero right-hand side: zero iterations, zero solution
    lam, it, ok = oracle.pcg(D, O, Pd, Po, np.zeros_like(gam), 1e-6, 50)
    assert ok and it == 0 and not lam.any()


def test_pcg_reports_cap():
    prob = oracle.solve_one(make_batch(WORKLOADS[4], M=1), 0)
    D, O, gam, _ = oracle.schur(prob)
    Pd, Po, _ = oracle.stair(D, O)
    lam, it, ok = oracle.pcg(D, O, Pd, Po, gam, 1e-6, 5)
    assert not ok and it == 5


def test_block_cholesky_matches_numpy():
    p = tiny_problem(7, 5, 2, seed=8, a_sigma=0.4)
    D, O, gam, _ = oracle.schur(p)
    ref = np.linalg.solve(oracle.bt_dense(D, O), gam.ravel())
    assert rel(oracle.block_cholesky(D, O, gam), ref) < 1e-11


# --------------------------------------------------------------------------
# P5: closed forms
# --------------------------------------------------------------------------

def test_single_knot_closed_form():
    """N = 1: S = Q_0^-1, lambda_0 = Q_0 s0 + q_0 and dx_0 = s0."""
    p = f64(tiny_problem(1, 5, 2, seed=13))
    D, O, gam, _ = oracle.schur(p)
    np.testing.assert_allclose(D[0], np.linalg.inv(p["Q"][0]), rtol=1e-10, atol=1e-12)
    dX, dU, lam = oracle.direct_solve(p)
    np.testing.assert_allclose(lam[0], p["Q"][0] @ p["s0"] + p["q"][0], rtol=1e-10)
    np.testing.assert_allclose(dX[0], p["s0"], rtol=1e-12, atol=1e-14)


def test_identity_chain_closed_form():
    """Q = R = I, A = I, B = 0: S is the grounded path Laplacian
    S_00 = I, S_jj = 2 I, S_{j,j-1} = -I, and gamma_j = e_{j-1} - q_{j-1} + q_j."""
    N, n, m = 5, 3, 2
    p = f64(tiny_problem(N, n, m, seed=17))
    p["Q"][:] = np.eye(n)
    p["R"][:] = np.eye(m)
    p["A"][:] = np.eye(n)
    p["B"][:] = 0.0
    D, O, gam, _ = oracle.schur(p)
    np.testing.assert_allclose(D[0], np.eye(n), atol=1e-15)
    for j in range(1, N):
        np.testing.assert_allclose(D[j], 2 * np.eye(n), atol=1e-15)
        np.testing.assert_allclose(O[j - 1], -np.eye(n), atol=1e-15)
        np.testing.assert_allclose(gam[j], p["e"][j - 1] - p["q"][j - 1] + p["q"][j], atol=1e-14)
    np.testing.assert_allclose(gam[0], p["s0"] + p["q"][0], atol=1e-15)


def merit_closed_form(p, dX, dU, alpha, mu):
    """M(alpha) = alpha g^T dz + 1/2 alpha^2 dz^T G dz + mu ||c(alpha)||_1 with
    c(alpha) = c_0 + alpha C dz, written from the quadratic's expansion."""
    Q, R, q, r, A, B, e, s0 = (p[k] for k in ("Q", "R", "q", "r", "A", "B", "e", "s0"))
    lin = np.einsum("ki,ki->", q, dX) + np.einsum("ki,ki->", r, dU)
    quad = np.einsum("ki,kij,kj->", dX, Q, dX) + np.einsum("ki,kij,kj->", dU, R, dU)
    Cdz = np.einsum("kij,kj->ki", A, dX[:-1]) + np.einsum("kij,kj->ki", B, dU) - dX[1:]
    viol = np.abs(alpha * dX[0] - s0).sum() + np.abs(e + alpha * Cdz).sum()
    return alpha * lin + 0.5 * alpha ** 2 * quad + mu * viol


@pytest.mark.parametrize("scale", [1.0, 3.0, 0.3, -1.0])
def test_merit_full_formula_equals_expansion(scale):
    p = f64(tiny_problem(9, 4, 2, seed=23))
    dX, dU, _ = oracle.direct_solve(p)
    dX, dU = scale * dX, scale * dU
    for a in [0.0, 1.0, 0.5, 0.125, 1 / 128]:
        val, J, viol = oracle.merit(p, dX, dU, a, 10.0)
        assert val == pytest.approx(merit_closed_form(p, dX, dU, a, 10.0), rel=1e-12, abs=1e-12)


def test_merit_at_zero_and_exact_step_violation():
    p = f64(tiny_problem(9, 4, 2, seed=29))
    dX, dU, _ = oracle.direct_solve(p)
    val0, J0, v0 = oracle.merit(p, dX, dU, 0.0, 10.0)
    c0 = np.abs(p["s0"]).sum() + np.abs(p["e"]).sum()
    assert J0 == 0.0 and v0 == pytest.approx(c0, rel=1e-14)
    assert val0 == pytest.approx(10.0 * c0, rel=1e-14)
    for a in [1.0, 0.5, 0.25]:
        _, _, v = oracle.merit(p, dX, dU, a, 10.0)
        assert v == pytest.approx((1 - a) * c0, rel=1e-9, abs=1e-12)


# --------------------------------------------------------------------------
# P6: line search selection against a brute-force scan of the closed form
# --------------------------------------------------------------------------

@pytest.mark.parametrize("scale", [1.0, 2.5, 6.0, 40.0])
def test_linesearch_selects_brute_force_best(scale):
    p = f64(tiny_problem(6, 3, 2, seed=31))
    dX, dU, _ = oracle.direct_solve(p)
    dX, dU = scale * dX, scale * dU
    merit, best = oracle.linesearch(p, dX, dU, 8, 2.0, 10.0)
    alphas = 2.0 ** -np.arange(8)
    closed = np.array([merit_closed_form(p, dX, dU, a, 10.0) for a in alphas])
    np.testing.assert_allclose(merit[1:], closed, rtol=1e-11, atol=1e-11)
    # brute force over a fine grid: the continuous minimiser lies within a
    # factor-2 bracket of the chosen candidate (the merit is convex in alpha)
    grid = np.linspace(1e-4, 1.0, 10000)
    a_star = grid[np.argmin([merit_closed_form(p, dX, dU, a, 10.0) for a in grid])]
    assert best == int(np.argmin(closed))
    assert alphas[best] / 2 <= a_star * (1 + 1e-9) and a_star <= min(2 * alphas[best], 1.0) + 1e-9
    if scale > 3:
        assert best > 0


def test_linesearch_rejects_ascent_direction():
    p = f64(tiny_problem(6, 3, 2, seed=37))
    dX, dU, _ = oracle.direct_solve(p)
    merit, best = oracle.linesearch(p, -dX, -dU, 8, 2.0, 10.0)
    assert best == -1
    assert (merit[1:] >= merit[0]).all()


def test_linesearch_ties_take_the_lowest_index():
    """A zero step makes every candidate equal to M(0): no decrease, and the
    argmin over tied values would be index 0."""
    p = f64(tiny_problem(4, 3, 2, seed=41))
    z = np.zeros((4, 3)), np.zeros((3, 2))
    merit, best = oracle.linesearch(p, *z, 8, 2.0, 10.0)
    assert (merit == merit[0]).all() and best == -1


def test_linesearch_exact_tie_keeps_larger_step():
    """N = 1, Q = 1, q = -3/4, s0 = 0, mu = 0 and dx = 1: M(1) = M(1/2) = -1/4
    exactly (dyadic values), so the tie must resolve to index 0 (alpha = 1)."""
    p = dict(Q=np.ones((1, 1, 1)), R=np.zeros((0, 1, 1)), q=np.array([[-0.75]]),
             r=np.zeros((0, 1)), A=np.zeros((0, 1, 1)), B=np.zeros((0, 1, 1)),
             e=np.zeros((0, 1)), s0=np.zeros(1))
    merit, best = oracle.linesearch(p, np.ones((1, 1)), np.zeros((0, 1)), 8, 2.0, 0.0)
    assert merit[1] == merit[2] == -0.25
    assert best == 0


# --------------------------------------------------------------------------
# whole path
# --------------------------------------------------------------------------

def test_solve_kkt_pipeline_status():
    prob = oracle.solve_one(make_batch(WORKLOADS[0]), 0)
    out = oracle.solve_kkt(prob, 1e-6, 200)
    assert out["status"] == 0 and out["best"] == 0 and 0 < out["iters"] < 200
    dX, dU, lam = oracle.direct_solve(prob)
    z = np.concatenate([out["dX"].ravel(), out["dU"].ravel()])
    zr = np.concatenate([dX.ravel(), dU.ravel()])
    assert rel(z, zr) < 1e-5
    capped = oracle.solve_kkt(prob, 1e-6, 3)
    assert capped["status"] & 1 and capped["iters"] == 3


def test_indefinite_Q_is_flagged():
    prob = dict(oracle.solve_one(make_batch(WORKLOADS[0]), 0))
    prob["Q"] = prob["Q"].copy()
    prob["Q"][3] = -np.eye(14, dtype=np.float32)
    out = oracle.solve_kkt(prob, 1e-6, 20)
    assert out["status"] & 2


# --------------------------------------------------------------------------
# stored regression values (written by tests/golden/make_golden.py)
# --------------------------------------------------------------------------

def test_golden_workload0_regression():
    path = os.path.join(GOLDEN, "workload0_oracle.npz")
    g = np.load(path)
    prob = oracle.solve_one(make_batch(WORKLOADS[0]), 0)
    for k in ("Q", "q", "A", "s0"):
        np.testing.assert_array_equal(prob[k], g["in_" + k])
    dX, dU, lam = oracle.direct_solve(prob)
    np.testing.assert_allclose(lam, g["lam"], rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(dX, g["dX"], rtol=1e-11, atol=1e-13)
    out = oracle.solve_kkt(prob, 1e-6, 200)
    assert out["iters"] == int(g["pcg_iters"])
    np.testing.assert_allclose(out["merit"], g["merit"], rtol=1e-11)
    assert out["best"] == int(g["best"])
