"""Pins for the oracle's SQP loop on the linear model (GATO paper Sec. II steps
1-3 with the rho damping of Sec. IV-C): each test ties oracle.sqp_linear to a
fact computed here independently of the oracle's C code (the condensed QP, a
dense proximal KKT solve, the merit by its definition) or to the damping
rule's exact trace."""
import numpy as np
import pytest

import oracle
from test_oracle_pins import condensed_qp, rel
from trajectory_optimization_kkt_gb300.workloads import linear_models


def model(N, n, m, seed=11):
    return {k: v.astype(np.float64) for k, v in oracle.model_one(
        linear_models(1, N, n, m, seed), 0).items()}


def true_merit(p, X, U, mu):
    """J(X, U) + mu ||c(X, U)||_1 of the linear model, by definition."""
    J, viol = 0.0, np.abs(X[0] - p["xs"]).sum()
    for k in range(len(X)):
        J += 0.5 * X[k] @ p["Q"][k] @ X[k] + p["q"][k] @ X[k]
        if k < len(X) - 1:
            J += 0.5 * U[k] @ p["R"][k] @ U[k] + p["r"][k] @ U[k]
            viol += np.abs(p["A"][k] @ X[k] + p["B"][k] @ U[k] + p["c"][k] - X[k + 1]).sum()
    return J + mu * viol


def optimum(p):
    X, U = condensed_qp(dict(p, e=p["c"], s0=p["xs"]))
    return X, U


def dense_damped_step(p, X, U, rho):
    """The damped subproblem at (X, U) assembled densely: minimise
    J(X + dX, U + dU) + rho/2 sum ||dx_k||^2 subject to the (linear)
    dynamics and x_0 = xs; returns (dX, dU)."""
    Q, R, A, B = p["Q"], p["R"], p["A"], p["B"]
    N, n, m = Q.shape[0], Q.shape[1], B.shape[-1]
    nz = N * n + (N - 1) * m
    ix = lambda k: slice(k * n, (k + 1) * n)  # noqa: E731
    iu = lambda k: slice(N * n + k * m, N * n + (k + 1) * m)  # noqa: E731
    H, g = np.zeros((nz, nz)), np.zeros(nz)
    for k in range(N):
        H[ix(k), ix(k)] = Q[k] + rho * np.eye(n)
        g[ix(k)] = Q[k] @ X[k] + p["q"][k]
    for k in range(N - 1):
        H[iu(k), iu(k)] = R[k]
        g[iu(k)] = R[k] @ U[k] + p["r"][k]
    C, d = np.zeros((N * n, nz)), np.zeros(N * n)
    C[:n, ix(0)] = np.eye(n)
    d[:n] = p["xs"] - X[0]
    for k in range(N - 1):
        rows = slice((k + 1) * n, (k + 2) * n)
        C[rows, ix(k)] = A[k]
        C[rows, iu(k)] = B[k]
        C[rows, ix(k + 1)] = -np.eye(n)
        d[rows] = -(A[k] @ X[k] + B[k] @ U[k] + p["c"][k] - X[k + 1])
    K = np.block([[H, C.T], [C, np.zeros((N * n, N * n))]])
    sol = np.linalg.solve(K, np.concatenate([-g, d]))
    return sol[:N * n].reshape(N, n), sol[N * n:nz].reshape(N - 1, m)


@pytest.mark.parametrize("N,n,m", [(2, 1, 1), (5, 3, 2), (16, 14, 7)])
def test_undamped_step_reaches_the_optimum(N, n, m):
    p = model(N, n, m)
    out = oracle.sqp_linear(p, 1, rho=0.0, rho_min=0.0)
    X, U = optimum(p)
    assert out["best_hist"][0] == 0  # the full step
    assert rel(out["X"], X) < 1e-9 and rel(out["U"], U) < 1e-9
    assert abs(out["merit_hist"][1] - true_merit(p, X, U, 10.0)) < 1e-9 * abs(
        out["merit_hist"][0])


@pytest.mark.parametrize("rho", [0.3, 5.0])
def test_damped_step_equals_dense_proximal_solve(rho):
    p = model(7, 4, 2, seed=5)
    rng = np.random.default_rng(0)
    X0, U0 = rng.standard_normal((7, 4)), rng.standard_normal((6, 2))
    out = oracle.sqp_linear(p, 1, rho=rho, X0=X0, U0=U0)
    best = out["best_hist"][0]
    assert best >= 0
    alpha = 2.0 ** -best
    dX, dU = dense_damped_step(p, X0, U0, rho)
    assert rel((out["X"] - X0) / alpha, dX) < 1e-9
    assert rel((out["U"] - U0) / alpha, dU) < 1e-9
    assert out["rho_hist"][0] == rho
    # the line search ranks the problem's own merit, not the damped model's
    h = out["merit_hist"]
    assert abs(h[0] - true_merit(p, X0, U0, 10.0)) < 1e-9 * abs(h[0])
    assert abs(h[1] - true_merit(p, out["X"], out["U"], 10.0)) < 1e-9 * abs(h[0])


def test_merit_history_is_the_true_merit_and_converges():
    p = model(16, 6, 3, seed=2)
    out = oracle.sqp_linear(p, 25, rho=1e-3)
    h = out["merit_hist"]
    assert np.all(np.diff(h) <= 1e-12 * abs(h[0]))  # accepted steps decrease, failures keep
    assert abs(h[-1] - true_merit(p, out["X"], out["U"], 10.0)) < 1e-9 * abs(h[0])
    assert abs(h[0] - true_merit(p, np.zeros((16, 6)), np.zeros((15, 3)), 10.0)) < 1e-12
    X, U = optimum(p)
    assert rel(out["X"], X) < 1e-7 and rel(out["U"], U) < 1e-7
    assert abs(h[-1] - true_merit(p, X, U, 10.0)) < 1e-9 * abs(h[0])


def test_rho_grows_while_every_line_search_fails():
    """Zero data at the zero trajectory: the step is exactly zero, no
    candidate beats alpha = 0, so rho is multiplied by the factor each
    iteration until it reaches rho_max."""
    p = model(6, 3, 2)
    for k in ("q", "r", "c", "xs"):
        p[k] = np.zeros_like(p[k])
    out = oracle.sqp_linear(p, 6, rho=1e-3, rho_factor=10.0, rho_max=5.0)
    assert (out["best_hist"] == -1).all() and out["status"] & 4
    np.testing.assert_array_equal(out["rho_hist"], [1e-3, 1e-2, 1e-1, 1.0, 5.0, 5.0, 5.0])
    assert (out["merit_hist"] == 0).all()


def test_rho_shrinks_after_accepted_steps():
    p = model(10, 4, 2, seed=9)
    out = oracle.sqp_linear(p, 4, rho=1.0, rho_factor=10.0, rho_min=1e-2)
    assert (out["best_hist"] >= 0).all()
    np.testing.assert_allclose(out["rho_hist"], [1.0, 0.1, 1e-2, 1e-2, 1e-2], rtol=0, atol=0)
