"""GPU parity of the SQP loop on the linear model (gato_sqp_linear) against
the fp64 oracle's loop.

Both loops run the same iterations independently.  Once a problem has
converged, fp32 cannot resolve the line search's merit differences (they are
rounding noise), so accept/reject decisions there are arbitrary on either
side; the merit histories are therefore compared on the scale of the initial
suboptimality, |h_gpu - h_oracle| <= 1e-3 (h_0 - J*) + 1e-5 |J*|, and the
damping traces exactly only where neither side has converged.  The damping
rule itself is checked exactly on runs whose decisions are certain.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import oracle  # noqa: E402
from trajectory_optimization_kkt_gb300 import gato  # noqa: E402
from trajectory_optimization_kkt_gb300.workloads import (  # noqa: E402
    linear_models, replicate, rho_logspace)

from test_oracle_sqp_pins import optimum, true_merit  # noqa: E402

PCG, CR = gato.GATO_LINSYS_PCG, gato.GATO_LINSYS_BDSV


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()


def run(model, rho0, iters, params, sqp=None, X0=None, U0=None, solver=None, lam0=None):
    M, N, n = model["Q"].shape[:3]
    m = model["B"].shape[-1]
    d = gato.to_device(model)
    f = dict(device="cuda", dtype=torch.float32)
    X = torch.zeros(M, N, n, **f) if X0 is None else torch.tensor(X0, **f)
    U = torch.zeros(M, N - 1, m, **f) if U0 is None else torch.tensor(U0, **f)
    lam = torch.zeros(M, N, n, **f) if lam0 is None else torch.tensor(lam0, **f)
    rho = torch.tensor(rho0, **f)
    hist = torch.full((M, iters + 1), np.nan, **f)
    ih = torch.full((M, iters), -1, device="cuda", dtype=torch.int32)
    status = torch.zeros(M, device="cuda", dtype=torch.int32)
    sp = sqp or gato.default_sqp_params()
    sp.iters = iters
    own = solver is None
    s = solver or gato.Solver(M, N, n, m)
    try:
        s.sqp_linear(params, sp, d, X, U, lam, rho, hist, status, iters_hist=ih)
        torch.cuda.synchronize()
    finally:
        if own:
            s.close()
    return dict(X=X.cpu().numpy(), U=U.cpu().numpy(), lam=lam.cpu().numpy(),
                rho=rho.cpu().numpy(), hist=hist.cpu().numpy(), iters=ih.cpu().numpy(),
                status=status.cpu().numpy())


def params(linsys=PCG, **kw):
    base = dict(pcg_max_iters=2000, refine_steps=1, linsys=linsys)
    base.update(kw)
    return gato.default_params(**base)


@pytest.mark.parametrize("use_graph", [1, 0], ids=["graph", "stream"])
@pytest.mark.parametrize("linsys", [PCG, CR], ids=["pcg", "direct"])
def test_rho_sweep_matches_oracle(linsys, use_graph):
    one = oracle.model_one(linear_models(1, 24, 12, 6, seed=41), 0)
    M, K = 8, 6
    model = replicate(one, M)
    rho0 = rho_logspace(M)
    out = run(model, rho0, K, params(linsys), gato.default_sqp_params(use_graph=use_graph))
    p64 = {k: v.astype(np.float64) for k, v in one.items()}
    Xs, Us = optimum(p64)
    Jstar = true_merit(p64, Xs, Us, 10.0)
    for j in range(M):
        ref = oracle.sqp_linear(p64, K, float(rho0[j]))
        h, hr = out["hist"][j], ref["merit_hist"]
        tol = 1e-3 * (hr[0] - Jstar) + 1e-5 * abs(Jstar)
        assert np.abs(h - hr).max() <= tol, (j, h, hr)
        # the GPU's history is the true merit of its own trajectory
        assert abs(h[-1] - true_merit(p64, out["X"][j].astype(np.float64),
                                      out["U"][j].astype(np.float64), 10.0)) <= tol
        # when every oracle step still lowers the merit by more than fp32
        # can blur, the decisions are certain and the damping ends the same
        if np.all(np.diff(hr) < -1e-4 * (hr[0] - Jstar)):
            np.testing.assert_allclose(out["rho"][j], ref["rho_hist"][K], rtol=1e-5)
        assert (out["iters"][j] >= 0).all()
        if linsys == CR:
            assert (out["iters"][j] == 0).all()


@pytest.mark.parametrize("refine_solver", [0, 1], ids=["pcg_corrections", "direct_corrections"])
def test_graph_and_stream_paths_are_bit_identical(refine_solver):
    """Also with direct corrections, whose factorisation runs on a side stream
    forked from the iteration's stream and joined back (inside the recorded
    graph as dependencies)."""
    model = linear_models(4, 16, 14, 7, seed=43)
    rho0 = np.array([1e-6, 1e-3, 0.1, 3.0], dtype=np.float32)
    p = params(refine_solver=refine_solver)
    a = run(model, rho0, 5, p, gato.default_sqp_params(use_graph=1))
    b = run(model, rho0, 5, p, gato.default_sqp_params(use_graph=0))
    for k in a:
        assert np.array_equal(a[k], b[k], equal_nan=True), k


def test_first_iteration_takes_the_damped_kkt_step():
    """From the zero trajectory the first subproblem is the LQ subproblem
    with Q + rho I: its step is gato_solve_kkt's on that data."""
    model = linear_models(3, 20, 10, 5, seed=44)
    rho0 = np.array([0.5, 2.0, 1e-4], dtype=np.float32)
    out = run(model, rho0, 1, params(refine_steps=2))
    for j in range(3):
        p = {k: model[k][j].astype(np.float64) for k in model}
        lq = dict(Q=p["Q"] + rho0[j] * np.eye(10), R=p["R"], q=p["q"], r=p["r"], A=p["A"],
                  B=p["B"], e=p["c"], s0=p["xs"])
        dX, dU, _ = oracle.direct_solve(lq)
        ref = oracle.sqp_linear(p, 1, float(rho0[j]))
        alpha = 2.0 ** -int(ref["best_hist"][0])
        z = np.concatenate([out["X"][j].ravel(), out["U"][j].ravel()]) / alpha
        zr = np.concatenate([dX.ravel(), dU.ravel()])
        assert np.linalg.norm(z - zr) <= 1e-4 * np.linalg.norm(zr)


def test_damping_rule_on_certain_decisions():
    # zero data at the zero trajectory: the step is zero, every line search
    # fails, rho grows by the factor until rho_max
    model = linear_models(2, 8, 4, 2, seed=45)
    for k in ("q", "r", "c", "xs"):
        model[k] = np.zeros_like(model[k])
    rho0 = np.array([1e-3, 1.0], dtype=np.float32)
    sp = gato.default_sqp_params(rho_factor=10.0, rho_max=5.0)
    out = run(model, rho0, 3, params(), sp)  # 1e-3 -> 1e-2 -> 1e-1 -> 1; 1 -> 5 (clamped)
    np.testing.assert_allclose(out["rho"], [1.0, 5.0], rtol=1e-5)
    assert (out["status"] & gato.GATO_STATUS_LINESEARCH_FAILED).all()
    assert (out["hist"] == 0).all()
    # far from the optimum with heavy damping every step is accepted
    model = linear_models(2, 8, 4, 2, seed=46)
    out = run(model, np.array([10.0, 10.0], dtype=np.float32), 3, params(),
              gato.default_sqp_params(rho_factor=4.0, rho_min=1e-3))
    np.testing.assert_allclose(out["rho"], [10.0 / 64, 10.0 / 64], rtol=1e-6)
    assert np.all(np.diff(out["hist"], axis=1) < 0)


def test_warm_start_saves_pcg_iterations():
    model = linear_models(4, 32, 12, 6, seed=47)
    rho0 = np.full(4, 1e-2, dtype=np.float32)
    warm = run(model, rho0, 4, params(refine_steps=0), gato.default_sqp_params(warm_start=1))
    cold = run(model, rho0, 4, params(refine_steps=0), gato.default_sqp_params(warm_start=0))
    assert warm["iters"][:, 1:].sum() < cold["iters"][:, 1:].sum()
    np.testing.assert_array_equal(warm["iters"][:, 0], cold["iters"][:, 0])


def test_recorded_graph_follows_new_arguments():
    model = linear_models(2, 12, 6, 3, seed=48)
    rho0 = np.array([0.1, 1.0], dtype=np.float32)
    with gato.Solver(2, 12, 6, 3) as s:
        a = run(model, rho0, 3, params(), solver=s)
        b = run(model, rho0, 3, params(), solver=s)  # new buffers, same parameters
        c = run(model, rho0, 3, params(linsys=CR), solver=s)  # another linear solver
    ref = run(model, rho0, 3, params(linsys=CR))
    for k in a:
        assert np.array_equal(a[k], b[k], equal_nan=True), k
        assert np.array_equal(c[k], ref[k], equal_nan=True), k


def test_invalid_sqp_parameters_rejected():
    model = gato.to_device(linear_models(1, 4, 3, 2, seed=49))
    f = dict(device="cuda", dtype=torch.float32)
    X, U, lam = torch.zeros(1, 4, 3, **f), torch.zeros(1, 3, 2, **f), torch.zeros(1, 4, 3, **f)
    # the history holds the default iteration count's columns, so that the
    # library's own parameter checks are reached
    rho, hist = torch.ones(1, **f), torch.zeros(1, gato.default_sqp_params().iters + 1, **f)
    status = torch.zeros(1, device="cuda", dtype=torch.int32)
    with gato.Solver(1, 4, 3, 2) as s:
        for bad in (dict(iters=0), dict(rho_factor=1.0), dict(rho_min=-1.0),
                    dict(rho_min=2.0, rho_max=1.0)):
            with pytest.raises(gato.GatoError) as e:
                s.sqp_linear(params(), gato.default_sqp_params(**bad), model, X, U, lam, rho,
                             hist, status)
            assert e.value.code == gato.GATO_ERR_INVALID_ARG
