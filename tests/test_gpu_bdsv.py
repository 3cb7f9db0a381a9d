"""GPU parity of the direct solve of S lambda = gamma (bdsv): cyclic reduction
and chronological block Cholesky, against the fp64 oracle.

The oracle's reference is the same as for PCG: its direct fp64 solution
(Schur complement, block Cholesky, recovery by eq. (4)); the direct solve's
result is unique, so dX, dU, lambda and the merits are compared with the PCG
tolerances (dX and dU each 1e-4 relative L2 per solve, merits 1e-5 per value
as in test_gpu_parity).
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import oracle  # noqa: E402
from trajectory_optimization_kkt_gb300 import gato  # noqa: E402
from trajectory_optimization_kkt_gb300.workloads import WORKLOADS, make_batch, random_lq  # noqa: E402

from test_gpu_parity import TOL_DZ, check_solution, params_for, rel  # noqa: E402

CR, CHRONO = gato.GATO_LINSYS_BDSV, gato.GATO_LINSYS_BDSV_CHRONO


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()


def solve(prob, params, bdsv_kernel=gato.GATO_BDSV_KERNEL_AUTO):
    M, N, n = prob["Q"].shape[:3]
    m = prob["B"].shape[-1]
    d = gato.to_device(prob)
    with gato.Solver(M, N, n, m) as s:
        s.set_bdsv_kernel(bdsv_kernel)
        out = s.outputs(params.n_alpha)
        s.solve_kkt(params, d, out["dX"], out["dU"], out["lam"], out["iters"], out["merit"],
                    out["best"], out["status"])
        torch.cuda.synchronize()
        return {k: v.cpu().numpy() for k, v in out.items()}


def check_lambda(prob, out, solves, tol):
    for j in solves:
        lam = oracle.direct_solve(oracle.solve_one(prob, j))[2]
        assert rel(out["lam"][j], lam) <= tol, (j, rel(out["lam"][j], lam))


@pytest.mark.parametrize("order", [CR, CHRONO], ids=["cyclic", "chrono"])
@pytest.mark.parametrize("w", WORKLOADS, ids=lambda w: w.name)
def test_direct_solve_matches_oracle(w, order):
    M = min(w.M, 8)
    prob = make_batch(w, M=M)
    out = solve(prob, params_for(w, linsys=order))
    assert not out["status"].any(), out["status"]
    assert (out["iters"] == 0).all()
    check_solution(prob, out, range(M), w.n_alpha, w.beta, w.mu)
    check_lambda(prob, out, range(M), 10 * TOL_DZ)


@pytest.mark.parametrize("order", [CR, CHRONO], ids=["cyclic", "chrono"])
def test_refined_direct_solve_of_workload4(order):
    """The exact solve of the fp32-formed system leaves dX 2e-4 to 4e-4 from
    the exact solution (the formation's rounding); one refinement round, its
    correction solved with the same factors, brings every solve within 1e-4."""
    w = WORKLOADS[4]
    prob = make_batch(w, M=8)
    raw = solve(prob, params_for(w, linsys=order, refine_steps=0))
    assert not raw["status"].any()
    worst = max(rel(raw["dX"][j], oracle.direct_solve(oracle.solve_one(prob, j))[0])
                for j in range(8))
    assert TOL_DZ < worst < 6e-4, worst
    out = solve(prob, params_for(w, linsys=order, refine_steps=1))
    assert not out["status"].any()
    check_solution(prob, out, range(8), w.n_alpha, w.beta, w.mu)


# horizons 1, 2, 3 and every parity of the reduction (odd N, powers of two
# and one past them), state sizes on both kernels (n <= 16 registers, else
# shared memory), and the horizons of the GATO documentation's sweep
SIZES = [
    ("N1_n14_m7", 2, 1, 14, 7),
    ("N2_n7_m3", 3, 2, 7, 3),
    ("N3_n5_m2", 2, 3, 5, 2),
    ("N5_n14_m7", 2, 5, 14, 7),
    ("N8_n16_m8", 2, 8, 16, 8),
    ("N9_n1_m1", 2, 9, 1, 1),
    ("N17_n12_m6", 2, 17, 12, 6),
    ("N37_n13_m5", 3, 37, 13, 5),
    ("N64_n17_m4_smem", 2, 64, 17, 4),
    ("N20_n24_m8_smem", 2, 20, 24, 8),  # the substitution's rows unrolled to 24
    ("N11_n30_m10_smem", 2, 11, 30, 10),  # ... and to 36, predicated
    ("N33_n36_m12_smem", 2, 33, 36, 12),
    ("N6_n64_m8_smem", 1, 6, 64, 8),
    ("N129_n14_m7", 2, 129, 14, 7),
    ("N256_n14_m7", 2, 256, 14, 7),
    ("N512_n14_m7", 2, 512, 14, 7),
]


@pytest.mark.parametrize("order", [CR, CHRONO], ids=["cyclic", "chrono"])
@pytest.mark.parametrize("name,M,N,n,m", SIZES, ids=[c[0] for c in SIZES])
def test_direct_solve_sizes(name, M, N, n, m, order):
    prob = random_lq(M, N, n, m, seed=700 + N + n)
    out = solve(prob, gato.default_params(linsys=order, refine_steps=1))
    assert not out["status"].any(), out["status"]
    check_solution(prob, out, range(M))


REG_SIZES = [c for c in SIZES if c[0] in ("N5_n14_m7", "N8_n16_m8", "N37_n13_m5", "N129_n14_m7")]


@pytest.mark.parametrize("name,M,N,n,m", REG_SIZES, ids=[c[0] for c in REG_SIZES])
def test_register_and_shared_kernels_agree(name, M, N, n, m):
    prob = random_lq(M, N, n, m, seed=800 + N)
    p = gato.default_params(linsys=CR, refine_steps=1)
    a = solve(prob, p, gato.GATO_BDSV_KERNEL_AUTO)
    b = solve(prob, p, gato.GATO_BDSV_KERNEL_SHARED)
    for j in range(M):
        assert rel(a["lam"][j], b["lam"][j]) < 1e-4
    check_solution(prob, a, range(M), tol_dz=TOL_DZ)
    check_solution(prob, b, range(M), tol_dz=TOL_DZ)


def test_auto_policy_follows_the_horizon():
    """GATO_LINSYS_AUTO: PCG below bdsv_horizon (iterations counted), the
    direct solve from it (no iterations)."""
    prob = random_lq(2, 40, 14, 7, seed=901)
    below = solve(prob, gato.default_params(bdsv_horizon=41, pcg_max_iters=2000,
                                            refine_steps=1))
    at = solve(prob, gato.default_params(bdsv_horizon=40, refine_steps=1))
    assert (below["iters"] > 0).all() and (at["iters"] == 0).all()
    for out in (below, at):
        assert not out["status"].any()
        check_solution(prob, out, range(2))


def test_separate_entry_point_equals_solve_kkt():
    w = WORKLOADS[2]
    prob = make_batch(w, M=3)
    for order in (CR, CHRONO):
        p = params_for(w, linsys=order, refine_steps=0)
        full = solve(prob, p)
        d = gato.to_device(prob)
        with gato.Solver(3, w.N, w.n, w.m) as s:
            o = s.outputs(p.n_alpha)
            s.form_schur(d, o["status"])
            s.bdsv_solve(p, o["lam"], o["dX"], o["dU"], o["iters"], o["status"])
            s.linesearch(p, d, o["dX"], o["dU"], o["merit"], o["best"], o["status"])
            torch.cuda.synchronize()
            for k in ("dX", "dU", "lam", "merit", "best", "iters", "status"):
                assert np.array_equal(o[k].cpu().numpy(), full[k]), (order, k)


def test_deterministic_and_batch_position_invariant():
    w = WORKLOADS[4]
    prob = make_batch(w, M=5)
    p = params_for(w, linsys=CR)
    a = solve(prob, p)
    b = solve(prob, p)
    for k in a:
        assert np.array_equal(a[k], b[k]), k
    one = solve({k: v[2:3] for k, v in prob.items()}, p)
    for k in ("dX", "dU", "lam", "merit", "best"):
        assert np.array_equal(one[k][0], a[k][2]), k


def test_pcg_refinement_and_direct_solve_agree():
    w = WORKLOADS[1]
    prob = make_batch(w, M=4)
    a = solve(prob, params_for(w, linsys=gato.GATO_LINSYS_PCG, refine_steps=2, refine_eps=0.01))
    b = solve(prob, params_for(w, linsys=CR, refine_steps=2))
    for j in range(4):
        assert rel(a["lam"][j], b["lam"][j]) < 1e-5


@pytest.mark.parametrize("order", [CR, CHRONO], ids=["cyclic", "chrono"])
def test_indefinite_Q_and_nan_are_flagged(order):
    w = WORKLOADS[0]
    prob = make_batch(w, M=3)
    prob["Q"] = prob["Q"].copy()
    prob["Q"][1, 3] = -np.eye(w.n, dtype=np.float32)
    prob["q"] = prob["q"].copy()
    prob["q"][2, 2, 1] = np.nan
    out = solve(prob, params_for(w, linsys=order))
    assert out["status"][1] & gato.GATO_STATUS_NONPOSITIVE_PIVOT
    assert out["status"][2] & gato.GATO_STATUS_NONFINITE
    assert out["status"][0] == 0
    check_solution(prob, out, [0], w.n_alpha, w.beta, w.mu)


def test_invalid_linear_solver_parameters_rejected():
    w = WORKLOADS[0]
    prob = make_batch(w, M=1)
    for bad in (dict(linsys=4), dict(linsys=-1), dict(bdsv_horizon=0)):
        with pytest.raises(gato.GatoError) as e:
            solve(prob, params_for(w, **bad))
        assert e.value.code == gato.GATO_ERR_INVALID_ARG
    d = gato.to_device(prob)
    with gato.Solver(1, w.N, w.n, w.m) as s:
        o = s.outputs()
        s.form_schur(d, o["status"])
        with pytest.raises(gato.GatoError):
            s.bdsv_solve(params_for(w, linsys=gato.GATO_LINSYS_PCG), o["lam"], o["dX"], o["dU"],
                         o["iters"], o["status"])
        with pytest.raises(gato.GatoError):
            s.set_bdsv_kernel(7)
