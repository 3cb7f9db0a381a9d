"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Tolerances
  dX, dU      relative L2 error of dX and, separately, of dU per solve <= 1e-4
              against the oracle's direct fp64 solution, PCG stopped at
              eps = 1e-6; every solve of every workload at its full batch
  merit       per value: |merit_gpu - merit_oracle| <= 1e-5 max(|merit_oracle|,
              1e-2 max|merit| of the solve), the oracle evaluating the GPU's own
              dz.  A merit 100 times below the solve's largest one is a sum
              whose terms cancelled by more than 100x; its fp32 rounding error
              scales with the terms, not with the value, so the value's
              magnitude is floored at 1 % of the solve's scale
  best        identical, unless the oracle's two best candidates are within
              1e-5 |M_best| of each other (then either of the two)
  S, Phi, gamma  relative Frobenius error per solve <= 1e-5 (fp32 formation:
              about 20 n u with u = 2^-24 for the sizes here)
  status      0 on every solve of the workloads: workloads 0 and 2 meet their
              stated iteration caps (200, 500) with the double-float PCG
The workloads use their own refinement setting (one PCG correction solved to
0.25 for workload 0 and to 0.1 for workload 4; one correction by substitution
with a direct factorisation of the same S for workloads 1 and 2, two for
workload 3): fp32 formation alone moves dX by 2e-4 to 1e-2, and refinement
brings the worst dX of each workload's batch to 1e-7 .. 5e-5.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import oracle  # noqa: E402
from trajectory_optimization_kkt_gb300 import gato  # noqa: E402
from trajectory_optimization_kkt_gb300.workloads import WORKLOADS, make_batch, random_lq  # noqa: E402

TOL_DZ = 1e-4
TOL_MERIT = 1e-5
MERIT_NEAR_ZERO = 1e-2
TOL_FORM = 1e-5


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()


def rel(a, b):
    a, b = np.ravel(a), np.ravel(b)
    return np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300)


def params_for(w, **kw):
    return gato.default_params(**{**w.solver_settings(), **kw})


def solve(prob, params, kernel=gato.GATO_PCG_AUTO, form_kind=gato.GATO_FORM_AUTO):
    M, N, n = prob["Q"].shape[:3]
    m = prob["B"].shape[-1]
    d = gato.to_device(prob)
    with gato.Solver(M, N, n, m) as s:
        s.set_pcg_kernel(kernel)
        s.set_form_kernel(form_kind)
        out = s.outputs(params.n_alpha)
        s.solve_kkt(params, d, out["dX"], out["dU"], out["lam"], out["iters"], out["merit"],
                    out["best"], out["status"])
        torch.cuda.synchronize()
        return {k: v.cpu().numpy() for k, v in out.items()}


def dz_errors(prob, out, j):
    """Relative L2 errors of dX and dU (0 when there is no control) of solve j
    against the oracle's direct fp64 solution."""
    dX, dU, _ = oracle.direct_solve(oracle.solve_one(prob, j))
    ex = rel(out["dX"][j], dX)
    eu = rel(out["dU"][j], dU) if dU.size else 0.0
    return ex, eu


def check_solution(prob, out, solves, n_alpha=8, beta=2.0, mu=10.0, tol_dz=TOL_DZ):
    for j in solves:
        ex, eu = dz_errors(prob, out, j)
        assert ex <= tol_dz and eu <= tol_dz, (j, ex, eu)
        pj = oracle.solve_one(prob, j)
        check_merit(pj, out["dX"][j], out["dU"][j], out["merit"][j], out["best"][j],
                    n_alpha, beta, mu)


def check_merit(pj, dX, dU, merit, best, n_alpha, beta, mu):
    ref, ref_best = oracle.linesearch(pj, dX, dU, n_alpha, beta, mu)
    floor = MERIT_NEAR_ZERO * np.abs(ref).max()
    tol = TOL_MERIT * np.maximum(np.abs(ref), floor)
    assert (np.abs(merit - ref) <= tol).all(), (merit, ref)
    cand = ref[1:]
    order = np.argsort(cand, kind="stable")
    gap = cand[order[1]] - cand[order[0]] if len(cand) > 1 else np.inf
    if ref_best >= 0 and gap > TOL_MERIT * abs(cand[order[0]]):
        assert int(best) == ref_best
    elif ref_best >= 0:
        assert int(best) in (int(order[0]), int(order[1]))


# --------------------------------------------------------------------------
# formation (a1, a2)
# --------------------------------------------------------------------------

def form(prob, kind=gato.GATO_FORM_AUTO):
    M, N, n = prob["Q"].shape[:3]
    m = prob["B"].shape[-1]
    d = gato.to_device(prob)
    f = dict(device="cuda", dtype=torch.float32)
    out = dict(D=torch.empty(M, N, n, n, **f), O=torch.empty(M, max(N - 1, 0), n, n, **f),
               g=torch.empty(M, N, n, **f), Pd=torch.empty(M, N, n, n, **f),
               Po=torch.empty(M, max(N - 1, 0), n, n, **f))
    status = torch.zeros(M, dtype=torch.int32, device="cuda")
    with gato.Solver(M, N, n, m) as s:
        s.set_form_kernel(kind)
        s.form_schur(d, status)
        s.get_schur(out["D"], out["O"] if N > 1 else None, out["g"], out["Pd"],
                    out["Po"] if N > 1 else None)
        torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in out.items()}, status.cpu().numpy()


FORM_CASES = [(w.name, make_batch(w, M=min(w.M, 6))) for w in WORKLOADS] + [
    ("ragged_N37_n13_m5", random_lq(3, 37, 13, 5, seed=501)),
    ("N1_n14", random_lq(2, 1, 14, 7, seed=502)),
    ("n3_m2", random_lq(2, 11, 3, 2, seed=503)),
    ("n64_m64", random_lq(1, 4, 64, 64, seed=504)),
    # register-row widths: controls wider than 8 (PM = 16) and every state width
    ("n9_m12", random_lq(2, 9, 9, 12, seed=505)),
    ("n16_m16", random_lq(2, 6, 16, 16, seed=506)),
    ("n11_m9", random_lq(2, 13, 11, 9, seed=507)),
]


@pytest.mark.parametrize("kind", [gato.GATO_FORM_AUTO, gato.GATO_FORM_SHARED])
@pytest.mark.parametrize("name,prob", FORM_CASES, ids=[c[0] for c in FORM_CASES])
def test_form_schur_matches_oracle(name, prob, kind):
    got, status = form(prob, kind)
    assert not status.any()
    N = prob["Q"].shape[1]
    for j in range(prob["Q"].shape[0]):
        D, O, g, rc = oracle.schur(oracle.solve_one(prob, j))
        Pd, Po, rc2 = oracle.stair(D, O)
        assert rc == 0 and rc2 == 0
        refs = dict(D=D, g=g, Pd=Pd)
        if N > 1:
            refs.update(O=O, Po=Po)
        for k, ref in refs.items():
            assert rel(got[k][j], ref) <= TOL_FORM, (name, j, k, rel(got[k][j], ref))


# --------------------------------------------------------------------------
# whole path (a1..a6) on the five workloads (subsets) and ragged sizes
# --------------------------------------------------------------------------

@pytest.mark.parametrize("w", WORKLOADS, ids=lambda w: w.name)
def test_solve_kkt_matches_oracle(w):
    M = min(w.M, 8)
    prob = make_batch(w, M=M)
    out = solve(prob, params_for(w))
    assert not out["status"].any(), out["status"]
    check_solution(prob, out, range(M), w.n_alpha, w.beta, w.mu)


@pytest.mark.parametrize("w", WORKLOADS, ids=lambda w: w.name)
def test_full_batch_in_the_benchmark_configuration(w):
    """Each workload at its full batch with the default kernels and parts (as
    bench.py times it): every solve ends with status 0 (workloads 0 and 2
    within their stated caps of 200 and 500 iterations per PCG solve) and
    every solve matches the oracle (dX, dU, merits, best)."""
    prob = make_batch(w)
    out = solve(prob, params_for(w))
    assert not out["status"].any(), np.nonzero(out["status"])
    check_solution(prob, out, range(w.M), w.n_alpha, w.beta, w.mu)
    assert (out["best"] >= 0).all()


@pytest.mark.parametrize("w", [WORKLOADS[1], WORKLOADS[4]], ids=lambda w: w.name)
def test_refinement_removes_the_fp32_formation_error(w):
    """Without refinement the fp32 formation of S (inverses and products
    rounded to fp32) leaves dX 2e-4 to 4e-4 from the exact solution; one
    correction round brings every solve within the 1e-4 tolerance."""
    M = 16
    prob = make_batch(w, M=M)
    raw = solve(prob, params_for(w, refine_steps=0))
    refined = solve(prob, params_for(w))
    assert not raw["status"].any() and not refined["status"].any()
    worst_raw = max(dz_errors(prob, raw, j)[0] for j in range(M))
    assert TOL_DZ < worst_raw < 6e-4, worst_raw
    check_solution(prob, refined, range(M), w.n_alpha, w.beta, w.mu)


CUSTOM = [
    ("ragged_N37_n13_m5", 3, 37, 13, 5, 1),
    ("N1_n14_m7", 2, 1, 14, 7, 0),
    ("N2_n7_m3", 3, 2, 7, 3, 0),
    ("N9_n16_m8", 2, 9, 16, 8, 1),
    ("N11_n3_m2_generic", 2, 11, 3, 2, 1),
    ("N6_n40_m12_generic", 2, 6, 40, 12, 1),
    ("N130_n14_m7_generic", 1, 130, 14, 7, 1),
    ("N128_n12_m6_tile", 2, 128, 12, 6, 1),
    ("N4_n64_m64_generic", 1, 4, 64, 64, 1),  # the largest state and control sizes
    ("N9_n9_m12", 2, 9, 9, 12, 1),  # controls wider than the state
    ("N7_n16_m16", 2, 7, 16, 16, 1),
]
WIDE = [c for c in CUSTOM if 7 <= c[3] <= 16 and c[2] <= 128] + [
    ("N33_n15_m4", 2, 33, 15, 4, 1), ("N5_n8_m3", 3, 5, 8, 3, 2)]


TILED_KINDS = [gato.GATO_PCG_WIDE, gato.GATO_PCG_TILE, gato.GATO_PCG_QUAD]
TILED_IDS = ["wide", "tile", "quad"]


@pytest.mark.parametrize("kind", TILED_KINDS, ids=TILED_IDS)
@pytest.mark.parametrize("name,M,N,n,m,refine", WIDE, ids=[c[0] for c in WIDE])
def test_tiled_kernels_custom_sizes(name, M, N, n, m, refine, kind):
    prob = random_lq(M, N, n, m, seed=600 + N + n)
    p = gato.default_params(pcg_max_iters=3000, refine_steps=refine)
    out = solve(prob, p, kind)
    assert not out["status"].any(), out["status"]
    check_solution(prob, out, range(M))


# the quad kernel's remaining row counts (n = 10, 11: three rows per lane,
# ragged last lanes), its largest block (N = 128: 512 threads), and more
# solves than resident blocks (each block takes several from the queue)
QUAD = [("N21_n10_m4", 3, 21, 10, 4, 1), ("N17_n11_m5", 3, 17, 11, 5, 1),
        ("N128_n14_m7_max", 2, 128, 14, 7, 1), ("N120_n16_m8", 2, 120, 16, 8, 1),
        ("N8_n14_m7_M400", 400, 8, 14, 7, 1)]


@pytest.mark.parametrize("name,M,N,n,m,refine", QUAD, ids=[c[0] for c in QUAD])
def test_quad_kernel_sizes(name, M, N, n, m, refine):
    prob = random_lq(M, N, n, m, seed=700 + N + n)
    p = gato.default_params(pcg_max_iters=3000, refine_steps=refine)
    out = solve(prob, p, gato.GATO_PCG_QUAD)
    assert not out["status"].any(), out["status"]
    check = range(M) if M <= 8 else [0, 1, M // 2, M - 2, M - 1]
    check_solution(prob, out, check)
    # the wide kernel runs the same iteration in another summation order; in
    # fp32 the iteration at which the residual crosses eps moves with the
    # rounding, by a few percent on the average and up to about 10 % on the
    # rare solve of a large batch
    ref = solve(prob, p, gato.GATO_PCG_WIDE)
    diff = np.abs(out["iters"] - ref["iters"])
    assert diff.mean() <= 0.02 * ref["iters"].mean() + 1
    assert diff.max() <= 0.1 * ref["iters"].max() + 2


@pytest.mark.parametrize("rule", [gato.GATO_STOP_RESIDUAL, gato.GATO_STOP_PRECOND,
                                  gato.GATO_STOP_SCALED], ids=["residual", "precond", "scaled"])
def test_quad_kernel_stopping_rules(rule):
    """Each stopping rule stops the quad kernel where it stops the wide
    kernel (the same iteration in another summation order), with lambda as
    close to the fp64 direct solution (workload 4's sizes, unrefined)."""
    w = WORKLOADS[4]
    prob = make_batch(w, M=3)
    p = params_for(w, stop_rule=rule, refine_steps=0)
    a = solve(prob, p, gato.GATO_PCG_QUAD)
    b = solve(prob, p, gato.GATO_PCG_WIDE)
    assert not a["status"].any() and not b["status"].any()
    for j in range(3):
        lam = oracle.direct_solve(oracle.solve_one(prob, j))[2]
        assert rel(a["lam"][j], lam) <= 2 * rel(b["lam"][j], lam) + 1e-5
    assert np.abs(a["iters"] - b["iters"]).max() <= 0.05 * b["iters"].max() + 2


def test_a_short_input_array_is_rejected_before_launch():
    prob = random_lq(4, 8, 14, 7, seed=790)
    d = gato.to_device(prob)
    d["A"] = d["A"][:3].contiguous()  # three solves of A for a batch of four
    p = gato.default_params(pcg_max_iters=500)
    with gato.Solver(4, 8, 14, 7) as s:
        out = s.outputs(p.n_alpha)
        with pytest.raises(ValueError, match="A holds"):
            s.solve_kkt(p, d, out["dX"], out["dU"], out["lam"], out["iters"], out["merit"],
                        out["best"], out["status"])


def test_kernel_choice_between_sizes_keeps_launches_valid():
    """The automatic choice queries the wide kernel's occupancy at each call's
    sizes; a later launch of that kernel at other sizes (its shared memory
    under the 48 KB default, above the size queried) still launches."""
    p = gato.default_params(pcg_max_iters=3000, refine_steps=0)
    small = random_lq(16, 16, 12, 6, seed=791)
    mid = random_lq(2, 32, 12, 6, seed=792)
    assert ran_kernels(small, p)[0] == gato.GATO_PCG_QUAD
    assert ran_kernels(mid, p, gato.GATO_PCG_WIDE)[0] == gato.GATO_PCG_WIDE
    out = solve(mid, gato.default_params(pcg_max_iters=3000, refine_steps=1), gato.GATO_PCG_WIDE)
    assert not out["status"].any()
    check_solution(mid, out, range(2))


def ran_kernels(prob, p, kernel=gato.GATO_PCG_AUTO, parts=0):
    """gato_stats.pcg_kernel and refine_kernel after one gato_solve_kkt."""
    M, N, n = prob["Q"].shape[:3]
    m = prob["B"].shape[-1]
    d = gato.to_device(prob)
    with gato.Solver(M, N, n, m) as s:
        s.set_pcg_kernel(kernel)
        s.set_parts(parts)
        out = s.outputs(p.n_alpha)
        s.solve_kkt(p, d, out["dX"], out["dU"], out["lam"], out["iters"], out["merit"],
                    out["best"], out["status"])
        torch.cuda.synchronize()
        st = s.get_stats()
        assert not out["status"].cpu().numpy().any()
        return st.pcg_kernel, st.refine_kernel


Q, W, C, FF = gato.GATO_PCG_QUAD, gato.GATO_PCG_WIDE, gato.GATO_PCG_CLUSTER, \
    gato.GATO_PCG_DOUBLE_FLOAT
# (name, M, N, n, m, settings, expected main kernel, expected correction kernel);
# the wide kernel's working warps per SM are 2N/32 per solve times the solves
# an SM holds (the whole batch's, by the SM count, at most its occupancy)
AUTO_CHOICE = [
    ("M16_N32_n12_quad", 16, 32, 12, 6, {}, Q, Q),        # 2 warps per SM
    ("M16_N64_n14_quad", 16, 64, 14, 7, {}, Q, Q),        # 4
    ("M16_N96_n14_wide", 16, 96, 14, 7, {}, W, W),        # 6
    ("M256_N128_n14_wide", 256, 128, 14, 7, {}, W, W),    # 8, in four parts
    ("M256_N128_n12_quad", 256, 128, 12, 6, {}, Q, Q),    # n = 12: the quad kernel
    # four parts of 80: one part alone would leave 2 warps per SM, the whole
    # batch (3 solves per SM) leaves 6
    ("M320_N32_n14_parts", 320, 32, 14, 7, {}, W, W),
    ("M2_N200_n14_cluster", 2, 200, 14, 7, {}, C, C),
    ("M2_N16_n36_rows", 2, 16, 36, 12, {}, gato.GATO_PCG_ROWS, gato.GATO_PCG_ROWS),
    ("M2_N16_n14_ff", 2, 16, 14, 7, {"pcg_precision": 1, "refine_eps": 0.25}, FF, Q),
    ("M2_N32_n12_direct_corr", 2, 32, 12, 6, {"refine_solver": 1}, Q, 0),
    ("M2_N16_n14_no_refine", 2, 16, 14, 7, {"refine_steps": 0}, Q, 0),
]


@pytest.mark.parametrize("name,M,N,n,m,kw,main,corr", AUTO_CHOICE,
                         ids=[c[0] for c in AUTO_CHOICE])
def test_automatic_kernel_choice_is_reported(name, M, N, n, m, kw, main, corr):
    if M > 16 and torch.cuda.get_device_properties(0).multi_processor_count < 128:
        pytest.skip("the expected choice assumes at least 128 SMs")
    prob = random_lq(M, N, n, m, seed=760 + N + n)
    p = gato.default_params(pcg_max_iters=3000, **{"refine_steps": 1, **kw})
    assert ran_kernels(prob, p) == (main, corr)


def test_chosen_kernels_are_reported():
    prob = random_lq(2, 16, 14, 7, seed=771)
    p = gato.default_params(pcg_max_iters=3000, refine_steps=1)
    for kind in (gato.GATO_PCG_GENERIC, gato.GATO_PCG_WIDE, gato.GATO_PCG_TILE,
                 gato.GATO_PCG_QUAD, gato.GATO_PCG_ROWS):
        assert ran_kernels(prob, p, kind) == (kind, kind)
    # a direct solve runs no PCG kernel
    assert ran_kernels(prob, gato.default_params(linsys=gato.GATO_LINSYS_BDSV)) == (0, 0)


@pytest.mark.parametrize("name,M,N,n,m,refine", CUSTOM, ids=[c[0] for c in CUSTOM])
def test_solve_kkt_custom_sizes(name, M, N, n, m, refine):
    prob = random_lq(M, N, n, m, seed=600 + N + n)
    p = gato.default_params(pcg_max_iters=3000, refine_steps=refine)
    out = solve(prob, p)
    assert not out["status"].any(), out["status"]
    check_solution(prob, out, range(M))


# horizons beyond 128 knots: the solve split over a cluster of 2 (N <= 256) or
# 4 (N <= 512) CTAs, ragged splits included
CLUSTER = [
    ("N129_n7_m3_c2", 2, 129, 7, 3),
    ("N200_n13_m5_c2", 2, 200, 13, 5),
    ("N256_n14_m7_c2", 2, 256, 14, 7),
    ("N300_n16_m8_c4", 2, 300, 16, 8),
    ("N512_n14_m7_c4", 1, 512, 14, 7),
]


@pytest.mark.parametrize("name,M,N,n,m", CLUSTER, ids=[c[0] for c in CLUSTER])
def test_cluster_kernel_long_horizons(name, M, N, n, m):
    prob = random_lq(M, N, n, m, seed=650 + N + n)
    p = gato.default_params(pcg_max_iters=4000, refine_steps=1)
    out = solve(prob, p)
    assert not out["status"].any(), out["status"]
    check_solution(prob, out, range(M))
    ref = solve(prob, p, gato.GATO_PCG_GENERIC)
    assert np.abs(out["iters"] - ref["iters"]).max() <= 0.05 * ref["iters"].max() + 2
    for j in range(M):
        assert rel(out["lam"][j], ref["lam"][j]) < 1e-3


# the register-row kernel (16 < n <= 64, and any n when chosen): every row
# width instantiation, ragged rows per thread, N = 1, and a block too large
# for it (the default then takes the generic kernel)
ROWS = [
    ("n17_m5", 3, 9, 17, 5), ("n20_m20", 2, 10, 20, 20), ("n24_m8", 2, 12, 24, 8),
    ("n27_m9", 2, 11, 27, 9), ("n32_m4", 2, 8, 32, 4), ("n36_m12", 2, 16, 36, 12),
    ("n40_m10", 1, 6, 40, 10), ("n45_m7", 1, 5, 45, 7), ("n53_m3", 1, 4, 53, 3),
    ("n64_m16", 1, 4, 64, 16), ("N1_n36", 2, 1, 36, 12),
    # the largest blocks the register budget allows, and one knot past them
    # (the cluster form: a solve's knots over 2, 4 or 8 CTAs)
    ("n36_N18_max", 1, 18, 36, 12), ("n36_N19_cluster2", 1, 19, 36, 12),
    ("n24_N42_max", 1, 42, 24, 8), ("n64_N5_max", 1, 5, 64, 8),
    ("n36_N40_cluster4", 1, 40, 36, 12), ("n36_N32_cluster2", 2, 32, 36, 12),
    ("n36_N37_cluster4_ragged", 2, 37, 36, 12), ("n24_N64_cluster2", 2, 64, 24, 8),
    ("n17_N100_cluster2", 1, 100, 17, 5), ("n64_N12_cluster4", 1, 12, 64, 8),
    ("n36_N128_cluster8", 1, 128, 36, 12),
    # one row per thread (n > 48): CTAs of 10 to 11 warps, whose pushed block
    # sums take more than eight slots per CTA
    ("n64_N10_cluster2_10warps", 1, 10, 64, 8), ("n56_N24_cluster4_11warps", 1, 24, 56, 8),
    ("n64_N40_cluster8_10warps", 1, 40, 64, 8),
]


@pytest.mark.parametrize("name,M,N,n,m", ROWS, ids=[c[0] for c in ROWS])
def test_rows_kernel_matches_oracle_and_generic(name, M, N, n, m):
    prob = random_lq(M, N, n, m, seed=800 + N + n)
    p = gato.default_params(pcg_max_iters=5000, refine_steps=1)
    out = solve(prob, p)
    assert not out["status"].any(), out["status"]
    check_solution(prob, out, range(M))
    ref = solve(prob, p, gato.GATO_PCG_GENERIC)
    assert np.abs(out["iters"] - ref["iters"]).max() <= 0.05 * ref["iters"].max() + 2
    for j in range(M):
        assert rel(out["lam"][j], ref["lam"][j]) < 1e-3


@pytest.mark.parametrize("rule", [gato.GATO_STOP_RESIDUAL, gato.GATO_STOP_PRECOND,
                                  gato.GATO_STOP_SCALED], ids=["residual", "precond", "scaled"])
def test_rows_kernel_stopping_rules(rule):
    """Each stopping rule stops the row kernel with a lambda as close to the
    fp64 direct solution as the generic kernel's, at about the same iteration
    (workload 3's sizes, unrefined).  The workload is ill-conditioned (1300
    to 1700 iterations): near fp32's attainable accuracy the iteration at
    which the recursive residual crosses eps depends on rounding, and the two
    kernels, which sum in different orders, differ by up to 12% there and
    move lambda by about 1e-3; hence 15% here against 5% on the well
    conditioned sizes."""
    w = WORKLOADS[3]
    prob = make_batch(w, M=3)
    p = params_for(w, stop_rule=rule, refine_steps=0)
    a = solve(prob, p, gato.GATO_PCG_ROWS)
    b = solve(prob, p, gato.GATO_PCG_GENERIC)
    assert not a["status"].any() and not b["status"].any()
    for j in range(3):
        lam = oracle.direct_solve(oracle.solve_one(prob, j))[2]
        assert rel(a["lam"][j], lam) <= 2 * rel(b["lam"][j], lam) + 1e-5
    assert np.abs(a["iters"] - b["iters"]).max() <= 0.15 * b["iters"].max() + 2


@pytest.mark.parametrize("rule", [gato.GATO_STOP_RESIDUAL, gato.GATO_STOP_PRECOND,
                                  gato.GATO_STOP_SCALED], ids=["residual", "precond", "scaled"])
def test_rows_cluster_form_stopping_rules_and_warm_start(rule):
    """The cluster form (n = 36, N = 32: two CTAs of 16 knots) under each
    stopping rule, against the oracle and the generic kernel, and warm-started
    from half the solution."""
    prob = random_lq(2, 32, 36, 12, seed=831)
    p = gato.default_params(pcg_max_iters=5000, refine_steps=1, stop_rule=rule)
    out = solve(prob, p)
    ref = solve(prob, p, gato.GATO_PCG_GENERIC)
    assert not out["status"].any() and not ref["status"].any()
    check_solution(prob, out, range(2))
    assert np.abs(out["iters"] - ref["iters"]).max() <= 0.05 * ref["iters"].max() + 2
    lam = np.stack([oracle.direct_solve(oracle.solve_one(prob, j))[2] for j in range(2)])
    d = gato.to_device(prob)
    with gato.Solver(2, 32, 36, 12) as s:
        o = s.outputs(p.n_alpha)
        s.form_schur(d, o["status"])
        q = gato.default_params(pcg_max_iters=5000, stop_rule=rule)
        s.pcg_solve(q, o["lam"], o["dX"], o["dU"], o["iters"], o["status"])
        cold = o["iters"].cpu().numpy().copy()
        s.pcg_solve(q, o["lam"], o["dX"], o["dU"], o["iters"], o["status"],
                    lambda0=torch.tensor(0.5 * lam, dtype=torch.float32, device="cuda"))
        torch.cuda.synchronize()
        assert not o["status"].cpu().numpy().any()
        assert (o["iters"].cpu().numpy() <= cold).all()
        assert s.get_stats().pcg_kernel == gato.GATO_PCG_ROWS


def test_rows_kernel_chosen_for_small_states():
    """GATO_PCG_ROWS also runs n <= 16 (the narrowest row width)."""
    w = WORKLOADS[1]
    prob = make_batch(w, M=4)
    out = solve(prob, params_for(w), gato.GATO_PCG_ROWS)
    assert not out["status"].any()
    check_solution(prob, out, range(4), w.n_alpha, w.beta, w.mu)


@pytest.mark.parametrize("kind", TILED_KINDS, ids=TILED_IDS)
@pytest.mark.parametrize("w", [WORKLOADS[1], WORKLOADS[4]], ids=lambda w: w.name)
def test_tiled_and_generic_kernels_agree(w, kind):
    prob = make_batch(w, M=4)
    a = solve(prob, params_for(w), kind)
    b = solve(prob, params_for(w), gato.GATO_PCG_GENERIC)
    assert np.abs(a["iters"] - b["iters"]).max() <= 0.05 * b["iters"].max() + 2
    for j in range(4):
        assert rel(a["dX"][j], b["dX"][j]) < 1e-3
    check_solution(prob, b, range(4), w.n_alpha, w.beta, w.mu)


@pytest.mark.parametrize("w", [WORKLOADS[0], WORKLOADS[2]], ids=lambda w: w.name)
def test_shared_memory_formation_path_solves(w):
    prob = make_batch(w, M=4)
    a = solve(prob, params_for(w), form_kind=gato.GATO_FORM_SHARED)
    b = solve(prob, params_for(w), form_kind=gato.GATO_FORM_AUTO)
    check_solution(prob, a, range(4), w.n_alpha, w.beta, w.mu)
    check_solution(prob, b, range(4), w.n_alpha, w.beta, w.mu)


@pytest.mark.parametrize("rule", [gato.GATO_STOP_PRECOND, gato.GATO_STOP_SCALED])
def test_other_stop_rules(rule):
    w = WORKLOADS[1]
    prob = make_batch(w, M=3)
    out = solve(prob, params_for(w, stop_rule=rule, refine_steps=1))
    assert not out["status"].any()
    check_solution(prob, out, range(3), w.n_alpha, w.beta, w.mu)
    for j in range(3):
        D, O, g, _ = oracle.schur(oracle.solve_one(prob, j))
        Pd, Po, _ = oracle.stair(D, O)
        _, it, ok = oracle.pcg(D, O, Pd, Po, g, w.pcg_eps, 5000, stop_rule=rule)
        # the same stopping quantity: fp32 iterations of the first solve track
        # the fp64 count (the refinement adds a short second solve)
        assert ok and it * 0.9 - 3 <= int(out["iters"][j]) <= it * 1.2 + 150


# --------------------------------------------------------------------------
# refinement corrections by substitution (GATO_REFINE_SOLVER_DIRECT)
# --------------------------------------------------------------------------

@pytest.mark.parametrize("wi,M,steps", [(1, 16, 1), (3, 16, 2), (4, 8, 1)],
                         ids=["M16_N32_n12", "M16_N16_n36", "M8_N128_n14"])
def test_direct_refinement_after_pcg(wi, M, steps):
    """The main solve is PCG; the corrections are solved with the cyclic-
    reduction factorisation of the same S, formed once: every solve matches
    the oracle, and iters counts the main solve's PCG iterations only (those
    of the unrefined call)."""
    w = WORKLOADS[wi]
    prob = make_batch(w, M=M)
    out = solve(prob, params_for(w, refine_solver=gato.GATO_REFINE_SOLVER_DIRECT,
                                 refine_steps=steps))
    assert not out["status"].any(), out["status"]
    check_solution(prob, out, range(M), w.n_alpha, w.beta, w.mu)
    raw = solve(prob, params_for(w, refine_steps=0))
    np.testing.assert_array_equal(out["iters"], raw["iters"])


# --------------------------------------------------------------------------
# the double-float PCG (GATO_PCG_PRECISION_FF)
# --------------------------------------------------------------------------

FF = gato.GATO_PCG_PRECISION_FF


def pcg_only(prob, p, lambda0=None):
    """gato_form_schur + gato_pcg_solve; also returns the S and gamma the GPU
    formed (exported) for a true-residual check."""
    M, N, n = prob["Q"].shape[:3]
    m = prob["B"].shape[-1]
    d = gato.to_device(prob)
    f = dict(device="cuda", dtype=torch.float32)
    with gato.Solver(M, N, n, m) as s:
        o = s.outputs(p.n_alpha)
        s.form_schur(d, o["status"])
        l0 = None if lambda0 is None else torch.tensor(lambda0, **f)
        s.pcg_solve(p, o["lam"], o["dX"], o["dU"], o["iters"], o["status"], lambda0=l0)
        D, g = torch.empty(M, N, n, n, **f), torch.empty(M, N, n, **f)
        O = torch.empty(M, N - 1, n, n, **f) if N > 1 else None
        s.get_schur(D, O, g)
        torch.cuda.synchronize()
        out = {k: v.cpu().numpy() for k, v in o.items()}
        out.update(D=D.cpu().numpy(), O=None if O is None else O.cpu().numpy(), g=g.cpu().numpy())
        return out


def true_relative_residual(out, j):
    """||gamma - S lambda|| / ||gamma|| of the returned lambda on the S and
    gamma the GPU formed (fp64), and the same for the exact solution of that
    system rounded to fp32: the floor that an fp32 lambda can reach."""
    N, n = out["g"].shape[1:]
    O = out["O"][j] if out["O"] is not None else np.zeros((0, n, n))
    S = oracle.bt_dense(out["D"][j], O)
    g = out["g"][j].astype(np.float64).ravel()
    exact = np.linalg.solve(S, g).astype(np.float32).astype(np.float64)
    res = lambda lam: np.linalg.norm(g - S @ lam) / np.linalg.norm(g)
    return res(out["lam"][j].astype(np.float64).ravel()), res(exact)


@pytest.mark.parametrize("w", [WORKLOADS[0], WORKLOADS[2]], ids=lambda w: w.name)
def test_double_float_pcg_meets_the_stated_cap(w):
    """Workloads 0 and 2 state caps of 200 and 500 iterations.  The double-
    float main solve stops on ||gamma - S lambda|| <= eps ||gamma|| within
    them on every solve, and its iteration count follows the fp64 oracle's
    (which needs up to 185 and 490) within 3 %.  The true residual of the
    returned lambda on the exported S and gamma stays within the fp32
    kernels' bound of 10 eps: it also carries the rounding of lambda to fp32
    and the fp32 formation's mismatch between the scaled blocks the solve
    uses and the exported S (measured 1.8e-6 and at most 2.7e-6 here)."""
    prob = make_batch(w)
    out = pcg_only(prob, params_for(w, refine_steps=0))
    assert not out["status"].any(), np.nonzero(out["status"])
    assert out["iters"].max() <= w.pcg_max_iters
    for j in range(w.M):
        res, floor = true_relative_residual(out, j)
        assert res <= 10 * w.pcg_eps, (j, res, floor)
        D, O, gam, _ = oracle.schur(oracle.solve_one(prob, j))
        Pd, Po, _ = oracle.stair(D, O)
        _, it, ok = oracle.pcg(D, O, Pd, Po, gam, w.pcg_eps, 5000, stop_rule=0)
        assert ok and it * 0.95 - 3 <= out["iters"][j] <= it * 1.03 + 3, (j, it, out["iters"][j])


FF_SIZES = [
    ("N1_n14_m7", 2, 1, 14, 7),
    ("N2_n3_m2", 2, 2, 3, 2),
    ("N37_n13_m5", 2, 37, 13, 5),
    ("N16_n36_m12", 2, 16, 36, 12),
    ("N4_n64_m16", 1, 4, 64, 16),
    ("N100_n14_m7_two_rows", 2, 100, 14, 7),   # 1400 rows: two per thread
    ("N128_n16_m8_two_rows", 1, 128, 16, 8),   # 2048 rows, the largest
    ("N45_n12_m4_cluster", 2, 45, 12, 4),      # two CTAs per solve, 23 + 22 knots
]


@pytest.mark.parametrize("name,M,N,n,m", FF_SIZES, ids=[c[0] for c in FF_SIZES])
def test_double_float_pcg_sizes(name, M, N, n, m):
    """Every size class of the double-float kernel (one and two rows per
    thread, n up to 64, N = 1, a solve split over two CTAs of a cluster with a
    ragged split) against the oracle, and against the fp32 kernel's lambda."""
    prob = random_lq(M, N, n, m, seed=950 + N + n)
    p = gato.default_params(pcg_max_iters=5000, refine_steps=1, pcg_precision=FF)
    out = solve(prob, p)
    assert not out["status"].any(), out["status"]
    check_solution(prob, out, range(M))
    ref = solve(prob, gato.default_params(pcg_max_iters=5000, refine_steps=1))
    for j in range(M):
        assert rel(out["lam"][j], ref["lam"][j]) < 1e-3


@pytest.mark.parametrize("rule", [gato.GATO_STOP_PRECOND, gato.GATO_STOP_SCALED],
                         ids=["precond", "scaled"])
def test_double_float_pcg_other_stop_rules(rule):
    """The other stopping rules stop the double-float solve where the fp64
    oracle's same rule stops (within 3 %)."""
    w = WORKLOADS[2]
    prob = make_batch(w, M=4)
    out = pcg_only(prob, params_for(w, stop_rule=rule, refine_steps=0))
    assert not out["status"].any()
    for j in range(4):
        D, O, gam, _ = oracle.schur(oracle.solve_one(prob, j))
        Pd, Po, _ = oracle.stair(D, O)
        _, it, ok = oracle.pcg(D, O, Pd, Po, gam, w.pcg_eps, 5000, stop_rule=rule)
        assert ok and it * 0.97 - 3 <= out["iters"][j] <= it * 1.03 + 3, (j, it, out["iters"][j])


@pytest.mark.parametrize("wi,N", [(0, 24), (2, 64)], ids=["one_cta", "cluster"])
def test_double_float_pcg_warm_start(wi, N):
    """From the exact multipliers no iteration is needed; from half of them
    fewer than from zero (one CTA per solve, and two CTAs of a cluster)."""
    w = WORKLOADS[wi]
    prob = make_batch(w, M=2, N=N)
    lam = np.stack([oracle.direct_solve(oracle.solve_one(prob, j))[2] for j in range(2)])
    p = params_for(w, refine_steps=0, pcg_max_iters=1000)
    at = pcg_only(prob, gato.default_params(pcg_eps=1e-3, pcg_precision=FF), lambda0=lam)
    assert (at["iters"] == 0).all()
    cold = pcg_only(prob, p)
    half = pcg_only(prob, p, lambda0=0.5 * lam)
    assert not cold["status"].any() and not half["status"].any()
    assert (half["iters"] <= cold["iters"]).all()
    for j in range(2):
        assert rel(half["lam"][j], lam[j]) < 1e-3


def test_double_float_pcg_rejects_sizes_beyond_it():
    """More than 2048 rows (or more than 1024 with n > 16): rejected as
    unsupported rather than solved at a lower precision."""
    for (N, n, m) in ((150, 14, 7), (30, 36, 12)):
        prob = random_lq(1, N, n, m, seed=990)
        with pytest.raises(gato.GatoError) as e:
            solve(prob, gato.default_params(pcg_max_iters=100, pcg_precision=FF))
        assert e.value.code == gato.GATO_ERR_UNSUPPORTED


# --------------------------------------------------------------------------
# invariance gates
# --------------------------------------------------------------------------

def test_merit_bit_identical_across_block_sizes():
    """The per-(knot, candidate) kernel sums rows and knots in a fixed order,
    so its merits are bit-identical at any block size."""
    w = WORKLOADS[1]
    prob = make_batch(w, M=4)
    ref = None
    for mt in (32, 64, 128, 256):
        out = solve(prob, params_for(w, merit_threads=mt,
                                     merit_kernel=gato.GATO_MERIT_PER_CANDIDATE))
        if ref is None:
            ref = out
        assert np.array_equal(out["merit"], ref["merit"])
        assert np.array_equal(out["best"], ref["best"])
    check_solution(prob, ref, range(4), w.n_alpha, w.beta, w.mu)


@pytest.mark.parametrize("w", [WORKLOADS[0], WORKLOADS[3], WORKLOADS[4]], ids=lambda w: w.name)
def test_merit_kernels_agree(w):
    """Fused (factored) and per-candidate (full formula) merit kernels agree
    within the merit tolerance and pick the same step."""
    prob = make_batch(w, M=min(w.M, 6))
    a = solve(prob, params_for(w, merit_kernel=gato.GATO_MERIT_FUSED))
    b = solve(prob, params_for(w, merit_kernel=gato.GATO_MERIT_PER_CANDIDATE))
    for j in range(a["merit"].shape[0]):
        scale = np.abs(b["merit"][j]).max()
        assert np.abs(a["merit"][j] - b["merit"][j]).max() <= TOL_MERIT * scale
    np.testing.assert_array_equal(a["best"], b["best"])
    np.testing.assert_array_equal(a["dX"], b["dX"])



# candidate counts 1..GATO_MAX_ALPHA, each merit kernel, on sizes that take the
# per-knot kernel (n, m <= 16: instantiations for up to 9 and up to 32 values
# of alpha) and the per-solve fused kernel (n > 16)
MERIT_COUNTS = [(1, 2.0, 10.0), (8, 2.0, 10.0), (9, 1.5, 3.0), (20, 1.25, 0.5),
                (gato.GATO_MAX_ALPHA, 2.0, 100.0)]


@pytest.mark.parametrize("kernel", [gato.GATO_MERIT_FUSED, gato.GATO_MERIT_PER_CANDIDATE],
                         ids=["fused", "per_candidate"])
@pytest.mark.parametrize("M,N,n,m", [(3, 32, 12, 6), (2, 9, 20, 8)], ids=["n12", "n20"])
@pytest.mark.parametrize("n_alpha,beta,mu", MERIT_COUNTS,
                         ids=[f"A{c[0]}" for c in MERIT_COUNTS])
def test_merit_candidate_counts(n_alpha, beta, mu, M, N, n, m, kernel):
    """Merit values of alpha = 0 and alpha_i = beta^-i, i < n_alpha, and the
    selected step against the oracle's line search on the GPU's own step."""
    prob = random_lq(M, N, n, m, seed=700 + n_alpha + n)
    out = solve(prob, gato.default_params(pcg_max_iters=3000, refine_steps=1, n_alpha=n_alpha,
                                          beta=beta, mu=mu, merit_kernel=kernel))
    assert out["merit"].shape == (M, n_alpha + 1)
    assert not out["status"].any(), out["status"]
    check_solution(prob, out, range(M), n_alpha, beta, mu)
    for j in range(M):  # alpha = 0 in closed form: mu times the L1 norm of (s0, e)
        ref0 = mu * (np.abs(prob["s0"][j]).astype(np.float64).sum()
                     + np.abs(prob["e"][j]).astype(np.float64).sum())
        assert abs(out["merit"][j, 0] - ref0) <= TOL_MERIT * ref0


def test_deterministic_and_batch_position_invariant():
    w = WORKLOADS[4]
    prob = make_batch(w, M=6)
    a = solve(prob, params_for(w))
    b = solve(prob, params_for(w))
    for k in a:
        assert np.array_equal(a[k], b[k]), k
    one = solve({k: v[3:4] for k, v in prob.items()}, params_for(w))
    for k in ("dX", "dU", "lam", "merit", "best", "iters"):
        assert np.array_equal(one[k][0], a[k][3]), k


def test_separate_entry_points_equal_solve_kkt():
    w = WORKLOADS[1]
    prob = make_batch(w, M=3)
    p = params_for(w, refine_steps=0)
    full = solve(prob, p)
    d = gato.to_device(prob)
    with gato.Solver(3, w.N, w.n, w.m) as s:
        o = s.outputs(p.n_alpha)
        s.form_schur(d, o["status"])
        s.pcg_solve(p, o["lam"], o["dX"], o["dU"], o["iters"], o["status"])
        s.linesearch(p, d, o["dX"], o["dU"], o["merit"], o["best"], o["status"])
        torch.cuda.synchronize()
        for k in ("dX", "dU", "lam", "merit", "best", "iters", "status"):
            assert np.array_equal(o[k].cpu().numpy(), full[k]), k


# --------------------------------------------------------------------------
# line search on given steps, update, warm start
# --------------------------------------------------------------------------

@pytest.mark.parametrize("kernel", [0, 1])
@pytest.mark.parametrize("scale", [2.5, 6.0, -1.0])
def test_linesearch_on_scaled_steps(scale, kernel):
    w = WORKLOADS[1]
    prob = make_batch(w, M=4)
    d = gato.to_device(prob)
    dX = np.stack([oracle.direct_solve(oracle.solve_one(prob, j))[0] for j in range(4)])
    dU = np.stack([oracle.direct_solve(oracle.solve_one(prob, j))[1] for j in range(4)])
    dXt = torch.tensor(scale * dX, dtype=torch.float32, device="cuda")
    dUt = torch.tensor(scale * dU, dtype=torch.float32, device="cuda")
    p = params_for(w, merit_kernel=kernel)
    with gato.Solver(4, w.N, w.n, w.m) as s:
        o = s.outputs(p.n_alpha)
        s.linesearch(p, d, dXt, dUt, o["merit"], o["best"], o["status"])
        torch.cuda.synchronize()
        merit, best, status = (o[k].cpu().numpy() for k in ("merit", "best", "status"))
    for j in range(4):
        pj = oracle.solve_one(prob, j)
        check_merit(pj, dXt[j].cpu().numpy(), dUt[j].cpu().numpy(), merit[j], best[j],
                    p.n_alpha, p.beta, p.mu)
        if scale < 0:
            assert best[j] == -1 and status[j] & gato.GATO_STATUS_LINESEARCH_FAILED
        else:
            assert best[j] > 0 and status[j] == 0


def test_apply_step():
    w = WORKLOADS[1]
    prob = make_batch(w, M=3)
    out = solve(prob, params_for(w))
    X0 = np.random.default_rng(1).standard_normal(out["dX"].shape).astype(np.float32)
    U0 = np.random.default_rng(2).standard_normal(out["dU"].shape).astype(np.float32)
    best = np.array([0, 2, -1], dtype=np.int32)
    X, U = torch.tensor(X0, device="cuda"), torch.tensor(U0, device="cuda")
    p = params_for(w)
    with gato.Solver(3, w.N, w.n, w.m) as s:
        s.apply_step(p, torch.tensor(best, device="cuda"), torch.tensor(out["dX"], device="cuda"),
                     torch.tensor(out["dU"], device="cuda"), X, U)
        torch.cuda.synchronize()
    alpha = np.array([1.0, 0.25, 0.0], dtype=np.float32)
    np.testing.assert_array_equal(X.cpu().numpy(), X0 + alpha[:, None, None] * out["dX"])
    np.testing.assert_array_equal(U.cpu().numpy(), U0 + alpha[:, None, None] * out["dU"])


WARM = [("n12_auto", 12, gato.GATO_PCG_AUTO), ("n12_generic", 12, gato.GATO_PCG_GENERIC),
        ("n12_tile", 12, gato.GATO_PCG_TILE), ("n12_quad", 12, gato.GATO_PCG_QUAD),
        ("n36_rows", 36, gato.GATO_PCG_AUTO),
        ("n36_generic", 36, gato.GATO_PCG_GENERIC)]


def _warm_problem(n):
    return make_batch(WORKLOADS[1], M=2) if n == 12 else random_lq(2, 8, 36, 12, seed=910)


@pytest.mark.parametrize("name,n,kind", WARM, ids=[c[0] for c in WARM])
def test_warm_start_at_solution_needs_no_iterations(name, n, kind):
    prob = _warm_problem(n)
    M, N, n_, m = 2, prob["Q"].shape[1], n, prob["R"].shape[-1]
    lam = np.stack([oracle.direct_solve(oracle.solve_one(prob, j))[2] for j in range(2)])
    d = gato.to_device(prob)
    p = gato.default_params(pcg_eps=1e-3, pcg_max_iters=3000)
    with gato.Solver(M, N, n_, m) as s:
        s.set_pcg_kernel(kind)
        o = s.outputs(p.n_alpha)
        s.form_schur(d, o["status"])
        s.pcg_solve(p, o["lam"], o["dX"], o["dU"], o["iters"], o["status"],
                    lambda0=torch.tensor(lam, dtype=torch.float32, device="cuda"))
        torch.cuda.synchronize()
        assert (o["iters"].cpu().numpy() == 0).all()
        for j in range(2):
            assert rel(o["lam"][j].cpu().numpy(), lam[j]) < 1e-4


@pytest.mark.parametrize("name,n,kind", WARM, ids=[c[0] for c in WARM])
def test_warm_start_from_a_partial_solution(name, n, kind):
    """From half the solution every kernel converges to it, in fewer
    iterations than from zero."""
    prob = _warm_problem(n)
    M, N, m = 2, prob["Q"].shape[1], prob["R"].shape[-1]
    lam = np.stack([oracle.direct_solve(oracle.solve_one(prob, j))[2] for j in range(2)])
    d = gato.to_device(prob)
    p = gato.default_params(pcg_eps=1e-6, pcg_max_iters=5000)
    with gato.Solver(M, N, n, m) as s:
        s.set_pcg_kernel(kind)
        o = s.outputs(p.n_alpha)
        s.form_schur(d, o["status"])
        s.pcg_solve(p, o["lam"], o["dX"], o["dU"], o["iters"], o["status"])
        cold = o["iters"].cpu().numpy().copy()
        s.pcg_solve(p, o["lam"], o["dX"], o["dU"], o["iters"], o["status"],
                    lambda0=torch.tensor(0.5 * lam, dtype=torch.float32, device="cuda"))
        torch.cuda.synchronize()
        assert not o["status"].cpu().numpy().any()
        assert (o["iters"].cpu().numpy() <= cold).all()
        for j in range(2):
            assert rel(o["lam"][j].cpu().numpy(), lam[j]) < 1e-3


# --------------------------------------------------------------------------
# failure detection (host-made faults; flags, never traps)
# --------------------------------------------------------------------------

def test_iteration_cap_is_flagged():
    w = WORKLOADS[1]
    prob = make_batch(w, M=2)
    out = solve(prob, params_for(w, pcg_max_iters=5, refine_steps=0))
    assert (out["iters"] == 5).all()
    assert (out["status"] & gato.GATO_STATUS_PCG_MAX_ITERS).all()


def test_indefinite_Q_is_flagged():
    w = WORKLOADS[0]
    prob = make_batch(w, M=2)
    prob["Q"] = prob["Q"].copy()
    prob["Q"][1, 3] = -np.eye(w.n, dtype=np.float32)
    out = solve(prob, params_for(w, pcg_max_iters=50))
    assert out["status"][1] & gato.GATO_STATUS_NONPOSITIVE_PIVOT
    assert not out["status"][0] & gato.GATO_STATUS_NONPOSITIVE_PIVOT


def test_nan_input_is_flagged():
    w = WORKLOADS[0]
    prob = make_batch(w, M=2)
    prob["q"] = prob["q"].copy()
    prob["q"][0, 2, 1] = np.nan
    out = solve(prob, params_for(w, pcg_max_iters=50))
    assert out["status"][0] & gato.GATO_STATUS_NONFINITE
    assert not out["status"][1] & gato.GATO_STATUS_NONFINITE


def test_invalid_parameters_rejected():
    w = WORKLOADS[0]
    prob = make_batch(w, M=1)
    for bad in (dict(merit_threads=48), dict(n_alpha=0), dict(beta=1.0), dict(stop_rule=7),
                dict(pcg_max_iters=-1), dict(merit_kernel=5), dict(refine_eps=-1.0),
                dict(pcg_precision=2), dict(pcg_precision=-1), dict(refine_solver=2)):
        with pytest.raises(gato.GatoError) as e:
            solve(prob, params_for(w, **bad))
        assert e.value.code == gato.GATO_ERR_INVALID_ARG


def test_stage_timing():
    w = WORKLOADS[1]
    prob = make_batch(w, M=4)
    d = gato.to_device(prob)
    p = params_for(w)
    with gato.Solver(4, w.N, w.n, w.m) as s:
        o = s.outputs(p.n_alpha)
        s.set_timing(True)
        s.solve_kkt(p, d, o["dX"], o["dU"], o["lam"], o["iters"], o["merit"], o["best"], o["status"])
        st = s.get_stats()
    assert st.form_us > 0 and st.pcg_us > 0 and st.merit_us > 0
    assert st.total_us >= st.pcg_us


def test_batch_beyond_the_grid_yz_limit():
    """70000 solves, more than a grid's y or z extent holds (65535): the
    per-candidate merit is launched in slices, the factored merit runs one
    block per solve for a single part, its per-knot form per part of four.
    All give the same steps; samples are checked against the oracle."""
    base = random_lq(7, 2, 2, 1, seed=991)
    M = 70000
    prob = {k: np.ascontiguousarray(np.tile(v, (M // 7,) + (1,) * (v.ndim - 1)))
            for k, v in base.items()}
    d = gato.to_device(prob)
    runs = {}
    with gato.Solver(M, 2, 2, 1) as s:
        for name, kind, parts in (("fused, one part", gato.GATO_MERIT_FUSED, 1),
                                  ("fused, four parts", gato.GATO_MERIT_FUSED, 4),
                                  ("per candidate", gato.GATO_MERIT_PER_CANDIDATE, 1)):
            s.set_parts(parts)
            p = gato.default_params(pcg_max_iters=200, merit_kernel=kind)
            out = s.outputs(p.n_alpha)
            s.solve_kkt(p, d, out["dX"], out["dU"], out["lam"], out["iters"], out["merit"],
                        out["best"], out["status"])
            torch.cuda.synchronize()
            runs[name] = {k: v.cpu().numpy() for k, v in out.items()}
    ref = runs["fused, one part"]
    for name, out in runs.items():
        assert np.array_equal(out["dX"], ref["dX"]), name
        assert np.array_equal(out["best"], ref["best"]), name
        scale = np.abs(ref["merit"]).max(axis=1, keepdims=True)
        assert (np.abs(out["merit"] - ref["merit"]) <= TOL_MERIT * scale).all(), name
    assert not ref["status"].any()
    check_solution(prob, ref, [0, 35000, 65534, 65535, 69999])


@pytest.mark.parametrize("w", [WORKLOADS[1], WORKLOADS[3], WORKLOADS[4]], ids=lambda w: w.name)
def test_default_stop_rule_reaches_the_relative_residual(w):
    """The default rule stops on ||gamma - S lambda|| <= eps ||gamma|| of the
    updated residual: the true residual of the returned lambda, against the S
    and gamma the GPU formed (exported, evaluated in fp64), stays within a
    small multiple of eps, and the iteration count tracks the fp64 oracle's.
    On the ill-conditioned workload 3 fp32 CG loses orthogonality and needs
    20 to 35% more iterations than fp64 CG (any kernel: the generic one
    too), so its upper bound is 1.5 times the oracle's."""
    M = 3
    prob = make_batch(w, M=M)
    p = params_for(w, refine_steps=0)
    d = gato.to_device(prob)
    N, n = w.N, w.n
    f = dict(device="cuda", dtype=torch.float32)
    with gato.Solver(M, N, n, w.m) as s:
        o = s.outputs(p.n_alpha)
        s.form_schur(d, o["status"])
        s.pcg_solve(p, o["lam"], o["dX"], o["dU"], o["iters"], o["status"])
        D = torch.empty(M, N, n, n, **f)
        O = torch.empty(M, N - 1, n, n, **f)
        g = torch.empty(M, N, n, **f)
        s.get_schur(D, O, g)
        torch.cuda.synchronize()
        lam, iters = o["lam"].cpu().numpy(), o["iters"].cpu().numpy()
        D, O, g = D.cpu().numpy(), O.cpu().numpy(), g.cpu().numpy()
    assert not o["status"].cpu().numpy().any()
    for j in range(M):
        S = oracle.bt_dense(D[j], O[j])
        gj = g[j].astype(np.float64).ravel()
        res = np.linalg.norm(gj - S @ lam[j].astype(np.float64).ravel()) / np.linalg.norm(gj)
        assert res <= 10 * w.pcg_eps, (j, res)
        Dj, Oj, gam, _ = oracle.schur(oracle.solve_one(prob, j))
        Pd, Po, _ = oracle.stair(Dj, Oj)
        _, it, ok = oracle.pcg(Dj, Oj, Pd, Po, gam, w.pcg_eps, 5000, stop_rule=0)
        upper = 1.5 if w.index == 3 else 1.2
        assert ok and it * 0.9 - 3 <= int(iters[j]) <= it * upper + 5, (j, it, iters[j])
