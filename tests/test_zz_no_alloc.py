"""gato_solve_kkt_noalloc against gato_solve_kkt.

The allocation-free entry point serves callers that cannot allocate device
memory while they run (a real-time MPC loop with memory fixed at start-up, a
host framework that owns every device allocation): its scratch is a static
device array inside the library of GATO_NOALLOC_MAX_BYTES, and a problem
needs the bytes of noalloc_bytes() below (the header's exact expression).
This file is collected last so that a run stopping at the first failure has
already run every other test.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import oracle  # noqa: E402
from trajectory_optimization_kkt_gb300 import gato  # noqa: E402
from trajectory_optimization_kkt_gb300.workloads import WORKLOADS, make_batch, random_lq  # noqa: E402

TOL_DZ = 1e-4            # relative L2 of dX and of dU, as in the parity tests
TOL_MERIT = 1e-5         # per value, the value's magnitude floored at 1 % of
MERIT_NEAR_ZERO = 1e-2   # the solve's largest merit, as in the parity tests


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()


def rel(a, b):
    a, b = np.ravel(a).astype(np.float64), np.ravel(b).astype(np.float64)
    return np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300)


def noalloc_bytes(M, N, n, m):
    """Scratch bytes of one call, the expression include/gato.h states."""
    def r(x):
        return max(64, -(-x // 64) * 64)
    K = N - 1
    per_solve = (9 * r(N * n * n) + 3 * r(K * n * n) + r(K * m * m) + r(K * n * m)
                 + 17 * r(N * n) + 6 * r(K * m) + 2 * r(N) + 64 * N + 36)
    return 4 * (M * per_solve + M + 64)


def largest_batch(N, n, m):
    M = 1
    while noalloc_bytes(M + 1, N, n, m) <= gato.GATO_NOALLOC_MAX_BYTES:
        M += 1
    return M


def params(w, linsys=gato.GATO_LINSYS_AUTO):
    return gato.default_params(**w.solver_settings(), linsys=linsys)


def fresh_outputs(M, N, n, m, n_alpha):
    f = dict(device="cuda", dtype=torch.float32)
    return dict(dX=torch.full((M, N, n), np.nan, **f),
                dU=torch.full((M, max(N - 1, 0), m), np.nan, **f),
                lam=torch.full((M, N, n), np.nan, **f),
                iters=torch.full((M,), -7, device="cuda", dtype=torch.int32),
                merit=torch.full((M, n_alpha + 1), np.nan, **f),
                best=torch.full((M,), -9, device="cuda", dtype=torch.int32),
                status=torch.zeros(M, device="cuda", dtype=torch.int32))


def reference(prob, p):
    M, N, n = prob["Q"].shape[:3]
    m = prob["B"].shape[-1]
    d = gato.to_device(prob)
    with gato.Solver(M, N, n, m) as s:
        ref = s.outputs(p.n_alpha)
        s.solve_kkt(p, d, ref["dX"], ref["dU"], ref["lam"], ref["iters"], ref["merit"],
                    ref["best"], ref["status"])
    torch.cuda.synchronize()
    return d, {k: v.cpu().numpy() for k, v in ref.items()}


def call_noalloc(p, d, M, N, n, m, null_optional=False):
    o = fresh_outputs(M, N, n, m, p.n_alpha)
    if null_optional:  # N == 1: the [N-1] arrays are empty and may be NULL
        d = dict(d, R=None, r=None, A=None, B=None, e=None)
        o_dU = None
    else:
        o_dU = o["dU"]
    gato.solve_kkt_noalloc(p, d, o["dX"], o_dU, o["lam"], o["iters"], o["merit"], o["best"],
                           o["status"], dims=(M, N, n, m))
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in o.items()}


def assert_matches(o, ref, M, tag):
    for j in range(M):
        assert rel(o["dX"][j], ref["dX"][j]) <= TOL_DZ, (tag, j)
        if ref["dU"][j].size:
            assert rel(o["dU"][j], ref["dU"][j]) <= TOL_DZ, (tag, j)
        floor = MERIT_NEAR_ZERO * np.abs(ref["merit"][j]).max()
        tol = TOL_MERIT * np.maximum(np.abs(ref["merit"][j]), floor)
        assert (np.abs(o["merit"][j] - ref["merit"][j]) <= tol).all(), (tag, j)
    np.testing.assert_array_equal(o["best"], ref["best"])
    np.testing.assert_array_equal(o["status"], ref["status"])
    np.testing.assert_array_equal(o["iters"], ref["iters"])


@pytest.mark.parametrize("wi,linsys", [(1, gato.GATO_LINSYS_AUTO), (2, gato.GATO_LINSYS_AUTO),
                                       (2, gato.GATO_LINSYS_BDSV)])
def test_noalloc_matches_solve_kkt_on_two_calls(wi, linsys):
    w = WORKLOADS[wi]
    M = min(w.M, 16)
    prob = make_batch(w, M=M)
    p = params(w, linsys)
    d, ref = reference(prob, p)
    for call in range(2):  # the second call finds the first call's scratch
        o = call_noalloc(p, d, M, w.N, w.n, w.m)
        assert_matches(o, ref, M, call)
    # and both agree with the fp64 oracle's direct solution
    dX, dU, _ = oracle.direct_solve(oracle.solve_one(prob, 0))
    assert rel(o["dX"][0], dX) <= TOL_DZ and rel(o["dU"][0], dU) <= TOL_DZ


def test_noalloc_at_the_largest_batch_that_fits():
    """Workload 2's problem at the largest batch whose scratch fits the
    static array (46 solves of 64 knots): the array at its fullest."""
    w = WORKLOADS[2]
    M = largest_batch(w.N, w.n, w.m)
    assert M == 46
    prob = make_batch(w, M=M)
    p = params(w)
    d, ref = reference(prob, p)
    for call in range(2):
        assert_matches(call_noalloc(p, d, M, w.N, w.n, w.m), ref, M, call)


def test_noalloc_single_knot_with_null_optional_arrays():
    """N = 1: no controls, no dynamics; R, r, A, B, e and dU may be NULL."""
    prob = random_lq(3, 1, 14, 7, seed=4242)
    p = gato.default_params(pcg_max_iters=100, refine_steps=1)
    d, ref = reference(prob, p)
    for call in range(2):
        assert_matches(call_noalloc(p, d, 3, 1, 14, 7, null_optional=True), ref, 3, call)


@pytest.mark.parametrize("wi,M", [(4, 256), (2, 64), (2, 47)])
def test_noalloc_rejects_problems_beyond_its_scratch(wi, M):
    """Workload 4 at its batch, workload 2 at its full batch of 64 (about 44
    MiB of scratch) and one solve past the largest batch that fits: rejected
    with GATO_ERR_UNSUPPORTED before anything runs."""
    w = WORKLOADS[wi]
    assert noalloc_bytes(M, w.N, w.n, w.m) > gato.GATO_NOALLOC_MAX_BYTES
    shape = make_batch(w, M=1)
    d = {k: torch.zeros((M,) + v.shape[1:], dtype=torch.float32, device="cuda")
         for k, v in shape.items()}
    o = fresh_outputs(M, w.N, w.n, w.m, w.n_alpha)
    with pytest.raises(gato.GatoError) as e:
        gato.solve_kkt_noalloc(params(w), d, o["dX"], o["dU"], o["lam"], o["iters"],
                               o["merit"], o["best"], o["status"])
    assert e.value.code == gato.GATO_ERR_UNSUPPORTED
    assert (o["iters"].cpu().numpy() == -7).all()  # nothing ran


@pytest.mark.parametrize("wi,M", [(1, 16), (2, 40)])
def test_forked_factorisation_gives_the_serial_results(wi, M):
    """With direct corrections after a PCG solve, gato_solve_kkt forms the
    corrections' factorisation on a low-priority side stream beside the main
    solve; the allocation-free entry has no side stream and forms it in
    stream order.  The same kernels on the same data: bit-identical outputs
    (workload 2 at 40 solves runs one part in both, and its double-float main
    solve over clusters of two CTAs)."""
    w = WORKLOADS[wi]
    prob = make_batch(w, M=M)
    p = params(w)
    assert p.refine_solver == gato.GATO_REFINE_SOLVER_DIRECT and p.refine_steps >= 1
    d, ref = reference(prob, p)
    o = call_noalloc(p, d, M, w.N, w.n, w.m)
    for k in ref:
        np.testing.assert_array_equal(o[k], ref[k], err_msg=k)
