"""gato_solve_kkt_noalloc against gato_solve_kkt.

The allocation-free entry point serves callers that cannot allocate device
memory while they run (a real-time MPC loop with memory fixed at start-up, a
host framework that owns every device allocation): its scratch is a static
device array inside the library.  This file is collected last so that a run
stopping at the first failure has already run every other test.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import oracle  # noqa: E402
from trajectory_optimization_kkt_gb300 import gato  # noqa: E402
from trajectory_optimization_kkt_gb300.workloads import WORKLOADS, make_batch  # noqa: E402

TOL_DZ = 1e-4     # relative L2 of the stacked dz, as in the parity tests
TOL_MERIT = 1e-5  # relative to max |merit| of the solve


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()


def rel(a, b):
    a, b = np.ravel(a), np.ravel(b)
    return np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300)


def params(w, linsys=gato.GATO_LINSYS_AUTO):
    return gato.default_params(pcg_eps=w.pcg_eps, pcg_max_iters=w.pcg_max_iters,
                               n_alpha=w.n_alpha, beta=w.beta, mu=w.mu,
                               refine_steps=w.refine_steps, refine_eps=w.refine_eps,
                               linsys=linsys)


def fresh_outputs(M, N, n, m, n_alpha):
    f = dict(device="cuda", dtype=torch.float32)
    return dict(dX=torch.full((M, N, n), np.nan, **f), dU=torch.full((M, N - 1, m), np.nan, **f),
                lam=torch.full((M, N, n), np.nan, **f),
                iters=torch.full((M,), -7, device="cuda", dtype=torch.int32),
                merit=torch.full((M, n_alpha + 1), np.nan, **f),
                best=torch.full((M,), -9, device="cuda", dtype=torch.int32),
                status=torch.zeros(M, device="cuda", dtype=torch.int32))


@pytest.mark.parametrize("wi,linsys", [(1, gato.GATO_LINSYS_AUTO), (2, gato.GATO_LINSYS_AUTO),
                                       (2, gato.GATO_LINSYS_BDSV)])
def test_noalloc_matches_solve_kkt_on_two_calls(wi, linsys):
    w = WORKLOADS[wi]
    M = min(w.M, 16)
    prob = make_batch(w, M=M)
    d = gato.to_device(prob)
    p = params(w, linsys)
    with gato.Solver(M, w.N, w.n, w.m) as s:
        ref = s.outputs(w.n_alpha)
        s.solve_kkt(p, d, ref["dX"], ref["dU"], ref["lam"], ref["iters"], ref["merit"],
                    ref["best"], ref["status"])
    torch.cuda.synchronize()
    ref = {k: v.cpu().numpy() for k, v in ref.items()}
    for call in range(2):  # the second call finds the first call's scratch
        o = fresh_outputs(M, w.N, w.n, w.m, w.n_alpha)
        gato.solve_kkt_noalloc(p, d, o["dX"], o["dU"], o["lam"], o["iters"], o["merit"],
                               o["best"], o["status"])
        torch.cuda.synchronize()
        o = {k: v.cpu().numpy() for k, v in o.items()}
        for j in range(M):
            z = np.concatenate([o["dX"][j].ravel(), o["dU"][j].ravel()])
            zr = np.concatenate([ref["dX"][j].ravel(), ref["dU"][j].ravel()])
            assert rel(z, zr) <= TOL_DZ, (call, j, rel(z, zr))
            scale = np.abs(ref["merit"][j]).max()
            assert np.abs(o["merit"][j] - ref["merit"][j]).max() <= TOL_MERIT * scale
        np.testing.assert_array_equal(o["best"], ref["best"])
        np.testing.assert_array_equal(o["status"], ref["status"])
        np.testing.assert_array_equal(o["iters"], ref["iters"])
    # and both agree with the fp64 oracle's direct solution
    dX, dU, _ = oracle.direct_solve(oracle.solve_one(prob, 0))
    assert rel(np.concatenate([o["dX"][0].ravel(), o["dU"][0].ravel()]),
               np.concatenate([dX.ravel(), dU.ravel()])) <= TOL_DZ


def test_noalloc_rejects_problems_beyond_its_scratch():
    w = WORKLOADS[4]  # 256 solves of 128 knots need far more than the static array
    prob = make_batch(w, M=2)
    d = {k: torch.zeros((w.M,) + v.shape[1:], dtype=torch.float32, device="cuda")
         for k, v in prob.items()}
    o = fresh_outputs(w.M, w.N, w.n, w.m, w.n_alpha)
    with pytest.raises(gato.GatoError) as e:
        gato.solve_kkt_noalloc(params(w), d, o["dX"], o["dU"], o["lam"], o["iters"],
                               o["merit"], o["best"], o["status"])
    assert e.value.code == gato.GATO_ERR_UNSUPPORTED
    assert (o["iters"].cpu().numpy() == -7).all()  # nothing ran
