"""gato_solve_kkt_host: the solve of a batch held in host memory, split into
parts whose copies overlap the other parts' solves.  Each part runs the
device path's arithmetic on its solves, so the outputs must equal
gato_solve_kkt's bit for bit, for every part count (ragged parts included),
and be within the oracle's tolerance."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from trajectory_optimization_kkt_gb300 import gato  # noqa: E402
from trajectory_optimization_kkt_gb300.workloads import WORKLOADS, make_batch, random_lq  # noqa: E402

from test_gpu_parity import check_solution, params_for  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()


def device_solve(s, p, prob):
    d = gato.to_device(prob)
    out = s.outputs(p.n_alpha)
    s.solve_kkt(p, d, out["dX"], out["dU"], out["lam"], out["iters"], out["merit"], out["best"],
                out["status"])
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in out.items()}


def host_solve(s, p, prob, status0=None):
    hp = gato.to_host(prob)
    out = s.host_outputs(p.n_alpha)
    if status0 is not None:
        out["status"].copy_(torch.as_tensor(status0, dtype=torch.int32))
    stream = torch.cuda.current_stream()
    s.solve_kkt_host(p, hp, out["dX"], out["dU"], out["lam"], out["iters"], out["merit"],
                     out["best"], out["status"], stream)
    stream.synchronize()
    return {k: v.numpy().copy() for k, v in out.items()}


@pytest.mark.parametrize("chunks", [0, 1, 2, 3, 7])
def test_host_path_equals_device_path(chunks):
    w = WORKLOADS[4]
    M = 23  # ragged parts for 2, 3 and 7
    prob = make_batch(w, M=M)
    p = params_for(w)
    with gato.Solver(M, w.N, w.n, w.m) as s:
        ref = device_solve(s, p, prob)
        s.set_host_chunks(chunks)
        out = host_solve(s, p, prob)
    for k in ref:
        assert np.array_equal(out[k], ref[k]), k
    check_solution(prob, out, [0, 11, 22], w.n_alpha, w.beta, w.mu)


def test_host_path_reuses_and_rebuilds_its_parts():
    w = WORKLOADS[1]
    prob = make_batch(w, M=9)
    p = params_for(w)
    with gato.Solver(9, w.N, w.n, w.m) as s:
        ref = device_solve(s, p, prob)
        results = []
        for chunks in (2, 2, 4, 1):
            s.set_host_chunks(chunks)
            results.append(host_solve(s, p, prob))
    for out in results:
        for k in ref:
            assert np.array_equal(out[k], ref[k]), k


def test_host_status_is_in_out_and_single_knot_problems():
    prob = random_lq(5, 1, 6, 3, seed=901)  # N = 1: no R, A, B, e, no controls
    prob = {k: v for k, v in prob.items() if k in ("Q", "q", "s0")}
    p = gato.default_params()
    with gato.Solver(5, 1, 6, 3) as s:
        s.set_host_chunks(2)
        out = host_solve(s, p, prob, status0=[0, 64, 0, 0, 64])
        ref = device_solve(s, p, prob)
    # the bit set before the call survives; the solver's own bits are the device path's
    assert list(out["status"] & 64) == [0, 64, 0, 0, 64]
    assert np.array_equal(out["status"] & ~64, ref["status"])
    for k in ("dX", "lam", "merit", "best", "iters"):
        assert np.array_equal(out[k], ref[k]), k


def test_host_path_rejects_bad_arguments():
    w = WORKLOADS[1]
    prob = make_batch(w, M=2)
    p = params_for(w)
    with gato.Solver(2, w.N, w.n, w.m) as s:
        for bad in (-1, gato.GATO_HOST_MAX_CHUNKS + 1):
            with pytest.raises(gato.GatoError) as e:
                s.set_host_chunks(bad)
            assert e.value.code == gato.GATO_ERR_INVALID_ARG
        out = s.host_outputs(p.n_alpha)
        with pytest.raises(ValueError):  # device tensors are refused by the binding
            s.solve_kkt_host(p, gato.to_device(prob), out["dX"], out["dU"], out["lam"],
                             out["iters"], out["merit"], out["best"], out["status"])
