"""The batch in parts: gato_solve_kkt and gato_solve_kkt_host split a batch
into parts of consecutive solves that run concurrently on internal streams
(gato_set_parts), the host entry also copying each part's slice in and out.
Each part runs the one-part path's arithmetic on its solves, so every output
must equal the one-part gato_solve_kkt's bit for bit, for every part count
(ragged parts included), and be within the oracle's tolerance."""
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


def device_solve(s, p, prob, parts):
    s.set_parts(parts)
    d = gato.to_device(prob)
    out = s.outputs(p.n_alpha)
    s.solve_kkt(p, d, out["dX"], out["dU"], out["lam"], out["iters"], out["merit"], out["best"],
                out["status"])
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in out.items()}


def host_solve(s, p, prob, parts, status0=None):
    s.set_parts(parts)
    hp = gato.to_host(prob)
    out = s.host_outputs(p.n_alpha)
    if status0 is not None:
        out["status"].copy_(torch.as_tensor(status0, dtype=torch.int32))
    stream = torch.cuda.current_stream()
    s.solve_kkt_host(p, hp, out["dX"], out["dU"], out["lam"], out["iters"], out["merit"],
                     out["best"], out["status"], stream)
    stream.synchronize()
    return {k: v.numpy().copy() for k, v in out.items()}


def same(a, b):
    for k in b:
        assert np.array_equal(a[k], b[k]), k


@pytest.mark.parametrize("parts", [0, 1, 2, 3, 7])
def test_parts_equal_one_part(parts):
    w = WORKLOADS[4]
    M = 23  # ragged parts for 2, 3 and 7
    prob = make_batch(w, M=M)
    p = params_for(w)
    with gato.Solver(M, w.N, w.n, w.m) as s:
        ref = device_solve(s, p, prob, 1)
        dev = device_solve(s, p, prob, parts)
        host = host_solve(s, p, prob, parts)
    same(dev, ref)
    same(host, ref)
    check_solution(prob, host, [0, 11, 22], w.n_alpha, w.beta, w.mu)


def test_default_parts_at_the_benchmark_batch():
    """256 solves: four parts by default, two on device buffers with the
    workload's direct corrections (their factorisation runs beside the PCG),
    four from host buffers; a sample against the oracle and every output
    against the one-part run."""
    w = WORKLOADS[4]
    prob = make_batch(w)
    p = params_for(w)
    assert p.refine_solver == gato.GATO_REFINE_SOLVER_DIRECT
    with gato.Solver(w.M, w.N, w.n, w.m) as s:
        s.set_parts(0)
        assert s.get_parts() == 4  # no call yet: the default parameters
        ref = device_solve(s, p, prob, 1)
        assert s.get_parts() == 1
        dev = device_solve(s, p, prob, 0)
        assert s.get_parts() == 2
        pcg_corr = device_solve(s, params_for(w, refine_solver=0), prob, 0)
        assert s.get_parts() == 4
        host = host_solve(s, p, prob, 0)
        assert s.get_parts() == 4
    same(dev, ref)
    same(host, ref)
    assert not pcg_corr["status"].any()
    assert not ref["status"].any()
    check_solution(prob, dev, [0, 63, 64, 191, 255], w.n_alpha, w.beta, w.mu)


def test_default_parts_by_batch_size():
    """With direct corrections on device buffers: one part while the PCG holds
    the whole batch at once, two beyond.  At N = 128, n = 14 the wide-tile
    kernel holds one solve per SM; at N = 32 an SM holds several, so one more
    solve than SMs still runs as one part.  The outputs equal the one-part
    run's."""
    n_sm = torch.cuda.get_device_properties(0).multi_processor_count
    for wi, M, expect in ((4, n_sm, 1), (4, n_sm + 1, 2), (1, n_sm + 1, 1)):
        w = WORKLOADS[wi]
        p = params_for(w)
        assert p.refine_solver == gato.GATO_REFINE_SOLVER_DIRECT
        prob = make_batch(w, M=M)
        with gato.Solver(M, w.N, w.n, w.m) as s:
            ref = device_solve(s, p, prob, 1)
            out = device_solve(s, p, prob, 0)
            assert s.get_parts() == expect, (wi, M)
        same(out, ref)
        assert not out["status"].any()


def test_parts_are_reused_and_rebuilt():
    w = WORKLOADS[1]
    prob = make_batch(w, M=9)
    p = params_for(w)
    with gato.Solver(9, w.N, w.n, w.m) as s:
        ref = device_solve(s, p, prob, 1)
        runs = [host_solve(s, p, prob, k) for k in (2, 2, 4, 1)]
        runs += [device_solve(s, p, prob, k) for k in (4, 3, 3)]
    for out in runs:
        same(out, ref)


def test_host_status_is_in_out_and_single_knot_problems():
    prob = random_lq(5, 1, 6, 3, seed=901)  # N = 1: no R, A, B, e, no controls
    prob = {k: v for k, v in prob.items() if k in ("Q", "q", "s0")}
    p = gato.default_params()
    with gato.Solver(5, 1, 6, 3) as s:
        out = host_solve(s, p, prob, 2, status0=[0, 64, 0, 0, 64])
        ref = device_solve(s, p, prob, 1)
        dev = device_solve(s, p, prob, 2)
    # the bit set before the call survives; the solver's own bits are the one-part run's
    assert list(out["status"] & 64) == [0, 64, 0, 0, 64]
    assert np.array_equal(out["status"] & ~64, ref["status"])
    for k in ("dX", "lam", "merit", "best", "iters"):
        assert np.array_equal(out[k], ref[k]), k
        assert np.array_equal(dev[k], ref[k]), k


def test_stage_timing_only_for_one_part():
    w = WORKLOADS[1]
    prob = make_batch(w, M=8)
    p = params_for(w)
    d = gato.to_device(prob)
    with gato.Solver(8, w.N, w.n, w.m) as s:
        o = s.outputs(p.n_alpha)
        s.set_timing(True)
        for parts, timed in ((2, False), (1, True)):
            s.set_parts(parts)
            s.solve_kkt(p, d, o["dX"], o["dU"], o["lam"], o["iters"], o["merit"], o["best"],
                        o["status"])
            st = s.get_stats()
            assert (st.pcg_us > 0) == timed and (st.total_us > 0) == timed


def test_parts_reject_bad_arguments():
    w = WORKLOADS[1]
    prob = make_batch(w, M=2)
    p = params_for(w)
    with gato.Solver(2, w.N, w.n, w.m) as s:
        for bad in (-1, gato.GATO_MAX_PARTS + 1):
            with pytest.raises(gato.GatoError) as e:
                s.set_parts(bad)
            assert e.value.code == gato.GATO_ERR_INVALID_ARG
        s.set_parts(gato.GATO_MAX_PARTS)
        assert s.get_parts() == 2  # capped at M
        out = s.host_outputs(p.n_alpha)
        with pytest.raises(ValueError):  # device tensors are refused by the binding
            s.solve_kkt_host(p, gato.to_device(prob), out["dX"], out["dU"], out["lam"],
                             out["iters"], out["merit"], out["best"], out["status"])


def test_call_in_parts_allocates_nothing_and_can_be_captured():
    """The parts are views into the handle's own allocation: a call that
    re-partitions the batch leaves the free device memory unchanged, and a
    call captured into a CUDA graph replays to the same outputs."""
    w = WORKLOADS[4]
    # one solve more than the SMs, so that the automatic choice runs two parts
    M = torch.cuda.get_device_properties(0).multi_processor_count + 1
    prob = make_batch(w, M=M)
    p = params_for(w)
    d = gato.to_device(prob)
    with gato.Solver(M, w.N, w.n, w.m) as s:
        ref = device_solve(s, p, prob, 1)  # loads every kernel once
        same(device_solve(s, p, prob, 4), ref)  # and uses every part's stream
        s.set_parts(2)
        out = s.outputs(p.n_alpha)
        torch.cuda.synchronize()
        free0 = torch.cuda.mem_get_info()[0]
        s.solve_kkt(p, d, out["dX"], out["dU"], out["lam"], out["iters"], out["merit"],
                    out["best"], out["status"])
        torch.cuda.synchronize()
        assert torch.cuda.mem_get_info()[0] == free0
        same({k: v.cpu().numpy() for k, v in out.items()}, ref)
        s.set_parts(0)
        cap = s.outputs(p.n_alpha)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, capture_error_mode="thread_local"):
            s.solve_kkt(p, d, cap["dX"], cap["dU"], cap["lam"], cap["iters"], cap["merit"],
                        cap["best"], cap["status"])
        g.replay()
        torch.cuda.synchronize()
        assert s.get_parts() == 2  # more solves than SMs, direct corrections
        same({k: v.cpu().numpy() for k, v in cap.items()}, ref)


def test_faults_stay_with_their_solve_across_parts():
    """An indefinite Q in one solve and a NaN in another set status bits for
    those solves only, the same in parts, through the host entry and as one
    part; the other solves' outputs are unchanged."""
    w = WORKLOADS[1]
    M = 9
    prob = make_batch(w, M=M)
    bad = {k: v.copy() for k, v in prob.items()}
    bad["Q"][4, 3] = -np.eye(w.n, dtype=np.float32)  # indefinite block: pivot <= 0
    bad["q"][7, 5, 2] = np.nan
    p = params_for(w)
    with gato.Solver(M, w.N, w.n, w.m) as s:
        clean = device_solve(s, p, prob, 1)
        ref = device_solve(s, p, bad, 1)
        dev = device_solve(s, p, bad, 3)
        host = host_solve(s, p, bad, 3)
    assert ref["status"][4] & gato.GATO_STATUS_NONPOSITIVE_PIVOT
    assert ref["status"][7] & gato.GATO_STATUS_NONFINITE
    others = [j for j in range(M) if j not in (4, 7)]
    assert not ref["status"][others].any()
    for k in ("dX", "dU", "lam", "merit", "best", "iters"):
        assert np.array_equal(ref[k][others], clean[k][others]), k
    for out in (dev, host):
        assert np.array_equal(out["status"], ref["status"])
        for k in ("dX", "dU", "lam", "merit", "best", "iters"):
            assert np.array_equal(out[k], ref[k], equal_nan=True), k


def test_host_entry_takes_pageable_buffers():
    """Pageable (unpinned) host arrays are copied without overlap but give
    the same outputs as pinned ones."""
    w = WORKLOADS[1]
    M = 11
    prob = make_batch(w, M=M)
    p = params_for(w)
    with gato.Solver(M, w.N, w.n, w.m) as s:
        ref = host_solve(s, p, prob, 3)
        s.set_parts(3)
        hp = {k: torch.from_numpy(np.ascontiguousarray(v, dtype=np.float32)) for k, v in prob.items()}
        assert not any(t.is_pinned() for t in hp.values())
        out = {k: torch.zeros(v.shape, dtype=v.dtype) for k, v in s.host_outputs(p.n_alpha).items()}
        assert not any(t.is_pinned() for t in out.values())
        stream = torch.cuda.current_stream()
        s.solve_kkt_host(p, hp, out["dX"], out["dU"], out["lam"], out["iters"], out["merit"],
                         out["best"], out["status"], stream)
        stream.synchronize()
    same({k: v.numpy() for k, v in out.items()}, ref)
