"""CPU-side checks of the C ABI: the library builds, loads without a GPU,
exports every entry point include/gato.h declares, and rejects bad arguments
before touching CUDA."""
import ctypes
import os
import re

import numpy as np
import pytest

from trajectory_optimization_kkt_gb300 import _build, gato
from trajectory_optimization_kkt_gb300.workloads import WORKLOADS, make_batch, normals, uniforms

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "gato.h")


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return gato.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gato_\w+)\s*\(", text)))


def test_header_declares_the_abi():
    names = declared_functions()
    for fn in ("gato_create", "gato_destroy", "gato_form_schur", "gato_pcg_solve",
               "gato_linesearch", "gato_solve_kkt", "gato_apply_step", "gato_get_schur",
               "gato_default_params", "gato_set_timing", "gato_get_stats",
               "gato_set_pcg_kernel", "gato_set_form_kernel", "gato_solve_kkt_noalloc",
               "gato_bdsv_solve", "gato_set_bdsv_kernel", "gato_sqp_linear",
               "gato_default_sqp_params", "gato_solve_kkt_host", "gato_set_parts",
               "gato_get_parts", "gato_probe_fp32"):
        assert fn in names



def header_constants():
    """Every integer #define GATO_* of the header, its value evaluated from the
    (parenthesised, unsigned-suffixed, multiplied) literal."""
    out = {}
    for name, expr in re.findall(r"^#define (GATO_\w+)[ \t]+([^/\n]+)", open(HEADER).read(), re.M):
        expr = re.sub(r"(\d+)u\b", r"\1", expr.strip())
        if re.fullmatch(r"[\d\s()*+-]+", expr):
            out[name] = eval(expr)  # digits, parentheses and arithmetic only
    return out


def test_binding_constants_equal_the_header():
    consts = header_constants()
    assert len(consts) >= 30, sorted(consts)
    missing = [k for k in consts if not hasattr(gato, k)]
    assert not missing, missing
    for k, v in consts.items():
        assert getattr(gato, k) == v, (k, getattr(gato, k), v)


def test_library_exports_every_declared_symbol(lib):
    missing = [fn for fn in declared_functions() if not hasattr(lib, fn)]
    assert not missing, missing


def test_default_params(lib):
    p = gato.default_params()
    assert p.pcg_eps == pytest.approx(1e-6)
    assert (p.pcg_max_iters, p.stop_rule, p.refine_steps, p.n_alpha, p.merit_threads) == (
        200, 0, 0, 8, 64)
    assert (p.beta, p.mu) == (2.0, 10.0)
    assert p.refine_eps == pytest.approx(0.1)
    assert p.merit_kernel == gato.GATO_MERIT_FUSED
    # the GATO documentation's policy: PCG below N = 256, the direct solve from it
    assert (p.linsys, p.bdsv_horizon) == (gato.GATO_LINSYS_AUTO, 256)


def test_default_sqp_params(lib):
    sp = gato.default_sqp_params()
    assert (sp.iters, sp.warm_start, sp.use_graph) == (10, 1, 1)
    assert (sp.rho_factor, sp.rho_max) == (10.0, 10.0)
    assert sp.rho_min == pytest.approx(1e-8)


def test_sqp_params_struct_matches_header():
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    body = re.search(r"typedef struct gato_sqp_params \{(.*?)\} gato_sqp_params;", text,
                     re.S).group(1)
    fields = re.findall(r"\b(int|float)\s+(\w+)\s*;", body)
    ctype = {"int": ctypes.c_int, "float": ctypes.c_float}
    assert [(name, ctype[t]) for t, name in fields] == list(gato.GatoSqpParams._fields_)


def test_params_struct_matches_header():
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    body = re.search(r"typedef struct gato_params \{(.*?)\} gato_params;", text, re.S).group(1)
    fields = re.findall(r"\b(int|float)\s+(\w+)\s*;", body)
    ctype = {"int": ctypes.c_int, "float": ctypes.c_float}
    assert [(name, ctype[t]) for t, name in fields] == list(gato.GatoParams._fields_)


def test_invalid_arguments_rejected_before_cuda(lib):
    h = ctypes.c_void_p()
    assert lib.gato_create(None, 1, 2, 3, 1) == gato.GATO_ERR_INVALID_ARG
    assert lib.gato_create(ctypes.byref(h), 0, 2, 3, 1) == gato.GATO_ERR_INVALID_ARG
    assert lib.gato_create(ctypes.byref(h), 1, 0, 3, 1) == gato.GATO_ERR_INVALID_ARG
    assert lib.gato_create(ctypes.byref(h), 1, 2, 0, 1) == gato.GATO_ERR_INVALID_ARG
    assert lib.gato_create(ctypes.byref(h), 1, 2, 3, 0) == gato.GATO_ERR_INVALID_ARG
    assert lib.gato_create(ctypes.byref(h), 1, 2, 65, 1) == gato.GATO_ERR_UNSUPPORTED
    assert lib.gato_create(ctypes.byref(h), 1, 2, 3, 65) == gato.GATO_ERR_UNSUPPORTED
    assert not h.value
    lib.gato_destroy(None)
    p = gato.default_params()
    assert lib.gato_set_timing(None, 1) == gato.GATO_ERR_INVALID_ARG
    assert lib.gato_set_pcg_kernel(None, 0) == gato.GATO_ERR_INVALID_ARG
    assert lib.gato_set_form_kernel(None, 0) == gato.GATO_ERR_INVALID_ARG
    assert lib.gato_set_bdsv_kernel(None, 0) == gato.GATO_ERR_INVALID_ARG
    assert lib.gato_get_stats(None, None) == gato.GATO_ERR_INVALID_ARG
    null = [None] * 8
    assert lib.gato_form_schur(None, *null, None, None) == gato.GATO_ERR_INVALID_ARG
    assert lib.gato_get_schur(None, *([None] * 5), None) == gato.GATO_ERR_INVALID_ARG
    assert lib.gato_pcg_solve(None, ctypes.byref(p), *([None] * 6), None) == gato.GATO_ERR_INVALID_ARG
    assert lib.gato_linesearch(None, ctypes.byref(p), *null, *([None] * 5), None) == gato.GATO_ERR_INVALID_ARG
    assert lib.gato_solve_kkt(None, ctypes.byref(p), *null, *([None] * 7), None) == gato.GATO_ERR_INVALID_ARG
    assert lib.gato_solve_kkt_host(None, ctypes.byref(p), *null, *([None] * 7), None) == gato.GATO_ERR_INVALID_ARG
    assert lib.gato_set_parts(None, 1) == gato.GATO_ERR_INVALID_ARG
    assert lib.gato_get_parts(None, None) == gato.GATO_ERR_INVALID_ARG
    assert lib.gato_apply_step(None, ctypes.byref(p), *([None] * 5), None) == gato.GATO_ERR_INVALID_ARG
    assert lib.gato_bdsv_solve(None, ctypes.byref(p), *([None] * 5), None) == gato.GATO_ERR_INVALID_ARG
    sp = gato.default_sqp_params()
    assert lib.gato_sqp_linear(None, ctypes.byref(p), ctypes.byref(sp), *null, *([None] * 7),
                               None) == gato.GATO_ERR_INVALID_ARG


def test_generator_is_deterministic_and_distributed():
    a = normals(123, 4, 100000)
    b = normals(123, 4, 100000)
    assert np.array_equal(a, b)
    assert abs(a.mean()) < 0.02 and abs(a.std() - 1) < 0.02
    u = uniforms(5, 1, 100000)
    assert u.min() > 0 and u.max() < 1 and abs(u.mean() - 0.5) < 0.01
    assert not np.array_equal(normals(1, 1, 10), normals(1, 2, 10))


@pytest.mark.parametrize("w", WORKLOADS, ids=lambda w: w.name)
def test_workload_shapes(w):
    b = make_batch(w, M=2)
    N, n, m = w.N, w.n, w.m
    assert b["Q"].shape == (2, N, n, n) and b["R"].shape == (2, N - 1, m, m)
    assert b["A"].shape == (2, N - 1, n, n) and b["B"].shape == (2, N - 1, n, m)
    assert b["q"].shape == (2, N, n) and b["r"].shape == (2, N - 1, m)
    assert b["e"].shape == (2, N - 1, n) and b["s0"].shape == (2, n)
    assert all(v.dtype == np.float32 for v in b.values())
    # per-solve seeds: solve 1 of a batch equals solve 0 of a batch starting there
    c = make_batch(w, M=1, first_solve=1)
    assert np.array_equal(b["Q"][1], c["Q"][0])
    assert np.linalg.eigvalsh(b["Q"][0].astype(np.float64)).min() > 0


def test_binding_argument_counts_match_header(lib):
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    for m in re.finditer(r"\b(gato_\w+)\s*\(([^)]*)\)\s*;", text):
        name, args = m.group(1), m.group(2).strip()
        count = 0 if args in ("", "void") else len(args.split(","))
        assert len(getattr(lib, name).argtypes) == count, name
