"""Thin ctypes binding of the C ABI in include/gato.h.

Argument marshalling only: every step of the computation runs in the CUDA
library (``_build/libgato.so``).  Tensors must be contiguous float32 (int32 /
uint32-as-int32 for iters, best and status) CUDA tensors on the handle's
device.  If the library is missing, loading raises instead of falling back.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

from . import _build

GATO_OK = 0
GATO_ERR_INVALID_ARG = -1
GATO_ERR_UNSUPPORTED = -2
GATO_ERR_CUDA = -3
GATO_ERR_NO_MEMORY = -4

GATO_STATUS_PCG_MAX_ITERS = 1
GATO_STATUS_NONPOSITIVE_PIVOT = 2
GATO_STATUS_LINESEARCH_FAILED = 4
GATO_STATUS_NONFINITE = 8
GATO_STATUS_BOUNDS = 16

GATO_PCG_AUTO = 0
GATO_PCG_GENERIC = 1
GATO_PCG_WIDE = 2
GATO_PCG_TILE = 3
GATO_PCG_ROWS = 4
GATO_PCG_QUAD = 5
GATO_PCG_CLUSTER = 6  # reported in the stats only
GATO_PCG_DOUBLE_FLOAT = 7  # reported in the stats only
GATO_MAX_PARTS = 8
GATO_MAX_STATE = 64
GATO_MAX_CONTROL = 64
GATO_MAX_ALPHA = 31
GATO_NOALLOC_MAX_BYTES = 32 * 1024 * 1024

GATO_LINSYS_AUTO = 0
GATO_LINSYS_PCG = 1
GATO_LINSYS_BDSV = 2
GATO_LINSYS_BDSV_CHRONO = 3

GATO_BDSV_KERNEL_AUTO = 0
GATO_BDSV_KERNEL_SHARED = 1

GATO_FORM_AUTO = 0
GATO_FORM_SHARED = 1

GATO_MERIT_FUSED = 0
GATO_MERIT_PER_CANDIDATE = 1

GATO_PCG_PRECISION_FP32 = 0
GATO_PCG_PRECISION_FF = 1

GATO_REFINE_SOLVER_SAME = 0
GATO_REFINE_SOLVER_DIRECT = 1

GATO_STOP_RESIDUAL = 0
GATO_STOP_PRECOND = 1
GATO_STOP_SCALED = 2

_ERRORS = {GATO_ERR_INVALID_ARG: "invalid argument", GATO_ERR_UNSUPPORTED: "unsupported sizes",
           GATO_ERR_CUDA: "CUDA error", GATO_ERR_NO_MEMORY: "out of device memory"}


class GatoParams(ctypes.Structure):
    _fields_ = [("pcg_eps", ctypes.c_float), ("pcg_max_iters", ctypes.c_int),
                ("stop_rule", ctypes.c_int), ("refine_steps", ctypes.c_int),
                ("n_alpha", ctypes.c_int), ("beta", ctypes.c_float), ("mu", ctypes.c_float),
                ("merit_threads", ctypes.c_int), ("refine_eps", ctypes.c_float),
                ("merit_kernel", ctypes.c_int), ("linsys", ctypes.c_int),
                ("bdsv_horizon", ctypes.c_int), ("pcg_precision", ctypes.c_int),
                ("refine_solver", ctypes.c_int)]


class GatoSqpParams(ctypes.Structure):
    _fields_ = [("iters", ctypes.c_int), ("rho_factor", ctypes.c_float),
                ("rho_min", ctypes.c_float), ("rho_max", ctypes.c_float),
                ("warm_start", ctypes.c_int), ("use_graph", ctypes.c_int)]


class GatoStats(ctypes.Structure):
    _fields_ = [("form_us", ctypes.c_float), ("pcg_us", ctypes.c_float),
                ("refine_us", ctypes.c_float), ("merit_us", ctypes.c_float),
                ("total_us", ctypes.c_float), ("pcg_kernel", ctypes.c_int),
                ("refine_kernel", ctypes.c_int)]


class GatoError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn} failed: {_ERRORS.get(code, 'error')} ({code})")
        self.code = code


_lib = None


def library_path() -> str:
    """libgato.so, or libgato_bounds.so when GATO_DEBUG_BOUNDS=1 is set."""
    return _build.library_path()


def load(path: Optional[str] = None):
    """Load the library (built by __graft_entry__.build()); raises if absent."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or library_path()
    if not os.path.exists(path):
        raise RuntimeError(f"CUDA library not built: {path} is missing (run build())")
    lib = ctypes.CDLL(path)
    vp, ip, fp = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    P = ctypes.POINTER(GatoParams)
    lib.gato_default_params.argtypes = [P]
    lib.gato_default_params.restype = None
    SP = ctypes.POINTER(GatoSqpParams)
    lib.gato_default_sqp_params.argtypes = [SP]
    lib.gato_default_sqp_params.restype = None
    lib.gato_sqp_linear.argtypes = [vp, P, SP] + [vp] * 8 + [vp] * 7 + [vp]
    lib.gato_create.argtypes = [ctypes.POINTER(vp), ip, ip, ip, ip]
    lib.gato_destroy.argtypes = [vp]
    lib.gato_destroy.restype = None
    lib.gato_set_timing.argtypes = [vp, ip]
    lib.gato_set_pcg_kernel.argtypes = [vp, ip]
    lib.gato_set_form_kernel.argtypes = [vp, ip]
    lib.gato_set_bdsv_kernel.argtypes = [vp, ip]
    lib.gato_get_stats.argtypes = [vp, ctypes.POINTER(GatoStats)]
    lib.gato_form_schur.argtypes = [vp] + [vp] * 8 + [vp, vp]
    lib.gato_get_schur.argtypes = [vp] + [vp] * 5 + [vp]
    lib.gato_pcg_solve.argtypes = [vp, P] + [vp] * 6 + [vp]
    lib.gato_bdsv_solve.argtypes = [vp, P] + [vp] * 5 + [vp]
    lib.gato_linesearch.argtypes = [vp, P] + [vp] * 8 + [vp] * 5 + [vp]
    lib.gato_solve_kkt.argtypes = [vp, P] + [vp] * 8 + [vp] * 7 + [vp]
    lib.gato_solve_kkt_host.argtypes = [vp, P] + [vp] * 8 + [vp] * 7 + [vp]
    lib.gato_set_parts.argtypes = [vp, ip]
    lib.gato_get_parts.argtypes = [vp, ctypes.POINTER(ctypes.c_int)]
    lib.gato_apply_step.argtypes = [vp, P] + [vp] * 5 + [vp]
    lib.gato_solve_kkt_noalloc.argtypes = [P, ip, ip, ip, ip] + [vp] * 8 + [vp] * 7 + [vp]
    lib.gato_probe_fp32.argtypes = [ip, ip, ip, ip, vp, vp]
    lib.gato_probe_fp32.restype = ctypes.c_longlong
    for fn in ("gato_create", "gato_set_timing", "gato_set_pcg_kernel", "gato_set_form_kernel",
               "gato_set_bdsv_kernel", "gato_get_stats", "gato_form_schur",
               "gato_get_schur", "gato_pcg_solve", "gato_bdsv_solve", "gato_linesearch",
               "gato_solve_kkt", "gato_apply_step", "gato_solve_kkt_noalloc",
               "gato_sqp_linear"):
        getattr(lib, fn).restype = ctypes.c_int
    _lib = lib
    return lib


def _check(fn: str, rc: int):
    if rc != GATO_OK:
        raise GatoError(fn, rc)


def default_params(**overrides) -> GatoParams:
    p = GatoParams()
    load().gato_default_params(ctypes.byref(p))
    for k, v in overrides.items():
        setattr(p, k, v)
    return p


def default_sqp_params(**overrides) -> GatoSqpParams:
    sp = GatoSqpParams()
    load().gato_default_sqp_params(ctypes.byref(sp))
    for k, v in overrides.items():
        setattr(sp, k, v)
    return sp


def _check_numel(t, numel, what):
    # the library reads or writes numel elements from the pointer: a shorter
    # tensor would be overrun
    if numel is not None and t.numel() < numel:
        raise ValueError(f"{what} holds {t.numel()} elements, the call needs {numel}")


def _ptr(t, dtype=None, what="tensor", numel=None):
    """Device pointer of a contiguous CUDA tensor of at least numel elements
    (None -> NULL)."""
    if t is None:
        return None
    import torch
    if not t.is_cuda:
        raise ValueError(f"{what} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{what} must be contiguous")
    want = dtype or torch.float32
    if t.dtype != want:
        raise ValueError(f"{what} must be {want}, got {t.dtype}")
    _check_numel(t, numel, what)
    return ctypes.c_void_p(t.data_ptr())


def _host_ptr(t, dtype=None, what="tensor", numel=None):
    """Host pointer of a contiguous CPU tensor of at least numel elements
    (None -> NULL); pin it for copies that overlap the solve."""
    if t is None:
        return None
    import torch
    if t.is_cuda:
        raise ValueError(f"{what} must be a CPU tensor")
    if not t.is_contiguous():
        raise ValueError(f"{what} must be contiguous")
    want = dtype or torch.float32
    if t.dtype != want:
        raise ValueError(f"{what} must be {want}, got {t.dtype}")
    _check_numel(t, numel, what)
    return ctypes.c_void_p(t.data_ptr())


def sizes(M: int, N: int, n: int, m: int, n_alpha: int = 8) -> dict:
    """Elements of every array argument of the entry points, by name, for a
    batch of M solves (the layouts include/gato.h gives)."""
    K = max(N - 1, 0)
    return dict(Q=M * N * n * n, R=M * K * m * m, q=M * N * n, r=M * K * m, A=M * K * n * n,
                B=M * K * n * m, e=M * K * n, s0=M * n, c=M * K * n, xs=M * n,
                dX=M * N * n, dU=M * K * m, lam=M * N * n, lambda0=M * N * n, iters=M,
                merit=M * (n_alpha + 1), best=M, status=M, X=M * N * n, U=M * K * m, rho=M,
                S_diag=M * N * n * n, S_off=M * K * n * n, gamma=M * N * n,
                Phi_diag=M * N * n * n, Phi_off=M * K * n * n)


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


_LQ = ("Q", "R", "q", "r", "A", "B", "e", "s0")
_MODEL = ("Q", "R", "q", "r", "A", "B", "c", "xs")


class Solver:
    """Owns a gato_handle; methods mirror the C entry points one to one."""

    def __init__(self, M: int, N: int, n: int, m: int):
        import torch
        self.lib = load()
        self.M, self.N, self.n, self.m = M, N, n, m
        self.device = torch.cuda.current_device()
        h = ctypes.c_void_p()
        _check("gato_create", self.lib.gato_create(ctypes.byref(h), M, N, n, m))
        self.h = h

    def close(self):
        if getattr(self, "h", None):
            self.lib.gato_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    # -- helpers --------------------------------------------------------------
    def _sz(self, params=None):
        return sizes(self.M, self.N, self.n, self.m, params.n_alpha if params else 8)

    def _lq(self, prob, keys=_LQ):
        sz = self._sz()
        return [_ptr(prob.get(k), what=k, numel=sz[k]) for k in keys]

    # -- entry points ---------------------------------------------------------
    def set_timing(self, on: bool):
        _check("gato_set_timing", self.lib.gato_set_timing(self.h, 1 if on else 0))

    def set_pcg_kernel(self, kind: int):
        _check("gato_set_pcg_kernel", self.lib.gato_set_pcg_kernel(self.h, kind))

    def set_bdsv_kernel(self, kind: int):
        _check("gato_set_bdsv_kernel", self.lib.gato_set_bdsv_kernel(self.h, kind))

    def set_form_kernel(self, kind: int):
        _check("gato_set_form_kernel", self.lib.gato_set_form_kernel(self.h, kind))

    def get_stats(self) -> GatoStats:
        s = GatoStats()
        _check("gato_get_stats", self.lib.gato_get_stats(self.h, ctypes.byref(s)))
        return s

    def form_schur(self, prob, status, stream=None):
        import torch
        _check("gato_form_schur", self.lib.gato_form_schur(
            self.h, *self._lq(prob), _ptr(status, torch.int32, "status"), _stream(stream)))

    def get_schur(self, S_diag=None, S_off=None, gamma=None, Phi_diag=None, Phi_off=None,
                  stream=None):
        z = self._sz()
        _check("gato_get_schur", self.lib.gato_get_schur(
            self.h, _ptr(S_diag, what="S_diag", numel=z["S_diag"]),
            _ptr(S_off, what="S_off", numel=z["S_off"]),
            _ptr(gamma, what="gamma", numel=z["gamma"]),
            _ptr(Phi_diag, what="Phi_diag", numel=z["Phi_diag"]),
            _ptr(Phi_off, what="Phi_off", numel=z["Phi_off"]), _stream(stream)))

    def pcg_solve(self, params, lam, dX, dU, iters, status, lambda0=None, stream=None):
        import torch
        z = self._sz(params)
        _check("gato_pcg_solve", self.lib.gato_pcg_solve(
            self.h, ctypes.byref(params), _ptr(lambda0, what="lambda0", numel=z["lambda0"]),
            _ptr(lam, what="lam", numel=z["lam"]), _ptr(dX, what="dX", numel=z["dX"]),
            _ptr(dU, what="dU", numel=z["dU"]),
            _ptr(iters, torch.int32, "iters", z["iters"]),
            _ptr(status, torch.int32, "status", z["status"]), _stream(stream)))

    def bdsv_solve(self, params, lam, dX, dU, iters, status, stream=None):
        import torch
        z = self._sz(params)
        _check("gato_bdsv_solve", self.lib.gato_bdsv_solve(
            self.h, ctypes.byref(params), _ptr(lam, what="lam", numel=z["lam"]),
            _ptr(dX, what="dX", numel=z["dX"]), _ptr(dU, what="dU", numel=z["dU"]),
            _ptr(iters, torch.int32, "iters", z["iters"]),
            _ptr(status, torch.int32, "status", z["status"]), _stream(stream)))

    def linesearch(self, params, prob, dX, dU, merit, best, status, stream=None):
        import torch
        z = self._sz(params)
        _check("gato_linesearch", self.lib.gato_linesearch(
            self.h, ctypes.byref(params), *self._lq(prob), _ptr(dX, what="dX", numel=z["dX"]),
            _ptr(dU, what="dU", numel=z["dU"]), _ptr(merit, what="merit", numel=z["merit"]),
            _ptr(best, torch.int32, "best", z["best"]),
            _ptr(status, torch.int32, "status", z["status"]), _stream(stream)))

    def solve_kkt(self, params, prob, dX, dU, lam, iters, merit, best, status, stream=None):
        import torch
        z = self._sz(params)
        _check("gato_solve_kkt", self.lib.gato_solve_kkt(
            self.h, ctypes.byref(params), *self._lq(prob), _ptr(dX, what="dX", numel=z["dX"]),
            _ptr(dU, what="dU", numel=z["dU"]), _ptr(lam, what="lam", numel=z["lam"]),
            _ptr(iters, torch.int32, "iters", z["iters"]),
            _ptr(merit, what="merit", numel=z["merit"]),
            _ptr(best, torch.int32, "best", z["best"]),
            _ptr(status, torch.int32, "status", z["status"]), _stream(stream)))

    def set_parts(self, parts: int):
        _check("gato_set_parts", self.lib.gato_set_parts(self.h, parts))

    def get_parts(self) -> int:
        v = ctypes.c_int(0)
        _check("gato_get_parts", self.lib.gato_get_parts(self.h, ctypes.byref(v)))
        return v.value

    def solve_kkt_host(self, params, prob, dX, dU, lam, iters, merit, best, status,
                       stream=None):
        """gato_solve_kkt_host: every array is a (preferably pinned) CPU
        tensor; synchronise the stream before reading the outputs."""
        import torch
        z = self._sz(params)
        _check("gato_solve_kkt_host", self.lib.gato_solve_kkt_host(
            self.h, ctypes.byref(params),
            *[_host_ptr(prob.get(k), what=k, numel=z[k]) for k in _LQ],
            _host_ptr(dX, what="dX", numel=z["dX"]), _host_ptr(dU, what="dU", numel=z["dU"]),
            _host_ptr(lam, what="lam", numel=z["lam"]),
            _host_ptr(iters, torch.int32, "iters", z["iters"]),
            _host_ptr(merit, what="merit", numel=z["merit"]),
            _host_ptr(best, torch.int32, "best", z["best"]),
            _host_ptr(status, torch.int32, "status", z["status"]), _stream(stream)))

    def sqp_linear(self, params, sqp_params, model, X, U, lam, rho, merit_hist, status,
                   iters_hist=None, stream=None):
        """gato_sqp_linear: model holds Q, R, q, r, A, B, c, xs (CUDA tensors);
        X, U, lam and rho are updated in place."""
        import torch
        z = self._sz(params)
        _check("gato_sqp_linear", self.lib.gato_sqp_linear(
            self.h, ctypes.byref(params), ctypes.byref(sqp_params), *self._lq(model, _MODEL),
            _ptr(X, what="X", numel=z["X"]), _ptr(U, what="U", numel=z["U"]),
            _ptr(lam, what="lam", numel=z["lam"]), _ptr(rho, what="rho", numel=z["rho"]),
            _ptr(merit_hist, what="merit_hist", numel=self.M * (sqp_params.iters + 1)),
            _ptr(iters_hist, torch.int32, "iters_hist", self.M * sqp_params.iters),
            _ptr(status, torch.int32, "status", z["status"]),
            _stream(stream)))

    def apply_step(self, params, best, dX, dU, X, U, stream=None):
        import torch
        z = self._sz(params)
        _check("gato_apply_step", self.lib.gato_apply_step(
            self.h, ctypes.byref(params), _ptr(best, torch.int32, "best", z["best"]),
            _ptr(dX, what="dX", numel=z["dX"]), _ptr(dU, what="dU", numel=z["dU"]),
            _ptr(X, what="X", numel=z["X"]), _ptr(U, what="U", numel=z["U"]), _stream(stream)))

    # -- convenience ------------------------------------------------------------
    def outputs(self, n_alpha: int = 8):
        """Freshly allocated output tensors for solve_kkt (status zeroed)."""
        import torch
        M, N, n, m = self.M, self.N, self.n, self.m
        dev = torch.device("cuda", self.device)
        f = dict(device=dev, dtype=torch.float32)
        return dict(dX=torch.empty(M, N, n, **f), dU=torch.empty(M, max(N - 1, 0), m, **f),
                    lam=torch.empty(M, N, n, **f),
                    iters=torch.zeros(M, device=dev, dtype=torch.int32),
                    merit=torch.empty(M, n_alpha + 1, **f),
                    best=torch.empty(M, device=dev, dtype=torch.int32),
                    status=torch.zeros(M, device=dev, dtype=torch.int32))

    def host_outputs(self, n_alpha: int = 8):
        """Pinned CPU output tensors for solve_kkt_host (status zeroed)."""
        import torch
        M, N, n, m = self.M, self.N, self.n, self.m
        f = dict(dtype=torch.float32, pin_memory=True)
        i = dict(dtype=torch.int32, pin_memory=True)
        return dict(dX=torch.empty(M, N, n, **f), dU=torch.empty(M, max(N - 1, 0), m, **f),
                    lam=torch.empty(M, N, n, **f), iters=torch.zeros(M, **i),
                    merit=torch.empty(M, n_alpha + 1, **f), best=torch.empty(M, **i),
                    status=torch.zeros(M, **i))


def to_host(prob):
    """numpy workload dict -> contiguous pinned float32 CPU tensors."""
    import torch
    return {k: torch.as_tensor(v, dtype=torch.float32).contiguous().pin_memory()
            for k, v in prob.items()}


def solve_kkt_noalloc(params, prob, dX, dU, lam, iters, merit, best, status, stream=None,
                      dims=None):
    """gato_solve_kkt_noalloc: the whole solve with the library's static scratch
    (no handle, no device allocation by the library).  dims = (M, N, n, m);
    by default read from the shapes of Q and B (give it when B is None)."""
    import torch
    if dims is None:
        M, N, n = prob["Q"].shape[:3]
        m = prob["B"].shape[-1]
    else:
        M, N, n, m = dims
    z = sizes(M, N, n, m, params.n_alpha)
    _check("gato_solve_kkt_noalloc", load().gato_solve_kkt_noalloc(
        ctypes.byref(params), M, N, n, m,
        *[_ptr(prob.get(k), what=k, numel=z[k]) for k in _LQ],
        _ptr(dX, what="dX", numel=z["dX"]), _ptr(dU, what="dU", numel=z["dU"]),
        _ptr(lam, what="lam", numel=z["lam"]), _ptr(iters, torch.int32, "iters", z["iters"]),
        _ptr(merit, what="merit", numel=z["merit"]), _ptr(best, torch.int32, "best", z["best"]),
        _ptr(status, torch.int32, "status", z["status"]), _stream(stream)))


def to_device(prob, device="cuda"):
    """numpy workload dict -> contiguous float32 CUDA tensors."""
    import torch
    return {k: torch.as_tensor(v, dtype=torch.float32).contiguous().to(device)
            for k, v in prob.items()}


def probe_fp32(packed: bool, blocks: int, threads: int, trips: int, sink, stream=None) -> int:
    """Launch the fp32 FMA throughput probe (gato_probe_fp32) on ``stream``
    (default: torch's current stream); returns the launch's flops."""
    import torch
    st = stream if stream is not None else torch.cuda.current_stream().cuda_stream
    rc = load().gato_probe_fp32(int(bool(packed)), int(blocks), int(threads), int(trips),
                                _ptr(sink, what="sink"), st)
    if rc < 0:
        raise GatoError("gato_probe_fp32", int(rc))
    return int(rc)
