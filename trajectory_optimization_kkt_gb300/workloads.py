"""Seeded synthetic LQ subproblems for the batched KKT path.

This module holds only random-number generation and the workload recipes.  It
contains none of the method's arithmetic, so that both the CUDA path and the
fp64 oracle can be fed from it.

Generator
---------
Counter-based splitmix64 (Steele, Lea & Flood, "Fast splittable pseudorandom
number generators", OOPSLA 2014): output i of a stream with base state s is
``mix64(s + (i + 1) * 0x9E3779B97F4A7C15)``.  Uniforms take the top 53 bits,
offset by half an ulp so that they lie strictly inside (0, 1).  Normals come
from the Box-Muller transform (Box & Muller, 1958) on consecutive uniform
pairs.  Each named tensor of each solve gets its own stream, so every element
is a pure function of (seed, tensor, index) and generation is vectorised.
Values are drawn in float64 and rounded once to float32.

Workloads (GATO paper, Section II eq. (1) for the LQ data; sizes, scalings and
solver settings from the benchmark configurations)
-----------------------------------------------------------------------------
Per solve j of workload c the seed is ``1000 * c + j``.
  A_k = I + a_sigma * N(0,1)         B_k = b_sigma * N(0,1)
  Q_k = L L^T / n + 0.01 I           R_k = L L^T / m + 0.01 I,  L ~ N(0,1)
  q, r ~ N(0,1)    e_k ~ N(0, 0.01^2)    s0 ~ N(0, 0.1^2)
  optional: Q_k <- D Q_k D, R_k <- D R_k D with D = diag(sqrt(w)),
            log10 w ~ U(-2, 2)          (diagonal log-uniform scaling)
  optional: Q_{N-1} <- 10 Q_{N-1}       (heavier terminal cost)
"""
from __future__ import annotations

import dataclasses
from typing import Dict

import numpy as np

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

# one stream per named tensor
_TAGS = {"LQ": 1, "LR": 2, "A": 3, "B": 4, "q": 5, "r": 6, "e": 7, "s0": 8,
         "wQ": 9, "wR": 10}


def _mix64(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def _stream_base(seed: int, tag: int) -> np.uint64:
    s = np.array([(int(seed) * 0x100000001B3 + tag * 0x51ED270B27D6F9C3) & (2**64 - 1)],
                 dtype=np.uint64)
    return _mix64(s)[0]


def uniforms(seed: int, tag: int, count: int) -> np.ndarray:
    """``count`` float64 uniforms in (0, 1) from stream (seed, tag)."""
    i = np.arange(1, count + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        x = _mix64(_stream_base(seed, tag) + i * _GAMMA)
    return ((x >> np.uint64(11)).astype(np.float64) + 0.5) * (2.0 ** -53)


def normals(seed: int, tag: int, count: int) -> np.ndarray:
    """``count`` float64 standard normals from stream (seed, tag), Box-Muller."""
    pairs = (count + 1) // 2
    u = uniforms(seed, tag, 2 * pairs).reshape(pairs, 2)
    rad = np.sqrt(-2.0 * np.log(u[:, 0]))
    ang = 2.0 * np.pi * u[:, 1]
    z = np.empty((pairs, 2))
    z[:, 0] = rad * np.cos(ang)
    z[:, 1] = rad * np.sin(ang)
    return z.reshape(-1)[:count]


@dataclasses.dataclass(frozen=True)
class Workload:
    """One benchmark workload: sizes, generator settings and solver settings."""
    index: int
    name: str
    M: int
    N: int
    n: int
    m: int
    a_sigma: float = 0.01
    b_sigma: float = 0.01
    log_scale: bool = False
    terminal_scale: float = 1.0
    pcg_eps: float = 1e-6
    pcg_max_iters: int = 200
    n_alpha: int = 8
    beta: float = 2.0
    mu: float = 10.0
    # rounds of KKT iterative refinement (compensated residual), each
    # correction solved by PCG to refine_eps or by substitution with a direct
    # factorisation of the same S (refine_solver): fp32 formation alone leaves
    # dX 2e-4 to 1e-2 from the exact solution on these workloads.  The setting
    # is the fastest of one or two rounds, PCG corrections at 0.25 / 0.1 /
    # 0.01 or direct ones, whose worst dX and worst dU error over the
    # workload's whole batch stay below 3/4 of the 1e-4 parity tolerance
    refine_steps: int = 1
    refine_eps: float = 0.1
    # arithmetic of the main PCG solve: 0 fp32, 1 double-float (the value of
    # GATO_PCG_PRECISION_FF), for the workloads whose stated iteration cap
    # fp32 PCG cannot meet
    pcg_precision: int = 0
    # how the refinement corrections are solved: 0 with the main solve's
    # solver, 1 by substitution with a direct factorisation of the same S
    # (the value of GATO_REFINE_SOLVER_DIRECT)
    refine_solver: int = 0

    def solver_settings(self) -> Dict[str, float]:
        """The gato_params fields this workload sets (keyword arguments of
        gato.default_params)."""
        return dict(pcg_eps=self.pcg_eps, pcg_max_iters=self.pcg_max_iters,
                    n_alpha=self.n_alpha, beta=self.beta, mu=self.mu,
                    refine_steps=self.refine_steps, refine_eps=self.refine_eps,
                    pcg_precision=self.pcg_precision, refine_solver=self.refine_solver)

    def with_batch(self, M: int, N: int | None = None) -> "Workload":
        return dataclasses.replace(self, M=M, N=self.N if N is None else N)


# Iteration caps: workloads 0 and 2 state theirs (200, 500).  fp64 PCG needs
# 180 and up to 487 iterations there, fp32 PCG 227 and up to 504, so these two
# run the main solve in double-float arithmetic (about 48 bits: 186 and up to
# 491).  The others state only eps = 1e-6; their cap is set high enough for
# fp32 PCG to reach it.  Refinement by the rule above: one direct correction
# for workloads 0, 1, 2 and 4 (dX about 1e-7; its factorisation runs beside
# the main PCG on the SMs that solve leaves idle, which made it the faster
# choice for workloads 0 and 4 too, against PCG corrections at 0.25 and 0.1);
# two direct ones for workload 3 (diagonal scaling over four decades: one
# leaves dX at 8.4e-5, two at 3e-6).
WORKLOADS = [
    Workload(0, "M1_N16_n14_m7", 1, 16, 14, 7, pcg_max_iters=200, pcg_precision=1,
             refine_solver=1),
    Workload(1, "M16_N32_n12_m6", 16, 32, 12, 6, pcg_max_iters=1000, refine_solver=1),
    Workload(2, "M64_N64_n14_m7_A05_QN10", 64, 64, 14, 7, a_sigma=0.05,
             terminal_scale=10.0, pcg_max_iters=500, pcg_precision=1, refine_solver=1),
    Workload(3, "M128_N16_n36_m12_logscaled", 128, 16, 36, 12, b_sigma=0.05,
             log_scale=True, pcg_max_iters=4000, refine_steps=2, refine_solver=1),
    Workload(4, "M256_N128_n14_m7", 256, 128, 14, 7, pcg_max_iters=1000, refine_solver=1),
]


def _spd_blocks(seed: int, tag: int, count: int, d: int) -> np.ndarray:
    L = normals(seed, tag, count * d * d).reshape(count, d, d)
    return L @ L.transpose(0, 2, 1) / d + 0.01 * np.eye(d)


def _log_scale(Mx: np.ndarray, seed: int, tag: int) -> np.ndarray:
    count, d, _ = Mx.shape
    w = 10.0 ** (-2.0 + 4.0 * uniforms(seed, tag, count * d).reshape(count, d))
    s = np.sqrt(w)
    return s[:, :, None] * Mx * s[:, None, :]


def make_solve(w: Workload, seed: int, N: int | None = None) -> Dict[str, np.ndarray]:
    """One solve's LQ data (float32) for workload ``w`` with the given seed."""
    N = w.N if N is None else N
    n, m = w.n, w.m
    K = N - 1
    Q = _spd_blocks(seed, _TAGS["LQ"], N, n)
    R = _spd_blocks(seed, _TAGS["LR"], K, m)
    if w.log_scale:
        Q = _log_scale(Q, seed, _TAGS["wQ"])
        R = _log_scale(R, seed, _TAGS["wR"])
    Q[N - 1] *= w.terminal_scale
    A = np.eye(n) + w.a_sigma * normals(seed, _TAGS["A"], K * n * n).reshape(K, n, n)
    B = w.b_sigma * normals(seed, _TAGS["B"], K * n * m).reshape(K, n, m)
    q = normals(seed, _TAGS["q"], N * n).reshape(N, n)
    r = normals(seed, _TAGS["r"], K * m).reshape(K, m)
    e = 0.01 * normals(seed, _TAGS["e"], K * n).reshape(K, n)
    s0 = 0.1 * normals(seed, _TAGS["s0"], n)
    f32 = lambda x: np.ascontiguousarray(x, dtype=np.float32)
    return dict(Q=f32(Q), R=f32(R), q=f32(q), r=f32(r), A=f32(A), B=f32(B),
                e=f32(e), s0=f32(s0))


def make_batch(w: Workload, M: int | None = None, N: int | None = None,
               first_solve: int = 0) -> Dict[str, np.ndarray]:
    """Batch of ``M`` solves, stacked on a leading axis, solve j seeded 1000*index + j."""
    M = w.M if M is None else M
    solves = [make_solve(w, 1000 * w.index + first_solve + j, N) for j in range(M)]
    return {k: np.ascontiguousarray(np.stack([s[k] for s in solves])) for k in solves[0]}


def random_lq(M: int, N: int, n: int, m: int, seed: int, **kw) -> Dict[str, np.ndarray]:
    """Batch with arbitrary sizes (tests), generated like workload 0."""
    w = Workload(99, "custom", M, N, n, m, **kw)
    solves = [make_solve(w, seed + j) for j in range(M)]
    return {k: np.ascontiguousarray(np.stack([s[k] for s in solves])) for k in solves[0]}


# ---------------------------------------------------------------------------
# linear-model problems for the SQP loop: minimise the quadratic cost subject
# to x_0 = xs and x_{k+1} = A_k x_k + B_k u_k + c_k.  The affine term c and the
# initial state xs are the generator's e and s0 draws; at the zero trajectory
# the SQP loop's first subproblem is therefore exactly the workload's LQ
# subproblem.
# ---------------------------------------------------------------------------

def as_linear_model(batch: Dict[str, np.ndarray]) -> Dict[str, np.ndarray]:
    """An LQ batch read as linear-model problems (e -> c, s0 -> xs)."""
    out = {k: v for k, v in batch.items() if k not in ("e", "s0")}
    out["c"], out["xs"] = batch["e"], batch["s0"]
    return out


def linear_models(M: int, N: int, n: int, m: int, seed: int, **kw) -> Dict[str, np.ndarray]:
    """``M`` linear-model problems of arbitrary sizes, generated like random_lq."""
    return as_linear_model(random_lq(M, N, n, m, seed, **kw))


def replicate(problem: Dict[str, np.ndarray], M: int) -> Dict[str, np.ndarray]:
    """One problem (arrays without the batch axis) repeated ``M`` times: the
    batch of a sweep over a solver parameter such as the damping rho."""
    return {k: np.repeat(np.asarray(v)[None], M, axis=0) for k, v in problem.items()}


def rho_logspace(M: int, lo: float = 1e-8, hi: float = 10.0) -> np.ndarray:
    """Initial damping of a batch of M solves of one problem: log-spaced from
    lo to hi (GATO paper Sec. IV-C); a single solve starts at 0.1 there."""
    if M == 1:
        return np.array([0.1], dtype=np.float32)
    return np.logspace(np.log10(lo), np.log10(hi), M).astype(np.float32)
