"""Writes tests/golden/workload0_oracle.npz from the fp64 oracle alone.

Run from the repository root:  python tests/golden/make_golden.py
The stored values are the oracle's direct solution, PCG iteration count,
merit values and chosen step for solve 0 of workload 0 (M=1, N=16, n=14,
m=7), plus a few input arrays so that a change in the generator shows up.
"""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from trajectory_optimization_kkt_gb300.workloads import WORKLOADS, make_batch  # noqa: E402


def main():
    prob = oracle.solve_one(make_batch(WORKLOADS[0]), 0)
    dX, dU, lam = oracle.direct_solve(prob)
    out = oracle.solve_kkt(prob, 1e-6, 200)
    np.savez(os.path.join(os.path.dirname(os.path.abspath(__file__)), "workload0_oracle.npz"),
             in_Q=prob["Q"], in_q=prob["q"], in_A=prob["A"], in_s0=prob["s0"],
             lam=lam, dX=dX, dU=dU, pcg_iters=out["iters"], merit=out["merit"],
             best=out["best"])


if __name__ == "__main__":
    main()
