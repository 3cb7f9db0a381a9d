"""bench.py's host-side pieces, without a GPU: the script loads and parses
its arguments, the kernel labels come from the library's reported kernels,
and the launch count per call follows the solver settings."""
import os
import subprocess
import sys
import types

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from trajectory_optimization_kkt_gb300 import gato  # noqa: E402


def test_bench_loads_and_parses_its_arguments():
    res = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--help"],
                         capture_output=True, text=True, cwd=ROOT)
    assert res.returncode == 0, res.stderr
    for flag in ("--gpus", "--steps", "--warmup", "--impl", "--pcg-kernel-sweep", "--workloads"):
        assert flag in res.stdout


def _stats(main, refine):
    return types.SimpleNamespace(pcg_kernel=main, refine_kernel=refine)


@pytest.mark.parametrize("main,refine,label", [
    (gato.GATO_PCG_WIDE, gato.GATO_PCG_WIDE, "k_pcg_wide"),
    (gato.GATO_PCG_QUAD, 0, "k_pcg_quad"),
    (gato.GATO_PCG_ROWS, gato.GATO_PCG_ROWS, "k_pcg_rows"),
    (gato.GATO_PCG_CLUSTER, gato.GATO_PCG_CLUSTER, "k_pcg_cluster"),
    (0, 0, "none"),
])
def test_kernel_labels_follow_the_reported_kernels(main, refine, label):
    assert bench._pcg_kernel_label(_stats(main, refine), 256, 128, 14, 152) == label


def test_double_float_label_names_the_cluster_form_and_the_corrections():
    ff = gato.GATO_PCG_DOUBLE_FLOAT
    # one solve of 16 knots: one CTA (fewer than 256 rows per CTA of a pair)
    assert bench._pcg_kernel_label(_stats(ff, gato.GATO_PCG_QUAD), 1, 16, 14, 152) == \
        "k_pcg_ff + k_pcg_quad"
    # 64 solves of 64 knots on 152 SMs: a cluster of two CTAs per solve
    assert bench._pcg_kernel_label(_stats(ff, 0), 64, 64, 14, 152) == "k_pcg_ff_cluster<2>"


def test_launches_per_call():
    assert bench.launches_per_solve("pcg", 0) == 6
    assert bench.launches_per_solve("pcg", 1) == 10
    assert bench.launches_per_solve("pcg", 1, refine_solver=1) == 11
    assert bench.launches_per_solve("pcg", 2, refine_solver=1) == 15
    assert bench.launches_per_solve("bdsv", 1) == 11
