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


# --------------------------------------------------------------------------
# the binding's size checks (host side)
# --------------------------------------------------------------------------

def test_binding_sizes_follow_the_header_layouts():
    z = gato.sizes(3, 5, 4, 2, n_alpha=6)
    assert z["Q"] == 3 * 5 * 16 and z["R"] == 3 * 4 * 4 and z["A"] == 3 * 4 * 16
    assert z["B"] == 3 * 4 * 4 * 2 and z["e"] == 3 * 4 * 4 and z["s0"] == 3 * 4
    assert z["dX"] == 3 * 5 * 4 and z["dU"] == 3 * 4 * 2 and z["merit"] == 3 * 7
    # one knot: no controls, no couplings
    z1 = gato.sizes(2, 1, 4, 2)
    assert z1["R"] == z1["A"] == z1["B"] == z1["dU"] == 0


def test_binding_rejects_a_short_array_before_any_call():
    torch = pytest.importorskip("torch")
    t = torch.zeros(10)
    assert gato._host_ptr(t, what="Q", numel=10) is not None
    with pytest.raises(ValueError, match="Q holds 10 elements"):
        gato._host_ptr(t, what="Q", numel=11)
    with pytest.raises(ValueError, match="CUDA tensor"):
        gato._ptr(t, what="Q", numel=10)


def test_pcg_kernel_names_match_the_header():
    assert bench.PCG_KERNELS == {"auto": gato.GATO_PCG_AUTO, "generic": gato.GATO_PCG_GENERIC,
                                 "wide": gato.GATO_PCG_WIDE, "tile": gato.GATO_PCG_TILE,
                                 "rows": gato.GATO_PCG_ROWS, "quad": gato.GATO_PCG_QUAD}
