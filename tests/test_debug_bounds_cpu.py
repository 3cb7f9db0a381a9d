"""Host-side wiring of the checking build (GATO_DEBUG_BOUNDS).

The library built with -DGATO_DEBUG_BOUNDS=1 checks, in its kernels, the
indices and shared-memory layouts it derives and records GATO_STATUS_BOUNDS
in the call's status instead of making an access that would fall outside its
array.  These tests need no GPU: the environment switch selects the checking
library's path, its compile commands carry the flag and a separate object
directory, a translation unit with checks compiles with it, and the status
bit is the header's.  The GPU suite runs with GATO_DEBUG_BOUNDS=1 to show
that no check fires on any tested size (every GPU test asserts zero status).
"""
import os
import subprocess
import tempfile

import pytest

from trajectory_optimization_kkt_gb300 import _build, gato


def test_environment_selects_the_checking_library(monkeypatch):
    monkeypatch.delenv("GATO_DEBUG_BOUNDS", raising=False)
    assert not _build.debug_bounds_requested()
    assert gato.library_path() == _build.LIB_PATH
    monkeypatch.setenv("GATO_DEBUG_BOUNDS", "0")
    assert gato.library_path() == _build.LIB_PATH
    monkeypatch.setenv("GATO_DEBUG_BOUNDS", "1")
    assert _build.debug_bounds_requested()
    assert gato.library_path() == _build.LIB_PATH_BOUNDS
    assert _build.LIB_PATH_BOUNDS != _build.LIB_PATH


def test_compile_commands_carry_the_flag_only_in_the_checking_build():
    src = os.path.join(_build.CSRC, "merit.cu")
    plain = _build.compile_command(src, "x.o", debug_bounds=False)
    checking = _build.compile_command(src, "x.o", debug_bounds=True)
    assert "-DGATO_DEBUG_BOUNDS=1" not in plain
    assert "-DGATO_DEBUG_BOUNDS=1" in checking
    # the same architecture and optimisation otherwise
    assert [a for a in checking if a != "-DGATO_DEBUG_BOUNDS=1"] == plain


def test_status_bit_is_distinct_from_the_solver_bits():
    bits = [gato.GATO_STATUS_PCG_MAX_ITERS, gato.GATO_STATUS_NONPOSITIVE_PIVOT,
            gato.GATO_STATUS_LINESEARCH_FAILED, gato.GATO_STATUS_NONFINITE]
    assert gato.GATO_STATUS_BOUNDS == 16
    assert all(gato.GATO_STATUS_BOUNDS & b == 0 for b in bits)


def test_a_checked_translation_unit_compiles():
    """merit.cu with the checks compiled in (cross-compiled for sm_103a)."""
    try:
        _build._nvcc()
    except RuntimeError:
        pytest.skip("nvcc not available")
    with tempfile.TemporaryDirectory() as d:
        obj = os.path.join(d, "merit.o")
        cmd = _build.compile_command(os.path.join(_build.CSRC, "merit.cu"), obj,
                                     debug_bounds=True)
        res = subprocess.run(cmd, capture_output=True, text=True)
        assert res.returncode == 0, res.stderr
        assert os.path.getsize(obj) > 0
