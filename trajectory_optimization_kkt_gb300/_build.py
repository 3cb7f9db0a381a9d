"""Compiles the CUDA library (csrc/*.cu) into _build/libgato.so with nvcc.

One translation unit per source file, compiled in parallel for sm_103a only,
then linked into a shared library with the CUDA runtime linked statically.

With the environment variable GATO_DEBUG_BOUNDS=1 the library is also built
with -DGATO_DEBUG_BOUNDS=1 into _build/libgato_bounds.so (objects in
_build/obj_bounds), and library_path() names that one, so that the binding
loads it: its kernels check their indices and shared-memory layouts and
record GATO_STATUS_BOUNDS instead of making the access (a stand-in for a
memory checker; it never traps).
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT_DIR = os.path.join(PKG, "_build")
LIB_PATH = os.path.join(OUT_DIR, "libgato.so")
LIB_PATH_BOUNDS = os.path.join(OUT_DIR, "libgato_bounds.so")
BOUNDS_FLAGS = ["-DGATO_DEBUG_BOUNDS=1"]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CFLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE,
                 "-I", CSRC]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libgato")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(
        os.path.join(INCLUDE, "*.h"))


def debug_bounds_requested() -> bool:
    """GATO_DEBUG_BOUNDS=1 in the environment selects the checking build."""
    return os.environ.get("GATO_DEBUG_BOUNDS", "0") not in ("", "0")


def library_path(debug_bounds=None) -> str:
    if debug_bounds is None:
        debug_bounds = debug_bounds_requested()
    return LIB_PATH_BOUNDS if debug_bounds else LIB_PATH


def compile_command(src: str, obj: str, debug_bounds: bool = False, extra_flags=()):
    """The nvcc command line of one translation unit."""
    flags = list(CFLAGS) + (BOUNDS_FLAGS if debug_bounds else []) + list(extra_flags)
    return [_nvcc(), *flags, "-c", src, "-o", obj]


def up_to_date(debug_bounds: bool = False) -> bool:
    path = library_path(debug_bounds)
    if not os.path.exists(path):
        return False
    t = os.path.getmtime(path)
    return all(os.path.getmtime(d) <= t for d in _deps())


def build(force: bool = False, verbose: bool = False, extra_flags=(), debug_bounds=None) -> str:
    """Build libgato.so if any source is newer than it (and, when the
    checking build is requested, libgato_bounds.so); returns the path of the
    library the binding will load."""
    if debug_bounds is None:
        debug_bounds = debug_bounds_requested()
    _build_one(force, verbose, extra_flags, False)
    if debug_bounds:
        _build_one(force, verbose, extra_flags, True)
    return library_path(debug_bounds)


def _build_one(force, verbose, extra_flags, debug_bounds):
    lib_path = library_path(debug_bounds)
    if not force and up_to_date(debug_bounds):
        return lib_path
    nvcc = _nvcc()
    obj_dir = os.path.join(OUT_DIR, "obj_bounds" if debug_bounds else "obj")
    os.makedirs(obj_dir, exist_ok=True)

    def compile_one(src):
        obj = os.path.join(obj_dir, os.path.basename(src)[:-3] + ".o")
        cmd = compile_command(src, obj, debug_bounds, extra_flags)
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{res.stderr}")
        if verbose and res.stderr:
            print(res.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
        objs = list(ex.map(compile_one, _sources()))
    tmp = lib_path + f".tmp{os.getpid()}"
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc link failed:\n{res.stderr}")
    os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    print(build(force=True, verbose=True, extra_flags=("-Xptxas", "-v")))
