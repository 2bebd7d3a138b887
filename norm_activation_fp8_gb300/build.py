"""Build ``libvg_fused.so`` in-tree with nvcc for sm_103a (no GPU needed).

Each ``.cu`` file compiles in its own nvcc process (in parallel), then one
link step makes the shared library with the CUDA runtime linked statically.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB_NAME = "libvg_fused.so"
LIB_PATH = os.path.join(BUILD, LIB_NAME)

SOURCES = ["vg_fused.cu", "norm_fp8.cu", "silu_fp8.cu", "mla_norm.cu", "qk_norm_rope.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
                     "-I", INCLUDE, "-I", CSRC]


def nvcc_path() -> str:
    for cand in (os.environ.get("NVCC"),
                 os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc"),
                 shutil.which("nvcc")):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: set CUDA_HOME or NVCC")


def _inputs():
    files = [os.path.join(CSRC, s) for s in SOURCES]
    files += [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    files += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE) if f.endswith(".h")]
    files.append(os.path.abspath(__file__))
    return files


def is_stale(lib_path: str = LIB_PATH) -> bool:
    if not os.path.exists(lib_path):
        return True
    built = os.path.getmtime(lib_path)
    return any(os.path.getmtime(f) > built for f in _inputs())


# A test-only copy of the library whose pipelined kernels give up their
# first wait (it also waits on a barrier nothing arrives on) after a short
# poll limit, so a GPU test can check the timeout report without a fault.
WAIT_TEST_LIB = os.path.join(BUILD, "libvg_fused_wait_timeout_test.so")
WAIT_TEST_FLAGS = ("-DVG_TEST_FORCE_WAIT_TIMEOUT", "-DVG_WAIT_LIMIT=4096u")


def build(force: bool = False, verbose: bool = False, extra_flags=(), out: str | None = None) -> str:
    """Compile and link the CUDA library (or, with ``out``, a copy built with
    ``extra_flags`` under that name); returns its path."""
    lib_path = out or LIB_PATH
    if not force and not is_stale(lib_path):
        return lib_path
    obj_dir = BUILD if out is None else os.path.join(BUILD, "obj_" + os.path.basename(out))
    os.makedirs(obj_dir, exist_ok=True)
    nvcc = nvcc_path()
    procs = []
    objs = []
    for src in SOURCES:
        obj = os.path.join(obj_dir, src.replace(".cu", ".o"))
        objs.append(obj)
        cmd = [nvcc, *NVCC_FLAGS, *extra_flags, "-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
    failed = []
    for src, p in procs:
        out, _ = p.communicate()
        if verbose or p.returncode:
            sys.stderr.write(out.decode(errors="replace"))
        if p.returncode:
            failed.append(src)
    if failed:
        raise RuntimeError(f"nvcc failed on {failed}")
    tmp = lib_path + f".tmp{os.getpid()}"
    subprocess.check_call([nvcc, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs])
    os.replace(tmp, lib_path)
    return lib_path


def build_wait_test(force: bool = False) -> str:
    return build(force, extra_flags=WAIT_TEST_FLAGS, out=WAIT_TEST_LIB)


# Test-only copies with device bounds checks: every store and bulk-copy
# source is checked against its tensor's extent; an access outside it is
# skipped and reported as VG_DEVICE_OUT_OF_BOUNDS.  The "shrunk" copy
# reports every tensor one row short, so that the checks must fire.
DEBUG_LIB = os.path.join(BUILD, "libvg_fused_debug_checks.so")
DEBUG_FLAGS = ("-DVG_DEBUG_CHECKS",)
DEBUG_SHRUNK_LIB = os.path.join(BUILD, "libvg_fused_debug_checks_shrunk.so")
DEBUG_SHRUNK_FLAGS = ("-DVG_DEBUG_CHECKS", "-DVG_DEBUG_SHRINK_EXTENT")


def build_debug(force: bool = False, shrunk: bool = False) -> str:
    if shrunk:
        return build(force, extra_flags=DEBUG_SHRUNK_FLAGS, out=DEBUG_SHRUNK_LIB)
    return build(force, extra_flags=DEBUG_FLAGS, out=DEBUG_LIB)


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
