"""Build libaaren.so (the CUDA library behind include/aaren.h) in-tree,
and its checked twin libaaren_checked.so.

nvcc compiles csrc/aaren_api.cu for sm_103a only; the shared libraries land
next to this file so the Python binding finds them without installation.
The checked library is the same source compiled with -DAAREN_CHECKED: every
kernel bounds-checks the extents it computes and reports a violation as
AAREN_ERR_BOUNDS (a test build, used in place of a memory checker).
"""
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(HERE, "libaaren.so")
CHECKED_LIB = os.path.join(HERE, "libaaren_checked.so")
SOURCES = [os.path.join(CSRC, "aaren_api.cu")]
DEPENDS = SOURCES + [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cuh")] + [
    os.path.join(INCLUDE, "aaren.h")]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-shared",
         "-Xptxas", "-v", "--expt-relaxed-constexpr"]


def nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found; the CUDA toolkit is required to build libaaren")
    return cand


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(f) <= t for f in DEPENDS)


def _compile(lib: str, extra: list, verbose: bool) -> str:
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [nvcc(), *ARCH, *FLAGS, *extra, "-I", INCLUDE, "-o", tmp, *SOURCES]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        sys.stderr.write(res.stdout + res.stderr)
        raise RuntimeError(f"nvcc failed building {os.path.basename(lib)}")
    if verbose:
        sys.stderr.write(res.stderr)
    os.replace(tmp, lib)
    return lib


def build(force: bool = False, verbose: bool = False) -> str:
    """Build libaaren.so if it is missing or older than its sources."""
    if force or not up_to_date(LIB):
        _compile(LIB, [], verbose)
    return LIB


def build_checked(force: bool = False, verbose: bool = False) -> str:
    """Build libaaren_checked.so (-DAAREN_CHECKED) if it is missing or stale."""
    if force or not up_to_date(CHECKED_LIB):
        _compile(CHECKED_LIB, ["-DAAREN_CHECKED"], verbose)
    return CHECKED_LIB


if __name__ == "__main__":
    print(build(force=True, verbose="-v" in sys.argv))
    print(build_checked(force=True, verbose="-v" in sys.argv))
