"""Build the sm_103a shared library in-tree (``_build/librmsnorm_gb300.so``).

Each kernel translation unit is compiled by its own nvcc process in parallel,
then linked with the C-ABI unit into one shared library that exports only
the ``rmsnorm_*`` symbols of ``include/rmsnorm.h``.  The CUDA runtime is
linked statically, so the library needs nothing but the driver at run time.

``build(checked=True)`` makes the bounds-checked debug library
(``_build/librmsnorm_gb300_checked.so``, compiled with -DRMSNORM_BOUNDS_CHECK):
every global access and ring copy of its kernels is checked against its
tensor's extent, and one out of range is skipped and reported in bit 1 of the
status word.  Point the binding at it with the environment variable
RMSNORM_GB300_LIB.
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG, "_build")
LIB_NAME = "librmsnorm_gb300.so"
LIB_PATH = os.path.join(BUILD_DIR, LIB_NAME)
CHECKED_PATH = os.path.join(BUILD_DIR, "librmsnorm_gb300_checked.so")
# the bench's C timing harness (not part of the library)
HOSTCOST_SRC = os.path.join(PKG, "bench_src", "host_cost.cu")
HOSTCOST_PATH = os.path.join(BUILD_DIR, "librmsn_hostcost.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler",
              "-fvisibility=hidden", "-I", INCLUDE]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build the library")


def sources() -> list[str]:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _inputs() -> list[str]:
    return (sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h"))
            + glob.glob(os.path.join(CSRC, "*.inc")) + glob.glob(os.path.join(INCLUDE, "*.h"))
            + [os.path.abspath(__file__)])


def up_to_date(checked: bool = False) -> bool:
    outs = [CHECKED_PATH] if checked else [LIB_PATH, HOSTCOST_PATH]
    if not all(os.path.exists(o) for o in outs):
        return False
    t = min(os.path.getmtime(o) for o in outs)
    return all(os.path.getmtime(f) <= t for f in _inputs() + [HOSTCOST_SRC])


def build(force: bool = False, verbose: bool = False, jobs: int | None = None,
          checked: bool = False) -> str:
    """Compile and link the library (the bounds-checked one with ``checked``)
    if a source is newer than it; return its path."""
    out = CHECKED_PATH if checked else LIB_PATH
    if not force and up_to_date(checked):
        return out
    obj_dir = os.path.join(BUILD_DIR, "checked") if checked else BUILD_DIR
    os.makedirs(obj_dir, exist_ok=True)
    cc = nvcc()
    srcs = sources()
    objs = [os.path.join(obj_dir, os.path.basename(s)[:-3] + ".o") for s in srcs]
    extra = ["-DRMSNORM_BOUNDS_CHECK"] if checked else []

    def compile_one(pair):
        src, obj = pair
        cmd = [cc, *ARCH, *NVCC_FLAGS, *extra, "-c", src, "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stdout}\n{r.stderr}")
        return r.stderr

    n = jobs or min(len(srcs), os.cpu_count() or 1)
    with ThreadPoolExecutor(max(1, n)) as ex:
        logs = list(ex.map(compile_one, zip(srcs, objs)))
    if verbose:
        for src, log in zip(srcs, logs):
            sys.stderr.write(f"== {os.path.basename(src)}\n{log}")
    tmp = out + f".tmp{os.getpid()}"
    link = [cc, *ARCH, "-shared", "-cudart", "static", *objs, "-o", tmp]
    r = subprocess.run(link, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, out)
    if checked:
        return out
    # the C timing harness, linked against the library it times
    tmp = HOSTCOST_PATH + f".tmp{os.getpid()}"
    cmd = [cc, *ARCH, *NVCC_FLAGS, "-shared", "-cudart", "static", HOSTCOST_SRC, "-o", tmp,
           "-L", BUILD_DIR, "-lrmsnorm_gb300", "-Xlinker", "-rpath,$ORIGIN"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"host-cost harness failed to build:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, HOSTCOST_PATH)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv,
                checked="--checked" in sys.argv))
