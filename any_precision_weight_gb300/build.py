"""Builds libpw.so in-tree with nvcc for sm_103a (no cmake, no torch extension
machinery): every translation unit is compiled in parallel, then linked into
one shared library next to this file; libpw_check.so is the same library with
PW_CHECK defined (device-side bounds checks).

    python -m any_precision_weight_gb300.build [-v]
"""
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libpw.so")
CHECK_LIB = os.path.join(HERE, "libpw_check.so")

SOURCES = ["pw_runtime.cpp", "pw_planner.cpp", "pw_kernels.cu", "pw_decode.cu", "pw_prefill.cu", "pw_static.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for c in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found")


def _flags(src: str, check: bool):
    f = ["-O3", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
         "-I", os.path.join(HERE, "..", "include")]
    if src.endswith(".cu"):
        f += ARCH + ["-lineinfo", "--expt-relaxed-constexpr", "-Xptxas", "-v"]
    if check:
        f += ["-DPW_CHECK=1"]
    return f


def _compile(job):
    src, check = job
    stem = os.path.splitext(src)[0] + ("_check" if check else "")
    obj = os.path.join(BUILD, stem + ".o")
    cmd = [nvcc()] + _flags(src, check) + ["-c", os.path.join(CSRC, src), "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
    with open(os.path.join(BUILD, stem + ".ptxas.txt"), "w") as fh:
        fh.write(r.stderr)
    return obj


def _link(objs, out):
    tmp = out + ".tmp"
    cmd = [nvcc(), "-shared"] + ARCH + ["-o", tmp] + objs
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, out)


def build(verbose: bool = False) -> str:
    """libpw.so, and libpw_check.so: the same sources with PW_CHECK defined
    (device-side bounds checks that report PW_STATUS_BOUNDS)."""
    os.makedirs(BUILD, exist_ok=True)
    jobs = [(s, c) for c in (False, True) for s in SOURCES]
    with ThreadPoolExecutor(max_workers=len(jobs)) as ex:
        objs = list(ex.map(_compile, jobs))
    n = len(SOURCES)
    _link(objs[:n], LIB)
    _link(objs[n:], CHECK_LIB)
    if verbose:
        for s in SOURCES:
            p = os.path.join(BUILD, os.path.splitext(s)[0] + ".ptxas.txt")
            if os.path.exists(p):
                sys.stdout.write(open(p).read())
    return LIB


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv))
