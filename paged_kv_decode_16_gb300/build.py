"""Build the CUDA library (libpagedkv.so) in-tree with nvcc for sm_103a.

Each translation unit is compiled in parallel with
``-gencode arch=compute_103a,code=sm_103a -O3 -lineinfo`` and the objects are
linked into ``paged_kv_decode_16_gb300/_build/libpagedkv.so`` (static CUDA
runtime, so loading it needs no GPU).  Rebuilds only when a source or header
is newer than the library.  Concurrent builds (two test processes, a test and
the benchmark) take an exclusive file lock on ``_build/.lock`` and compile
into an object directory of their own, so they never share a half-written
object; the second one to get the lock finds the library up to date.
"""
from __future__ import annotations

import concurrent.futures as cf
import contextlib
import fcntl
import glob
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "libpagedkv.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    for cand in (os.environ.get("CUDA_HOME", ""), "/usr/local/cuda"):
        p = os.path.join(cand, "bin", "nvcc") if cand else ""
        if p and os.path.exists(p):
            return p
    p = shutil.which("nvcc")
    if not p:
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libpagedkv.so")
    return p


def sources() -> list[str]:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cpp")))


def _inputs() -> list[str]:
    return sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(
        os.path.join(CSRC, "*.hpp")) + glob.glob(os.path.join(INCLUDE, "*.h")) + [__file__]


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(f) <= t for f in _inputs())


@contextlib.contextmanager
def _build_lock():
    os.makedirs(OUT_DIR, exist_ok=True)
    with open(os.path.join(OUT_DIR, ".lock"), "w") as f:
        fcntl.flock(f, fcntl.LOCK_EX)
        try:
            yield
        finally:
            fcntl.flock(f, fcntl.LOCK_UN)


def build(force: bool = False, verbose: bool = False, ptxas_verbose: bool = False) -> str:
    """Compile every source for sm_103a and link libpagedkv.so; return its path."""
    if not force and up_to_date():
        return LIB
    with _build_lock():
        if not force and up_to_date():  # built by another process meanwhile
            return LIB
        return _build_locked(verbose, ptxas_verbose)


def _build_locked(verbose: bool, ptxas_verbose: bool) -> str:
    nvcc = _nvcc()
    obj_dir = os.path.join(OUT_DIR, f"obj{os.getpid()}")
    os.makedirs(obj_dir, exist_ok=True)
    common = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC,
              *ARCH]
    if ptxas_verbose:
        common += ["-Xptxas", "-v"]

    def compile_one(src: str):
        obj = os.path.join(obj_dir, os.path.basename(src) + ".o")
        cmd = [nvcc, "-c", src, "-o", obj, *common]
        if src.endswith(".cpp"):
            cmd = [nvcc, "-x", "cu", "-c", src, "-o", obj, *common]
        r = subprocess.run(cmd, capture_output=True, text=True)
        return src, obj, r

    objs = []
    errors = []
    with cf.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 4)) as ex:
        for src, obj, r in ex.map(compile_one, sources()):
            if verbose or ptxas_verbose:
                sys.stderr.write(r.stdout + r.stderr)
            if r.returncode != 0:
                errors.append(f"{os.path.basename(src)}:\n{r.stderr}")
            objs.append(obj)
    if errors:
        raise RuntimeError("nvcc failed:\n" + "\n".join(errors))
    # the temporary name keeps the .so suffix: nvcc picks the link step from it
    tmp = os.path.join(OUT_DIR, f"libpagedkv.tmp{os.getpid()}.so")
    cmd = [nvcc, "-shared", *ARCH, "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n" + r.stderr)
    os.replace(tmp, LIB)
    shutil.rmtree(obj_dir, ignore_errors=True)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, ptxas_verbose="-v" in sys.argv))
