"""Build ``libgbrouter.so`` in-tree with nvcc for sm_103a.

Each ``csrc/*.cu`` compiles to an object in parallel, then nvcc links the
shared library next to this file. Rebuilds only when a source or header is
newer than the library.

``build(variant="stamps")`` builds the measurement variant
``libgbrouter_stamps.so`` from the same sources with ``-DGBR_PHASE_STAMPS``
(per-phase timestamps in the single-cluster kernel); nothing loads it
unless asked to.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
LIB = os.path.join(HERE, "libgbrouter.so")
OBJ_DIR = os.path.join(HERE, "_build")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xptxas", "-v",
              f"-I{INCLUDE}"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the router library needs the CUDA toolkit to build")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + \
        glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(INCLUDE, "*.h"))


VARIANTS = {None: ("libgbrouter.so", "_build", []),
            "stamps": ("libgbrouter_stamps.so", "_build_stamps", ["-DGBR_PHASE_STAMPS"])}


def lib_path(variant=None) -> str:
    return os.path.join(HERE, VARIANTS[variant][0])


def is_stale(variant=None) -> bool:
    lib = lib_path(variant)
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(p) > t for p in _deps())


def build(force: bool = False, verbose: bool = False, variant=None) -> str:
    LIB = lib_path(variant)
    if not force and not is_stale(variant):
        return LIB
    nvcc = _nvcc()
    obj_dir = os.path.join(HERE, VARIANTS[variant][1])
    defines = VARIANTS[variant][2]
    os.makedirs(obj_dir, exist_ok=True)
    srcs = _sources()

    def compile_one(src):
        obj = os.path.join(obj_dir, os.path.basename(src)[:-3] + ".o")
        cmd = [nvcc, *ARCH, *NVCC_FLAGS, *defines, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stderr}")
        return obj, r.stderr

    with cf.ThreadPoolExecutor(max_workers=len(srcs)) as ex:
        results = list(ex.map(compile_one, srcs))
    if verbose:
        for obj, log in results:
            sys.stderr.write(f"== {os.path.basename(obj)}\n{log}")
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *[o for o, _ in results]]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc link failed:\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv,
                variant="stamps" if "--stamps" in sys.argv else None))
