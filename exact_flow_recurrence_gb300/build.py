"""Build libefla_gb300.so in-tree from csrc/*.cu for sm_103a (nvcc, no cmake).

Each translation unit compiles in parallel; the objects are linked into one
shared library next to this file.  The same sources compiled with -DEFLA_DEBUG
(tile-level bounds checks on the tensor-core kernels' global writes) give
libefla_gb300_debug.so beside it, built in the same pass.  ``python -m exact_flow_recurrence_gb300.build``
builds it; ``--force`` rebuilds; ``--ptxas`` prints ptxas resource usage.
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
OBJ = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libefla_gb300.so")
DEBUG_OBJ = os.path.join(HERE, "_build_debug")
DEBUG_LIB = os.path.join(HERE, "libefla_gb300_debug.so")
# (object folder, library, extra nvcc flags) per variant
VARIANTS = ((OBJ, LIB, []), (DEBUG_OBJ, DEBUG_LIB, ["-DEFLA_DEBUG"]))
INCLUDE = os.path.join(os.path.dirname(HERE), "include")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE]


def nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found; the CUDA 13 toolkit is required to build the library")
    return cand


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) \
        + glob.glob(os.path.join(INCLUDE, "*.h"))


def up_to_date() -> bool:
    for _, lib, _ in VARIANTS:
        if not os.path.exists(lib):
            return False
        t = os.path.getmtime(lib)
        if any(os.path.getmtime(p) > t for p in _deps()):
            return False
    return True


def build(force: bool = False, ptxas_verbose: bool = False, jobs: int = 0) -> str:
    if not force and not ptxas_verbose and up_to_date():
        return LIB
    cc = nvcc()
    srcs = _sources()
    extra = ["-Xptxas", "-v"] if ptxas_verbose else []
    for obj_dir, _, _ in VARIANTS:
        os.makedirs(obj_dir, exist_ok=True)

    def compile_one(task):
        src, (obj_dir, _, flags) = task
        obj = os.path.join(obj_dir, os.path.basename(src) + ".o")
        cmd = [cc, *ARCH, *FLAGS, *flags, *extra, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {os.path.basename(src)} {' '.join(flags)}:\n{r.stderr}")
        return obj, r.stderr

    # the largest sources first, so that the longest compilations overlap the rest
    tasks = sorted(((src, v) for v in VARIANTS for src in srcs), key=lambda t: -os.path.getsize(t[0]))
    jobs = jobs or min(len(tasks), os.cpu_count() or 4)
    with cf.ThreadPoolExecutor(max_workers=jobs) as ex:
        results = list(ex.map(compile_one, tasks))
    if ptxas_verbose:
        for (_, (_, _, flags)), (_, err) in zip(tasks, results):
            if not flags:
                sys.stderr.write(err)
    for obj_dir, lib, _ in VARIANTS:
        objs = [o for (_, (d, _, _)), (o, _) in zip(tasks, results) if d == obj_dir]
        tmp = lib + ".tmp"
        r = subprocess.run([cc, *ARCH, "-shared", "-o", tmp, *sorted(objs)], capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link of {os.path.basename(lib)} failed:\n{r.stderr}")
        os.replace(tmp, lib)
    return LIB


if __name__ == "__main__":  # pragma: no cover
    print(build(force="--force" in sys.argv, ptxas_verbose="--ptxas" in sys.argv))
