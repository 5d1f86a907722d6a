"""Build libppsched.so in-tree with nvcc for sm_103a (no cmake, no torch).

Each translation unit under csrc/ is compiled in parallel, then linked into
``pipeline_schedule_simulation_gb300/_build/libppsched.so`` with the CUDA
runtime linked statically, so the library loads on machines without a GPU
(calls then fail with PP_ERR_CUDA).
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(BUILD, "libppsched.so")
# The bounds-checked build (-DPPS_CHECKED: every table-driven address checked
# in the kernels, failures recorded for pp_sched_debug_checks), in a folder of
# its own so that both builds can coexist.
BUILD_CHECKED = os.path.join(PKG, "_build_checked")
LIB_CHECKED = os.path.join(BUILD_CHECKED, "libppsched_checked.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++20", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
         "-I", os.path.join(ROOT, "include")]


def _nvcc():
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libppsched")
    return cand


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _stale(out, deps):
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, extra=(), checked: bool = False) -> str:
    build_dir, lib_path = (BUILD_CHECKED, LIB_CHECKED) if checked else (BUILD, LIB)
    if checked:
        extra = ["-DPPS_CHECKED", *extra]
    os.makedirs(build_dir, exist_ok=True)
    nvcc = _nvcc()
    headers = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    headers.append(os.path.join(ROOT, "include", "ppsched.h"))
    jobs = []
    objs = []
    for src in sources():
        obj = os.path.join(build_dir, os.path.basename(src)[:-3] + ".o")
        objs.append(obj)
        if force or _stale(obj, [src, *headers]):
            jobs.append((src, obj))

    def compile_one(job):
        src, obj = job
        cmd = [nvcc, *ARCH, *FLAGS, *extra, "-c", src, "-o", obj + ".tmp"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        os.replace(obj + ".tmp", obj)
        return src, r.stdout + r.stderr

    if jobs:
        with cf.ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 4)) as ex:
            for src, log in ex.map(compile_one, jobs):
                if verbose and log.strip():
                    print(f"== {os.path.basename(src)}\n{log}", file=sys.stderr)
    if force or jobs or _stale(lib_path, objs):
        tmp = lib_path + f".tmp{os.getpid()}"
        cmd = [nvcc, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    v = "-v" in sys.argv
    extra = ["-Xptxas", "-v"] if "--ptxas" in sys.argv else []
    print(build(force="--force" in sys.argv or bool(extra), verbose=v or bool(extra), extra=extra,
                checked="--checked" in sys.argv))
