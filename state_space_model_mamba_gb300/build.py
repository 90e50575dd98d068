"""Build ``libssd.so`` (the CUDA library behind include/ssd.h) in-tree.

Compiles every ``csrc/*.cu`` for sm_103a only, in parallel, and links them
into ``state_space_model_mamba_gb300/lib/libssd.so`` against the shared CUDA
runtime (so the process shares one runtime with PyTorch).  Run as
``python -m state_space_model_mamba_gb300.build``.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OBJ_DIR = os.path.join(PKG, "_build")
LIB_DIR = os.path.join(PKG, "lib")
LIB_PATH = os.path.join(LIB_DIR, "libssd.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _cuda_lib_dir(nvcc: str) -> str:
    root = os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))
    for sub in ("lib64", "lib", os.path.join("targets", "sbsa-linux", "lib"),
                os.path.join("targets", "x86_64-linux", "lib")):
        d = os.path.join(root, sub)
        if os.path.exists(os.path.join(d, "libcudart.so")):
            return d
    return os.path.join(root, "lib64")


def _flags(verbose_ptxas: bool) -> list:
    f = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC,
                "--expt-relaxed-constexpr", "-Xcompiler", "-Wall"]
    if verbose_ptxas:
        f += ["-Xptxas", "-v"]
    return f


def _stale(target: str, deps: list) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose_ptxas: bool = False, jobs: int | None = None) -> str:
    nvcc = _nvcc()
    os.makedirs(OBJ_DIR, exist_ok=True)
    os.makedirs(LIB_DIR, exist_ok=True)
    sources = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    headers = (sorted(glob.glob(os.path.join(CSRC, "*.cuh")))
               + sorted(glob.glob(os.path.join(INCLUDE, "*.h"))))
    objs = []
    todo = []
    for src in sources:
        obj = os.path.join(OBJ_DIR, os.path.basename(src)[:-3] + ".o")
        objs.append(obj)
        if force or _stale(obj, [src] + headers + [__file__]):
            todo.append((src, obj))

    def compile_one(item):
        src, obj = item
        cmd = [nvcc] + _flags(verbose_ptxas) + ["-c", src, "-o", obj + ".tmp"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stdout}\n{r.stderr}")
        os.replace(obj + ".tmp", obj)
        return src, r.stderr

    logs = []
    if todo:
        with cf.ThreadPoolExecutor(max_workers=jobs or min(len(todo), os.cpu_count() or 4)) as ex:
            for src, err in ex.map(compile_one, todo):
                if err.strip():
                    logs.append(f"== {os.path.basename(src)}\n{err}")
    if force or todo or _stale(LIB_PATH, objs):
        libdir = _cuda_lib_dir(nvcc)
        tmp = LIB_PATH + f".tmp{os.getpid()}"
        cmd = ([nvcc] + ARCH + ["-shared", "-cudart", "shared", "-o", tmp] + objs
               + ["-L", libdir, "-Xlinker", "-rpath", "-Xlinker", libdir])
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, LIB_PATH)
    if verbose_ptxas and logs:
        sys.stderr.write("\n".join(logs))
    return LIB_PATH


if __name__ == "__main__":
    force = "--force" in sys.argv
    build(force=force, verbose_ptxas="-v" in sys.argv)
    print(LIB_PATH)
