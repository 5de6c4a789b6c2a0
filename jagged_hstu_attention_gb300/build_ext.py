"""Builds the CUDA libraries in-tree for sm_103a.

``libhstu_attn.so`` is the release build. ``libhstu_attn_checked.so`` is the
same sources compiled with ``HSTU_CHECKED``: its kernels validate every
work-list entry before using it (a debugging aid, results bit-identical).
Every translation unit of both is compiled by nvcc in one parallel pool, then
each set is linked into one shared library next to this file (the CUDA
runtime is linked statically). A library newer than every source is not
rebuilt.
"""
from __future__ import annotations

import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(ROOT, "_build")
LIB_NAME = "libhstu_attn.so"
LIB_PATH = os.path.join(PKG, LIB_NAME)
CHECKED_LIB_PATH = os.path.join(PKG, "libhstu_attn_checked.so")
# variant -> (library, object directory, extra nvcc flags)
VARIANTS = {
    "release": (LIB_PATH, BUILD_DIR, []),
    "checked": (CHECKED_LIB_PATH, os.path.join(BUILD_DIR, "checked"), ["-DHSTU_CHECKED"]),
}
SOURCES = ["plan.cu", "attn_fwd_bf16.cu", "attn_fwd_f16.cu", "attn_bwd_bf16.cu", "attn_bwd_f16.cu", "targets_only.cu", "api.cu", "noalloc.cu", "selftest.cu", "func_build.cu", "project.cu",
           "shard.cpp"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
         "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC]


def _nvcc() -> str:
    cuda_home = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    cand = os.path.join(cuda_home, "bin", "nvcc")
    if os.path.exists(cand):
        return cand
    found = shutil.which("nvcc")
    if not found:
        raise RuntimeError("nvcc not found (set CUDA_HOME)")
    return found


def _deps():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(INCLUDE, "hstu_attn.h"))
    return files


def up_to_date(lib: str = LIB_PATH) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(f) <= t for f in _deps())


def build(force: bool = False, verbose: bool = False, variants=("release", "checked")) -> str:
    """Builds the requested variants; returns the release library's path."""
    todo = [v for v in variants if force or not up_to_date(VARIANTS[v][0])]
    if not todo:
        return LIB_PATH
    nvcc = _nvcc()

    def compile_one(job):
        variant, src = job
        _, obj_dir, extra = VARIANTS[variant]
        obj = os.path.join(obj_dir, os.path.splitext(src)[0] + ".o")
        cmd = [nvcc, *ARCH, *FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            print(" ".join(cmd), flush=True)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src} ({variant}):\n{r.stdout}\n{r.stderr}")
        return obj

    for v in todo:
        os.makedirs(VARIANTS[v][1], exist_ok=True)
    jobs = [(v, src) for v in todo for src in SOURCES]
    with ThreadPoolExecutor(max_workers=min(len(jobs), max(os.cpu_count() or 1, len(SOURCES)))) as ex:
        objs = list(ex.map(compile_one, jobs))
    for v in todo:
        lib = VARIANTS[v][0]
        tmp = lib + ".tmp"
        cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *[o for (vv, _), o in zip(jobs, objs) if vv == v]]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed ({v}):\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, lib)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force=True, verbose=True))
