"""Builds libgrpo.so in-tree with nvcc for sm_103a (GB300).

    python -m rl_fine_tuning_gb300.build [--force]

Two libraries from the same sources, all translation units compiled in
parallel, in rl_fine_tuning_gb300/_build/ (git-ignored):
  libgrpo.so          the library;
  libgrpo_checked.so  the same with device-side index checks
                      (GRPO_DEVICE_CHECKS; see grpo_device_checks in grpo.h).
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "libgrpo.so")
LIB_CHECKED = os.path.join(BUILD, "libgrpo_checked.so")
VARIANTS = {LIB: [], LIB_CHECKED: ["-DGRPO_DEVICE_CHECKS"]}
SOURCES = ["tc_kernels.cu", "small_kernels.cu", "grpo_abi.cu"]
HEADERS = ["ptx.cuh", "internal.h"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I" + INCLUDE, "-I" + CSRC]


def nvcc() -> str:
    p = shutil.which("nvcc")
    if p:
        return p
    cand = "/usr/local/cuda/bin/nvcc"
    if os.path.exists(cand):
        return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libgrpo")


def _stale(lib: str) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    deps = [os.path.join(CSRC, f) for f in SOURCES + HEADERS] + [os.path.join(INCLUDE, "grpo.h")]
    return any(os.path.getmtime(p) > t for p in deps)


def build(force: bool = False, verbose: bool = False) -> str:
    """Builds both libraries if needed; returns the path of libgrpo.so."""
    todo = [lib for lib in VARIANTS if force or _stale(lib)]
    if not todo:
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    exe = nvcc()

    def compile_one(job):
        lib, src = job
        tag = os.path.splitext(os.path.basename(lib))[0]
        obj = os.path.join(BUILD, f"{tag}_{src.replace('.cu', '.o')}")
        cmd = [exe, *ARCH, *FLAGS, *VARIANTS[lib], "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src} ({tag}):\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout, r.stderr, file=sys.stderr)
        return lib, obj

    jobs = [(lib, src) for lib in todo for src in SOURCES]
    with cf.ThreadPoolExecutor(max_workers=len(jobs)) as ex:
        done = list(ex.map(compile_one, jobs))
    for lib in todo:
        objs = [obj for l2, obj in done if l2 == lib]
        tmp = lib + f".tmp{os.getpid()}"
        r = subprocess.run([exe, *ARCH, "-shared", "-o", tmp, *objs], capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, lib)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
