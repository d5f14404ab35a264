"""Compile the CUDA library in-tree with nvcc for sm_103a (no torch headers).

Each translation unit under csrc/ is compiled on its own (in parallel) and the
objects are linked into libtopk_bf16.so.
"""
from __future__ import annotations

import glob
import os
import subprocess
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
HEADER = os.path.join(ROOT, "include", "topk_bf16.h")
LIB_PATH = os.path.join(PKG, "libtopk_bf16.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = [*ARCH, "-O3", "-lineinfo", "-std=c++20", "-Xcompiler", "-fPIC"]


def sources() -> list[str]:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _inputs() -> list[str]:
    return [*sources(), *glob.glob(os.path.join(CSRC, "*.cuh")), *glob.glob(os.path.join(CSRC, "*.h")),
            HEADER, __file__]


def _nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def up_to_date(out: str = LIB_PATH) -> bool:
    if not os.path.exists(out):
        return False
    t = os.path.getmtime(out)
    return all(os.path.getmtime(f) <= t for f in _inputs())


def _run(cmd: list[str]) -> str:
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc failed ({res.returncode}): {' '.join(cmd)}\n{res.stdout}\n{res.stderr}")
    return res.stderr


def build(force: bool = False, out: str = LIB_PATH, extra_flags=(), verbose: bool = False) -> str:
    """Build libtopk_bf16.so next to this file (or at `out`); returns its path.

    extra_flags go to every compile (e.g. ["-DTOPK_DEBUG"]); a build with extra
    flags is always redone.
    """
    if not force and not extra_flags and up_to_date(out):
        return out
    tag = f"{os.getpid()}"
    objdir = f"{out}.obj{tag}"
    os.makedirs(objdir, exist_ok=True)
    inc = ["-I", os.path.dirname(HEADER), "-I", CSRC]
    flags = [*NVCC_FLAGS, *extra_flags, *(["-Xptxas", "-v"] if verbose else [])]
    jobs = []
    for src in sources():
        obj = os.path.join(objdir, os.path.basename(src) + ".o")
        jobs.append((obj, [_nvcc(), *flags, *inc, "-c", "-o", obj, src]))
    try:
        with ThreadPoolExecutor(len(jobs)) as ex:
            logs = list(ex.map(lambda j: _run(j[1]), jobs))
        tmp = f"{out}.tmp{tag}"
        _run([_nvcc(), *ARCH, "-shared", "-o", tmp, *[j[0] for j in jobs]])
        os.replace(tmp, out)
    finally:
        for obj, _ in jobs:
            if os.path.exists(obj):
                os.remove(obj)
        if os.path.isdir(objdir):
            os.rmdir(objdir)
    if verbose:
        print("\n".join(logs))
    return out
