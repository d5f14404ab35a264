"""Compile the CUDA library in-tree with nvcc for sm_103a (no torch headers)."""
from __future__ import annotations

import os
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
SRC = os.path.join(PKG, "csrc", "topk_bf16.cu")
HEADER = os.path.join(ROOT, "include", "topk_bf16.h")
LIB_PATH = os.path.join(PKG, "libtopk_bf16.so")

NVCC_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-lineinfo", "-std=c++20",
              "-shared", "-Xcompiler", "-fPIC", "-Xptxas", "-v"]


def _nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def up_to_date(out: str = LIB_PATH) -> bool:
    if not os.path.exists(out):
        return False
    t = os.path.getmtime(out)
    return all(os.path.getmtime(f) <= t for f in (SRC, HEADER, __file__))


def build(force: bool = False, out: str = LIB_PATH, extra_flags=(), verbose: bool = False) -> str:
    """Build libtopk_bf16.so next to this file; returns its path."""
    if not force and not extra_flags and up_to_date(out):
        return out
    tmp = f"{out}.tmp{os.getpid()}"
    cmd = [_nvcc(), *NVCC_FLAGS, *extra_flags, "-I", os.path.dirname(HEADER), "-o", tmp, SRC]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc failed ({res.returncode}):\n{res.stdout}\n{res.stderr}")
    if verbose:
        print(res.stderr)
    os.replace(tmp, out)
    return out
