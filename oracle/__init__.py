"""CPU oracle for exact per-row BF16 top-k.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` use it; the product path never imports it.

The definition lives in ``topk_oracle.c`` (plain C, one qsort per row); this
module compiles it with gcc on first use and calls it through ctypes. It shares
no code with the CUDA library.

Pages followed (see the C file's header for the full statement):
  * vLLM "decode_topk_cute", module docstring, "What this module computes";
  * sglang PR #39305 "Exact bf16 consumer top-k adapted from DeepSelect",
    Modifications (order key, NaN never selected);
  * vLLM kimi_k3 "dsa/indexer", IndexerSelect (lowest-index ties; emit's
    block-table transform; the ordered output with per-row counts) and
    IndexerScore.rows_out (the per-8 maxima, "tops", the select is bounded by).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

TOKEN = 0
BLOCK8 = 1

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "topk_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libtopk_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False, src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile the oracle with gcc (-O2, pthreads) into a shared library."""
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    subprocess.run(["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-pthread", "-o", tmp, src],
                   check=True)
    os.replace(tmp, out)
    return out


def _bind(path: str):
    lib = ctypes.CDLL(path)
    f = lib.oracle_topk_bf16
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32,
                  ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32,
                  ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32,
                  ctypes.c_void_p, ctypes.c_int32]
    g = lib.oracle_topk_bf16_paged
    g.restype = ctypes.c_int
    g.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32,
                  ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32,
                  ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                  ctypes.c_void_p, ctypes.c_int32]
    o = lib.oracle_topk_bf16_ordered
    o.restype = ctypes.c_int
    o.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32,
                  ctypes.c_void_p, ctypes.c_int32,
                  ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                  ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32]
    wd = lib.oracle_topk_bf16_words
    wd.restype = ctypes.c_int
    wd.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32,
                   ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p]
    t = lib.oracle_tops
    t.restype = ctypes.c_int
    t.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32,
                  ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64]
    return lib


def load(path: str | None = None):
    """The oracle library (built on first use); ``path`` loads another build."""
    global _lib
    if path is not None:
        return _bind(path)
    with _lock:
        if _lib is None:
            _lib = _bind(build())
        return _lib


def topk(logits, valid_len, k: int, mode: int = TOKEN, block_table=None, page_size: int = 64,
         width: int | None = None, threads: int = 1, lib=None, block_rows: int | None = None,
         rows_per_request: int = 1) -> np.ndarray:
    """Exact top-k of every row; returns int32 [rows, k] (selected indices, then -1).

    logits: uint16/int16 array [rows, row_stride] of BF16 bits (a torch tensor
    of dtype bfloat16/int16 on the CPU is accepted too); valid_len: int [rows];
    block_table: None (identity) or int32 [ceil(rows / rows_per_request), pages];
    width: the row width (defaults to row_stride); block_rows: physical rows per
    page (default page_size); rows_per_request: rows sharing one table row.
    """
    logits = _as_u16(logits)
    if logits.ndim != 2:
        raise ValueError("logits must be 2-D [rows, row_stride]")
    rows, stride = logits.shape
    width = stride if width is None else int(width)
    valid = np.ascontiguousarray(np.asarray(valid_len, dtype=np.int32).reshape(-1))
    if valid.shape[0] != rows:
        raise ValueError("valid_len must have one entry per row")
    table_ptr, table_stride = None, 0
    if block_table is not None:
        table = np.ascontiguousarray(np.asarray(block_table, dtype=np.int32))
        if table.ndim != 2 or table.shape[0] < -(-rows // rows_per_request):
            raise ValueError("block_table needs ceil(rows / rows_per_request) rows of pages")
        table_ptr, table_stride = table.ctypes.data, table.shape[1]
    out = np.empty((rows, k), dtype=np.int32)
    lib = lib or load()
    rc = lib.oracle_topk_bf16_paged(logits.ctypes.data, stride, rows, width, valid.ctypes.data, k,
                                    mode, table_ptr, table_stride, page_size,
                                    page_size if block_rows is None else block_rows,
                                    rows_per_request, out.ctypes.data, threads)
    if rc != 0:
        raise RuntimeError("oracle_topk_bf16 failed (bad argument or out of memory)")
    return out


def _table(block_table, rows: int, rows_per_request: int):
    if block_table is None:
        return None, 0, None
    table = np.ascontiguousarray(np.asarray(block_table, dtype=np.int32))
    if table.ndim != 2 or table.shape[0] < -(-rows // rows_per_request):
        raise ValueError("block_table needs ceil(rows / rows_per_request) rows of pages")
    return table.ctypes.data, table.shape[1], table


def topk_ordered(logits, valid_len, k: int, block_table=None, page_size: int = 64,
                 width: int | None = None, threads: int = 1, lib=None,
                 block_rows: int | None = None, rows_per_request: int = 1):
    """Token mode, IndexerSelect's output: (out, valid, ids) with out and ids
    int32 [rows, k] (the selection in ascending index order, transformed / not,
    then -1) and valid int32 [rows] (the counts). Arguments as topk()."""
    logits = _as_u16(logits)
    if logits.ndim != 2:
        raise ValueError("logits must be 2-D [rows, row_stride]")
    rows, stride = logits.shape
    width = stride if width is None else int(width)
    valid_len = np.ascontiguousarray(np.asarray(valid_len, dtype=np.int32).reshape(-1))
    if valid_len.shape[0] != rows:
        raise ValueError("valid_len must have one entry per row")
    table_ptr, table_stride, _keep = _table(block_table, rows, rows_per_request)
    out = np.empty((rows, k), dtype=np.int32)
    ids = np.empty((rows, k), dtype=np.int32)
    counts = np.empty(rows, dtype=np.int32)
    lib = lib or load()
    rc = lib.oracle_topk_bf16_ordered(logits.ctypes.data, stride, rows, width, valid_len.ctypes.data, k,
                                      table_ptr, table_stride, page_size,
                                      page_size if block_rows is None else block_rows,
                                      rows_per_request, out.ctypes.data, counts.ctypes.data,
                                      ids.ctypes.data, threads)
    if rc != 0:
        raise RuntimeError("oracle_topk_bf16_ordered failed (bad argument or out of memory)")
    return out, counts, ids


def topk_words(logits, valid_len, n: int, width: int | None = None, lib=None):
    """Token mode, IndexerLocalTopk's output: (out, valid) with out int32
    [rows, n + n / 32] (B' words of the selection: keys above the n-th largest in
    index order, then the ties taken; then the plane of each index's bit 16) and
    valid int32 [rows]."""
    logits = _as_u16(logits)
    rows, stride = logits.shape
    width = stride if width is None else int(width)
    valid_len = np.ascontiguousarray(np.asarray(valid_len, dtype=np.int32).reshape(-1))
    out = np.empty((rows, n + n // 32), dtype=np.int32)
    counts = np.empty(rows, dtype=np.int32)
    lib = lib or load()
    if lib.oracle_topk_bf16_words(logits.ctypes.data, stride, rows, width, valid_len.ctypes.data, n,
                                  out.ctypes.data, counts.ctypes.data) != 0:
        raise RuntimeError("oracle_topk_bf16_words failed (bad argument or out of memory)")
    return out, counts


def tops(logits, valid_len, width: int | None = None, lib=None) -> np.ndarray:
    """The per-8 maxima the ordered select is bounded by: uint16 [rows,
    ceil(width / 8)], each aligned group's largest order key among its valid,
    non-NaN logits (0 for none)."""
    logits = _as_u16(logits)
    rows, stride = logits.shape
    width = stride if width is None else int(width)
    valid_len = np.ascontiguousarray(np.asarray(valid_len, dtype=np.int32).reshape(-1))
    groups = (width + 7) // 8
    out = np.empty((rows, groups), dtype=np.uint16)
    lib = lib or load()
    if lib.oracle_tops(logits.ctypes.data, stride, rows, width, valid_len.ctypes.data,
                       out.ctypes.data, groups) != 0:
        raise RuntimeError("oracle_tops failed (bad argument)")
    return out


def _as_u16(x) -> np.ndarray:
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().cpu().contiguous().view(torch.int16).numpy()
    except ImportError:  # pragma: no cover - torch is always present here
        pass
    x = np.asarray(x)
    if x.dtype == np.int16:
        x = x.view(np.uint16)
    if x.dtype != np.uint16:
        raise TypeError("logits must hold BF16 bits as uint16/int16")
    return np.ascontiguousarray(x)
