"""Exact per-row top-k of BF16 logits on GB300: Python binding of libtopk_bf16.

Argument marshalling only: every step of the selection runs in the CUDA kernels
of the kernels under ``csrc/`` behind the C ABI declared in ``include/topk_bf16.h``.
Torch supplies device memory and the current stream. There is no CPU fallback:
if the library is missing or the tensors are not on a CUDA device, the call
raises.

The operation (vLLM "decode_topk_cute", module docstring): for every row, the
indices of its k largest elements (token mode: one BF16 logit; block mode: the
NaN-propagating maximum of each aligned group of 8 logits, the newest block
pinned at +inf, -inf blocks written as -1), ties at the k-th largest broken by
the lowest index, NaN never selected, a row of at most k elements returning
0..n-1 then -1, and an optional per-row block table applied to the indices.
"""
from __future__ import annotations

import ctypes
import os
import threading

from ._build import LIB_PATH, build

TOKEN = 0
BLOCK8 = 1
MAX_K = 2048
MAX_WIDTH = 1 << 20
NUM_COUNTERS = 40
COUNTER_NAMES = ("bypass_rows", "tile_sampled", "tile_exact", "tile_unbounded", "tile_overflow",
                 "tile_take_all", "compactions", "refills", "cluster_merges", "rounds",
                 "cyc_wait", "cyc_select", "cyc_filter", "cyc_finish", "cyc_compact",
                 "cyc_reps", "cyc_cut", "cyc_survivors", "cyc_exact", "guess_hit", "guess_miss",
                 "cyc_f_prep", "cyc_f_queue", "cyc_f_append", "cyc_f_sync", "cyc_f_find", "cyc_f_loop",
                 "tie_fills", "direct_rows", "cyc_kernel", "cyc_align", "ordered_tops",
                 "ordered_exact")

_STATUS = {0: "ok", 1: "invalid argument", 2: "misaligned", 3: "bad k", 4: "bad width",
           5: "CUDA error", 6: "more rows or wider rows than select_static takes"}


class TopkError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        super().__init__(f"topk_bf16: {_STATUS.get(status, status)}{(': ' + what) if what else ''}")
        self.status = status


class _Options(ctypes.Structure):
    _fields_ = [("force_direct", ctypes.c_int32), ("cluster", ctypes.c_int32),
                ("counters", ctypes.c_void_p), ("path", ctypes.c_int32), ("hold", ctypes.c_int32)]


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return LIB_PATH


def load(path: str | None = None):
    """Load libtopk_bf16.so (it must have been built: see ``_build.build``)."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise ImportError(f"libtopk_bf16.so not built at {p}; run __graft_entry__.build()")
        lib = ctypes.CDLL(p)
        sel_args = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32,
                    ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p,
                    ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p]
        lib.topk_bf16_select.argtypes = sel_args
        lib.topk_bf16_select.restype = ctypes.c_int
        lib.topk_bf16_select_ex.argtypes = sel_args + [ctypes.POINTER(_Options)]
        lib.topk_bf16_select_paged.restype = ctypes.c_int
        lib.topk_bf16_select_paged.argtypes = (sel_args[:10] + [ctypes.c_int32, ctypes.c_int32]
                                               + sel_args[10:])
        lib.topk_bf16_select_ex.restype = ctypes.c_int
        lib.topk_bf16_select_static.argtypes = sel_args
        lib.topk_bf16_select_static.restype = ctypes.c_int
        lib.topk_bf16_tops.restype = ctypes.c_int
        lib.topk_bf16_tops.argtypes = sel_args[:5] + [ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p]
        lib.topk_bf16_select_words.restype = ctypes.c_int
        lib.topk_bf16_select_words.argtypes = (sel_args[:6] + [ctypes.c_void_p, ctypes.c_int64]
                                               + [ctypes.c_void_p] * 3 + [ctypes.POINTER(_Options)])
        lib.topk_bf16_select_ordered.restype = ctypes.c_int
        lib.topk_bf16_select_ordered.argtypes = (sel_args[:6] + [ctypes.c_void_p, ctypes.c_int64]
                                                 + [ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32,
                                                    ctypes.c_int32, ctypes.c_int32]
                                                 + [ctypes.c_void_p] * 4 + [ctypes.POINTER(_Options)])
        lib.topk_bf16_status_string.argtypes = [ctypes.c_int]
        lib.topk_bf16_status_string.restype = ctypes.c_char_p
        i32p = ctypes.POINTER(ctypes.c_int32)
        lib.topk_bf16_plan.argtypes = [ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                       ctypes.c_int32, i32p, i32p, i32p, i32p, i32p]
        lib.topk_bf16_plan.restype = ctypes.c_int
        lib.topk_bf16_device_status.argtypes = [ctypes.POINTER(ctypes.c_uint32), ctypes.c_int32]
        lib.topk_bf16_device_status.restype = ctypes.c_int
        if path is None:
            _lib = lib
        return lib


def _check(status: int, what: str = ""):
    if status != 0:
        raise TopkError(status, what)


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def select(logits, valid_len, k: int, mode: int = TOKEN, block_table=None, page_size: int = 64,
           out=None, width: int | None = None, stream=None, *, force_direct: bool = False,
           cluster: int = 0, counters=None, path: int = 0, block_rows: int | None = None,
           rows_per_request: int = 1, hold: bool = False):
    """Exact top-k of every row of ``logits`` -> int32 [rows, k] on the same device.

    logits: CUDA bfloat16 (or int16/uint16 holding BF16 bits) [rows, row_stride]
    with unit inner stride, 16-byte aligned rows; valid_len: CUDA int32 [rows];
    block_table: None or CUDA int32 [rows, pages] (unit inner stride);
    width: logits per row that may be valid (default: logits.shape[1]);
    stream: a torch.cuda.Stream (default: the current stream);
    block_rows / rows_per_request: the full transform (see topk_bf16_select_paged):
    physical rows per page (default page_size) and rows sharing one table row;
    force_direct / cluster / counters / path: test hooks (see topk_bf16_select_ex);
    hold: do not let the next kernel on the stream start before this one completes
    (topk_bf16_options_t.hold).
    """
    import torch
    rows, width, row_stride, table_stride = _inputs(logits, valid_len, block_table, width,
                                                    rows_per_request)
    if out is None:
        out = torch.empty((rows, k), dtype=torch.int32, device=logits.device)
    elif not (out.is_cuda and out.dtype == torch.int32 and out.shape == (rows, k) and out.is_contiguous()):
        raise ValueError("out must be a contiguous CUDA int32 tensor [rows, k]")
    if stream is None:
        stream = torch.cuda.current_stream(logits.device)
    lib = load()
    with torch.cuda.device(logits.device):
        args = (_ptr(logits), row_stride, rows, width, _ptr(valid_len), int(k), int(mode),
                _ptr(block_table), table_stride, int(page_size), _ptr(out),
                ctypes.c_void_p(stream.cuda_stream))
        paged = (block_rows is not None and int(block_rows) != int(page_size)) or int(rows_per_request) != 1
        if paged:
            if force_direct or cluster or counters is not None or path or hold:
                raise ValueError("the options do not combine with block_rows / rows_per_request")
            st = lib.topk_bf16_select_paged(*args[:10], int(page_size if block_rows is None else block_rows),
                                            int(rows_per_request), *args[10:])
        elif force_direct or cluster or counters is not None or path or hold:
            opt = _Options(1 if force_direct else 0, int(cluster),
                           None if counters is None else counters.data_ptr(), int(path), 1 if hold else 0)
            st = lib.topk_bf16_select_ex(*args, ctypes.byref(opt))
        else:
            st = lib.topk_bf16_select(*args)
    _check(st)
    return out


def select_static(logits, valid_len, k: int, out, mode: int = TOKEN, block_table=None,
                  page_size: int = 64, width: int | None = None, stream=None):
    """select() through topk_bf16_select_static: no allocation on the call.

    For callers that cannot allocate device memory, so ``out`` (a contiguous CUDA
    int32 [rows, k]) is required. Rows of at most 16384 logits, at most 65536
    rows; each row starts from the cut that held for the same row index in the
    library's previous call of this entry point on the device (a static table
    of the library; results are exact whatever it holds). Other arguments as
    select().
    """
    import torch
    rows, width, row_stride, table_stride = _inputs(logits, valid_len, block_table, width, 1)
    if not (out.is_cuda and out.dtype == torch.int32 and out.shape == (rows, k) and out.is_contiguous()):
        raise ValueError("out must be a contiguous CUDA int32 tensor [rows, k]")
    if stream is None:
        stream = torch.cuda.current_stream(logits.device)
    lib = load()
    with torch.cuda.device(logits.device):
        st = lib.topk_bf16_select_static(_ptr(logits), row_stride, rows, width, _ptr(valid_len), int(k),
                                         int(mode), _ptr(block_table), table_stride, int(page_size),
                                         _ptr(out), ctypes.c_void_p(stream.cuda_stream))
    _check(st)
    return out


def select_ordered(logits, valid_len, k: int, tops=None, block_table=None, page_size: int = 64,
                   width: int | None = None, stream=None, *, block_rows: int | None = None,
                   rows_per_request: int = 1, ids: bool = False, out=None, valid=None,
                   counters=None, force_exact: bool = False, hold: bool = False):
    """The ordered select of the indexer page (token mode): (out, valid, ids) with
    out int32 [rows, k] the selection in ascending index order (transformed),
    then -1; valid int32 [rows] the counts; ids int32 [rows, k] the untransformed
    indices (None unless ``ids``). tops: None, or CUDA uint16/int16 [rows,
    tops_stride] (unit inner stride, 16-byte aligned rows): each aligned group of
    8 logits' largest order key among its valid non-NaN logits, 0 for none (see
    topk_bf16_select_ordered). Other arguments as select(); counters /
    force_exact: test hooks; hold as for select().
    """
    import torch
    rows, width, row_stride, table_stride = _inputs(logits, valid_len, block_table, width,
                                                    rows_per_request)
    tops_stride = _tops_stride(tops, rows, width)
    dev = logits.device
    if out is None:
        out = torch.empty((rows, k), dtype=torch.int32, device=dev)
    if valid is None:
        valid = torch.empty(rows, dtype=torch.int32, device=dev)
    ids_t = torch.empty((rows, k), dtype=torch.int32, device=dev) if ids else None
    _outputs(out, valid, rows, k)
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    opt = None
    if counters is not None or force_exact or hold:
        opt = ctypes.byref(_Options(1 if force_exact else 0, 0,
                                    None if counters is None else counters.data_ptr(), 0, 1 if hold else 0))
    lib = load()
    with torch.cuda.device(dev):
        st = lib.topk_bf16_select_ordered(
            _ptr(logits), row_stride, rows, width, _ptr(valid_len), int(k), _ptr(tops), tops_stride,
            _ptr(block_table), table_stride, int(page_size),
            int(page_size if block_rows is None else block_rows), int(rows_per_request),
            _ptr(out), _ptr(valid), _ptr(ids_t), ctypes.c_void_p(stream.cuda_stream), opt)
    _check(st)
    return out, valid, ids_t


def select_words(logits, valid_len, n: int, tops=None, width: int | None = None, stream=None, *,
                 out=None, valid=None, counters=None, force_exact: bool = False, hold: bool = False):
    """The local top-n as B' words (topk_bf16_select_words): (out, valid) with out
    int32 [rows, n + n / 32] and valid int32 [rows]. tops: None or the per-8
    maxima (as for select_ordered); other arguments as select_ordered."""
    import torch
    rows, width, row_stride, _ = _inputs(logits, valid_len, None, width, 1)
    tops_stride = _tops_stride(tops, rows, width)
    dev = logits.device
    if out is None:
        out = torch.empty((rows, n + n // 32), dtype=torch.int32, device=dev)
    if valid is None:
        valid = torch.empty(rows, dtype=torch.int32, device=dev)
    _outputs(out, valid, rows, n + n // 32)
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    opt = None
    if counters is not None or force_exact or hold:
        opt = ctypes.byref(_Options(1 if force_exact else 0, 0,
                                    None if counters is None else counters.data_ptr(), 0, 1 if hold else 0))
    with torch.cuda.device(dev):
        st = load().topk_bf16_select_words(_ptr(logits), row_stride, rows, width, _ptr(valid_len), int(n),
                                           _ptr(tops), tops_stride, _ptr(out), _ptr(valid),
                                           ctypes.c_void_p(stream.cuda_stream), opt)
    _check(st)
    return out, valid


def tops(logits, valid_len, width: int | None = None, stream=None):
    """The per-8 maxima select_ordered is bounded by (topk_bf16_tops): int16
    [rows, ceil(ceil(width / 8) / 8) * 8] holding uint16 order keys."""
    import torch
    rows, width, row_stride, _ = _inputs(logits, valid_len, None, width, 1)
    stride = -(-(-(-width // 8)) // 8) * 8
    out = torch.empty((rows, max(stride, 8)), dtype=torch.int16, device=logits.device)
    if stream is None:
        stream = torch.cuda.current_stream(logits.device)
    with torch.cuda.device(logits.device):
        _check(load().topk_bf16_tops(_ptr(logits), row_stride, rows, width, _ptr(valid_len), _ptr(out),
                                     out.shape[1], ctypes.c_void_p(stream.cuda_stream)))
    return out


def _tops_stride(tops, rows: int, width: int) -> int:
    """Checks the per-8 maxima tensor of select_ordered / select_words and
    returns its row stride (0 for None). Every row must hold the row's whole
    16-byte pieces of maxima: ceil(ceil(width / 8) / 8) * 8 entries."""
    if tops is None:
        return 0
    need = -(-(-(-width // 8)) // 8) * 8
    if not (tops.is_cuda and tops.element_size() == 2 and tops.dim() == 2 and tops.shape[0] >= rows
            and tops.stride(1) == 1 and tops.shape[1] >= need):
        raise ValueError(f"tops must be CUDA 16-bit [rows, >= {need}] with unit inner stride")
    return tops.stride(0) if tops.shape[0] > 1 else tops.shape[1]


def _outputs(out, valid, rows: int, cols: int):
    """Checks caller-provided output tensors (the kernels write rows x cols
    int32 words to out and rows words to valid)."""
    import torch
    for t, shape in ((out, (rows, cols)), (valid, (rows,))):
        if not (isinstance(t, torch.Tensor) and t.is_cuda and t.dtype == torch.int32
                and tuple(t.shape) == shape and t.is_contiguous()):
            raise ValueError(f"out / valid must be contiguous CUDA int32 {list((rows, cols))} / [{rows}]")


def _inputs(logits, valid_len, block_table, width, rows_per_request):
    """Checks shared by the entry points; returns (rows, width, row_stride, table_stride)."""
    import torch
    if not (isinstance(logits, torch.Tensor) and logits.is_cuda):
        raise TypeError("logits must be a CUDA tensor")
    if logits.dtype not in (torch.bfloat16, torch.int16) and str(logits.dtype) != "torch.uint16":
        raise TypeError("logits must be bfloat16 (or 16-bit BF16 bits)")
    if logits.dim() != 2 or (logits.shape[1] > 1 and logits.stride(1) != 1):
        raise ValueError("logits must be 2-D with unit inner stride")
    rows, cols = logits.shape
    width = cols if width is None else int(width)
    if width > cols:
        raise ValueError("width exceeds the logits' columns")
    row_stride = logits.stride(0) if rows > 1 else -(-cols // 8) * 8
    # The kernels read whole 16-byte vectors: each row must be readable up to
    # the next multiple of 8 logits.
    span = logits.storage_offset() + max(rows - 1, 0) * row_stride + -(-width // 8) * 8
    if rows and span * 2 > logits.untyped_storage().nbytes():
        raise ValueError("each row must be readable up to a multiple of 8 logits")
    if not (valid_len.is_cuda and valid_len.dtype == torch.int32 and valid_len.numel() == rows
            and valid_len.is_contiguous()):
        raise ValueError("valid_len must be a contiguous CUDA int32 tensor with one entry per row")
    table_stride = 0
    if block_table is not None:
        requests = -(-rows // max(int(rows_per_request), 1))
        if not (block_table.is_cuda and block_table.dtype == torch.int32 and block_table.dim() == 2
                and block_table.shape[0] >= requests and block_table.stride(1) == 1):
            raise ValueError("block_table must be CUDA int32 [ceil(rows / rows_per_request), pages] "
                             "with unit inner stride")
        table_stride = block_table.stride(0) if block_table.shape[0] > 1 else block_table.shape[1]
    return rows, width, row_stride, table_stride


def select_raw(logits_ptr: int, row_stride: int, rows: int, width: int, valid_len_ptr: int, k: int,
               mode: int, table_ptr: int | None, table_stride: int, page_size: int, out_ptr: int,
               stream_handle: int) -> None:
    """The C entry point on raw device pointers (no checks beyond the library's)."""
    _check(load().topk_bf16_select(logits_ptr, row_stride, rows, width, valid_len_ptr, k, mode,
                                   table_ptr, table_stride, page_size, out_ptr,
                                   ctypes.c_void_p(stream_handle)))


def plan(rows: int, width: int, k: int, mode: int = TOKEN) -> dict:
    """The launch the library would make: CTAs per row, threads, shared bytes, variant,
    CTAs launched."""
    c, t, s, v, n = (ctypes.c_int32() for _ in range(5))
    _check(load().topk_bf16_plan(rows, width, k, mode, ctypes.byref(c), ctypes.byref(t),
                                 ctypes.byref(s), ctypes.byref(v), ctypes.byref(n)))
    return {"cluster": c.value, "threads": t.value, "smem_bytes": s.value,
            "variant": ("one-tile", "streamed", "direct")[v.value], "ctas": n.value}


def device_status(clear: bool = True) -> int:
    """Device-side status bits (bounded wait gave up = 1, capacity or range check = 2,
    shared-memory index out of range in a -DTOPK_DEBUG build = 4); syncs the device."""
    flags = ctypes.c_uint32()
    _check(load().topk_bf16_device_status(ctypes.byref(flags), 1 if clear else 0))
    return flags.value


def status_string(status: int) -> str:
    return load().topk_bf16_status_string(status).decode()
