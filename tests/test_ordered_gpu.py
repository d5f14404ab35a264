"""Parity of the ordered select (bounded by per-8 maxima) and of the per-8
maxima kernel with the CPU oracle: out, valid and ids element by element."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import exact_bf16_top_gb300 as tk
import oracle
import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _setup():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    tk._build.build()


def _dev(case):
    logits = torch.from_numpy(np.ascontiguousarray(case.logits).view(np.int16)).cuda()
    valid = torch.from_numpy(case.valid_len).cuda()
    table = None if case.block_table is None else torch.from_numpy(case.block_table).cuda()
    return logits, valid, table


def run_ordered(case, use_tops=True, counters=None, force_exact=False, tops=None):
    logits, valid, table = _dev(case)
    if use_tops and tops is None:
        tops = tk.tops(logits, valid, width=case.width)
    out, cnt, ids = tk.select_ordered(logits, valid, case.k, tops if use_tops else None, table,
                                      case.page_size, width=case.width,
                                      block_rows=case.block_rows, rows_per_request=case.rows_per_request,
                                      ids=True, counters=counters, force_exact=force_exact)
    torch.cuda.synchronize()
    assert tk.device_status() == 0
    return out.cpu().numpy(), cnt.cpu().numpy(), ids.cpu().numpy()


def expected(case):
    return oracle.topk_ordered(case.logits, case.valid_len, case.k, case.block_table, case.page_size,
                               width=case.width, threads=16, block_rows=case.block_rows,
                               rows_per_request=case.rows_per_request)


def assert_same(got, exp, name):
    for g, e, what in zip(got, exp, ("out", "valid", "ids")):
        if not np.array_equal(g, e):
            bad = np.flatnonzero((g != e).reshape(g.shape[0], -1).any(axis=1))
            r = int(bad[0])
            raise AssertionError(f"{name}: {what} differs in {len(bad)} rows; row {r}: "
                                 f"got {g[r][:12]} exp {e[r][:12]}")


def test_tops_kernel_matches_oracle():
    for case in [W.paged_case(80, rows=29, width=20003, k=64, q=1),
                 W.edge_cases(3, width=4000, k=100)[0]]:
        logits, valid, _ = _dev(case)
        got = tk.tops(logits, valid, width=case.width).cpu().numpy().view(np.uint16)
        exp = oracle.tops(case.logits, case.valid_len, width=case.width)
        assert np.array_equal(got[:, :exp.shape[1]], exp), case.name
        assert (got[:, exp.shape[1]:] == 0).all()


@pytest.mark.parametrize("width,k,q,block_rows", [(16384, 512, 1, 64), (100003, 2048, 2, 2048),
                                                  (300000, 512, 4, 64), (1 << 20, 2048, 1, 64)])
def test_ordered_parity(width, k, q, block_rows):
    case = W.paged_case(90 + q, rows=37 if width < (1 << 20) else 9, width=width, k=k, q=q,
                        block_rows=block_rows)
    counters = torch.zeros(tk.NUM_COUNTERS, dtype=torch.int32, device="cuda")
    got = run_ordered(case, counters=counters)
    assert_same(got, expected(case), case.name)
    c = dict(zip(tk.COUNTER_NAMES, counters.cpu().numpy().tolist()))
    assert c["ordered_tops"] > 0, c


def test_ordered_wide_workload_sampled():
    """The benchmark's workload at full size, in the launch bench.py times; rows
    sampled for the oracle."""
    case = W.ordered_wide(0, rows=64)
    got = run_ordered(case)
    pick = [0, 17, 42, 63]
    sub = W.Case(case.name, case.logits[pick], case.width, case.valid_len[pick], case.k, W.TOKEN,
                 case.block_table[pick])
    exp = expected(sub)
    assert_same(tuple(g[pick] for g in got), exp, case.name)


def test_ordered_edges_and_exact_path():
    """Edge rows (ties, constants, -inf, signed zeros, NaN, short rows) through
    the bounded path, the exact path (forced), and without tops."""
    counters = torch.zeros(tk.NUM_COUNTERS, dtype=torch.int32, device="cuda")
    for width, k in ((16384, 512), (40000, 2048)):
        case = W.edge_cases(4, width=width, k=k)[0]
        exp = expected(case)
        assert_same(run_ordered(case, counters=counters), exp, case.name)
        assert_same(run_ordered(case, counters=counters, force_exact=True), exp, case.name + " exact")
        assert_same(run_ordered(case, use_tops=False), exp, case.name + " no tops")
    case = W.config3(1, rows=16, width=60000, k=512)   # crowded ties: lists overflow
    assert_same(run_ordered(case, counters=counters), expected(case), case.name)
    c = dict(zip(tk.COUNTER_NAMES, counters.cpu().numpy().tolist()))
    assert c["ordered_tops"] > 0 and c["ordered_exact"] > 0 and c["bypass_rows"] > 0, c


def run_words(case, n, use_tops=True, counters=None, force_exact=False):
    logits, valid, _ = _dev(case)
    tops = tk.tops(logits, valid, width=case.width) if use_tops else None
    out, cnt = tk.select_words(logits, valid, n, tops, width=case.width, counters=counters,
                               force_exact=force_exact)
    torch.cuda.synchronize()
    assert tk.device_status() == 0
    return out.cpu().numpy(), cnt.cpu().numpy()


@pytest.mark.parametrize("width,n", [(3000, 32), (20000, 512), (131072, 2048), (100000, 256)])
def test_words_parity(width, n):
    """The local top-n as B' words (every path: whole short rows, the bounded
    select, the exact one), bit-exact against the oracle, index plane included."""
    case = W.paged_case(110 + n, rows=24, width=width, k=n, q=1)
    exp = oracle.topk_words(case.logits, case.valid_len, n, width=case.width)
    counters = torch.zeros(tk.NUM_COUNTERS, dtype=torch.int32, device="cuda")
    for kw in ({}, {"force_exact": True}, {"use_tops": False}):
        got = run_words(case, n, counters=counters, **kw)
        assert np.array_equal(got[1], exp[1]), (case.name, kw)
        assert np.array_equal(got[0], exp[0]), (case.name, kw)
    c = dict(zip(tk.COUNTER_NAMES, counters.cpu().numpy().tolist()))
    assert c["ordered_exact"] > 0 and c["ordered_tops"] > 0, c


def test_words_edges():
    """Edge rows, short ones (lengths 0, 1, 7, ...) taken whole among them."""
    counters = torch.zeros(tk.NUM_COUNTERS, dtype=torch.int32, device="cuda")
    for width, n in ((16384, 512), (70000, 64)):
        case = W.edge_cases(5, width=width, k=n)[0]
        exp = oracle.topk_words(case.logits, case.valid_len, n, width=case.width)
        got = run_words(case, n, counters=counters)
        assert np.array_equal(got[0], exp[0]) and np.array_equal(got[1], exp[1]), case.name
    c = dict(zip(tk.COUNTER_NAMES, counters.cpu().numpy().tolist()))
    assert c["bypass_rows"] > 0, c


def test_binding_rejects_bad_outputs_and_tops():
    """Outputs and per-8 maxima the kernels would write or read past are refused
    on the host, before any launch: a short or wrongly typed out / valid for
    the B' words and the ordered select, and maxima narrower than the row's
    whole 16-byte pieces."""
    case = W.paged_case(3, rows=4, width=4000, k=256, q=1, block_rows=64)
    logits, valid, _ = _dev(case)
    tops = tk.tops(logits, valid, width=case.width)
    n = 256
    short = torch.empty((case.rows, n), dtype=torch.int32, device="cuda")   # needs n + n / 32
    with pytest.raises(ValueError):
        tk.select_words(logits, valid, n, tops, width=case.width, out=short)
    with pytest.raises(ValueError):
        tk.select_words(logits, valid, n, tops, width=case.width,
                        valid=torch.empty(case.rows - 1, dtype=torch.int32, device="cuda"))
    with pytest.raises(ValueError):
        tk.select_words(logits, valid, n, tops, width=case.width,
                        out=torch.empty((case.rows, n + n // 32), dtype=torch.int64, device="cuda"))
    with pytest.raises(ValueError):
        tk.select_ordered(logits, valid, n, tops, width=case.width,
                          out=torch.empty((case.rows, n + 1), dtype=torch.int32, device="cuda"))
    narrow = tops[:, :8]  # a column view: the row stride covers the row, the view does not
    with pytest.raises(ValueError):
        tk.select_ordered(logits, valid, n, narrow, width=case.width)
    with pytest.raises(ValueError):
        tk.select_words(logits, valid, n, narrow, width=case.width)
    torch.cuda.synchronize()
    assert tk.device_status() == 0
