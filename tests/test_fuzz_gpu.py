"""Seeded random configurations through every entry point, bit-exact against
the oracle: row counts, widths (ragged strides), k, mode, tables, requests of
several rows, value mixes (N(0,1), few distinct values, constants, ascending,
raw bit patterns with NaN and infinities), cluster sizes and paths."""
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


def _values(rng, rows, stride, kind):
    if kind == 0:
        return W.normal_bf16(rng, (rows, stride))
    if kind == 1:   # few distinct values: crowded bins and ties
        pool = W.normal_bf16(rng, (7,))
        return pool[rng.integers(0, 7, size=(rows, stride))]
    if kind == 2:   # constant rows
        return np.full((rows, stride), W.normal_bf16(rng, (1,))[0], np.uint16)
    if kind == 3:   # ascending rows
        return W.to_bf16_bits(np.sort(rng.standard_normal((rows, stride), dtype=np.float32), axis=1))
    return rng.integers(0, 1 << 16, size=(rows, stride)).astype(np.uint16)   # raw bit patterns


def _case(seed, token_only=False):
    rng = W.rng_for(1000 + seed)
    mode = int(rng.integers(0, 2))
    if token_only:
        mode = W.TOKEN
    width = int(rng.choice([int(rng.integers(1, 5000)), int(rng.integers(5000, 40000)),
                            int(rng.integers(40000, 300000))]))
    stride = -(-width // 8) * 8 + 8 * int(rng.integers(0, 3))
    rows = int(rng.integers(1, 60 if width > 40000 else 300))
    k = int(rng.choice([1, int(rng.integers(2, 200)), 512, int(rng.integers(512, 2049))]))
    logits = _values(rng, rows, stride, int(rng.integers(0, 5)))
    valid = rng.integers(0, width + 1, size=rows).astype(np.int32)
    q = int(rng.choice([1, 1, 2, 3]))
    table, block_rows = None, None
    if rng.random() < 0.6:
        n_width = width if mode == W.TOKEN else -(-width // 8)
        table = W.permuted_table(rng, -(-rows // q), n_width)
        block_rows = int(rng.choice([64, 128, 2048]))
    else:
        q = 1
    case = W.Case(f"fuzz{seed}", logits, width, valid, k, mode, table, 64,
                  block_rows=block_rows, rows_per_request=q)
    return case, rng


def _dev(case):
    return (torch.from_numpy(np.ascontiguousarray(case.logits).view(np.int16)).cuda(),
            torch.from_numpy(case.valid_len).cuda(),
            None if case.block_table is None else torch.from_numpy(case.block_table).cuda())


@pytest.mark.parametrize("seed", range(96))
def test_fuzz_select(seed):
    case, rng = _case(seed)
    logits, valid, table = _dev(case)
    exp = oracle.topk(case.logits, case.valid_len, case.k, case.mode, case.block_table, 64,
                      width=case.width, threads=16, block_rows=case.block_rows,
                      rows_per_request=case.rows_per_request)
    opts = {}
    if case.rows_per_request == 1 and (case.block_rows in (None, 64)):
        opts = dict(rng.choice([{}, {"cluster": 2}, {"cluster": 8}, {"path": 1}, {"path": 2},
                                {"force_direct": True}]))
    paged = dict(block_rows=case.block_rows, rows_per_request=case.rows_per_request) \
        if (case.block_rows not in (None, 64) or case.rows_per_request != 1) else {}
    got = tk.select(logits, valid, case.k, case.mode, table, 64, width=case.width, **opts, **paged)
    torch.cuda.synchronize()
    assert tk.device_status() == 0
    g, e = np.sort(got.cpu().numpy(), 1), np.sort(exp, 1)
    assert np.array_equal(g, e), (case.name, case.rows, case.width, case.k, case.mode, opts,
                                  int((g != e).any(1).sum()))


@pytest.mark.parametrize("seed", range(96, 144))
def test_fuzz_ordered_and_words(seed):
    case, rng = _case(seed, token_only=True)
    logits, valid, table = _dev(case)
    tops = tk.tops(logits, valid, width=case.width)
    out, cnt, ids = tk.select_ordered(logits, valid, case.k, tops if rng.random() < 0.8 else None, table, 64,
                                      width=case.width, block_rows=case.block_rows,
                                      rows_per_request=case.rows_per_request, ids=True)
    exp = oracle.topk_ordered(case.logits, case.valid_len, case.k, case.block_table, 64, width=case.width,
                              threads=16, block_rows=case.block_rows, rows_per_request=case.rows_per_request)
    torch.cuda.synchronize()
    for g, e, what in zip((out, cnt, ids), exp, ("out", "valid", "ids")):
        assert np.array_equal(g.cpu().numpy(), e), (case.name, what)
    if case.width <= (1 << 17):
        n = max(32, (min(case.k, 2048) // 32) * 32)
        w, wc = tk.select_words(logits, valid, n, tops, width=case.width)
        ew, ec = oracle.topk_words(case.logits, case.valid_len, n, width=case.width)
        torch.cuda.synchronize()
        assert np.array_equal(w.cpu().numpy(), ew) and np.array_equal(wc.cpu().numpy(), ec), (case.name, "words")
    assert tk.device_status() == 0
