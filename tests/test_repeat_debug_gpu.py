"""Parity repeated under changing L2 state, in the release library and in the
bounds-checked debug build (-DTOPK_DEBUG: every shared-memory index a kernel
computes from data is checked; a violation sets status bit 2 and the access is
skipped, never a trap). Each case runs 20 times through every entry point it
uses, with a 256 MB write between runs that evicts the previous run's data from
the 129 MB L2; every run must match the oracle bit for bit and leave the device
status word clean."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import exact_bf16_top_gb300 as tk
import oracle
import workloads as W
from gpu_util import run_oracle, upload

pytestmark = pytest.mark.gpu

REPEATS = 20


@pytest.fixture(scope="module", autouse=True)
def _setup():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    tk._build.build()
    oracle.build()


@pytest.fixture(scope="module", params=["release", "debug"])
def library(request, tmp_path_factory):
    """The library under test, installed as the binding's library for the test."""
    if request.param == "release":
        lib = tk.load()
    else:
        path = str(tmp_path_factory.mktemp("dbg") / "libtopk_bf16_debug.so")
        tk._build.build(force=True, out=path, extra_flags=["-DTOPK_DEBUG"])
        lib = tk.load(path)
    saved = tk._lib
    tk._lib = lib
    tk.device_status(clear=True)
    yield request.param
    status = tk.device_status(clear=True)
    tk._lib = saved
    assert status == 0, f"{request.param} library: device status {status:#x}"


def _cases():
    return [
        ("edges token", W.edge_cases(0)[0], {}),
        ("edges block", W.edge_cases(0)[1], {}),
        ("consumer", W.config2(64, 9000, 512, seed=5), {}),
        ("consumer k2048", W.config2(64, 4096, 2048, seed=6), {}),
        ("crowded streamed", W.config3(1, rows=16, width=60000), {}),
        ("block resident keys", W.config4(1, rows=4, width=1 << 18), {}),
        ("ragged streamed cluster", W.ragged_case(seed=21, rows=6, width=100003, row_stride=100008, k=512,
                                                  with_table=True), {"cluster": 4}),
        ("fallback rows", W.fallback_rows(2, rows=6, width=16384, k=512), {}),
    ]


def test_select_repeated(library):
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    for name, case, opts in _cases():
        exp = np.sort(run_oracle(case), 1)
        logits, valid, table = upload(case)
        for rep in range(REPEATS):
            flush.fill_(rep & 0xFF)
            got = tk.select(logits, valid, case.k, case.mode, table, case.page_size, width=case.width, **opts)
            torch.cuda.synchronize()
            assert np.array_equal(np.sort(got.cpu().numpy(), 1), exp), (library, name, rep)
        assert tk.device_status() == 0, (library, name)


def test_ordered_and_words_repeated(library):
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    case = W.paged_case(7, rows=8, width=40000, k=512, q=2, block_rows=2048)
    exp = oracle.topk_ordered(case.logits, case.valid_len, case.k, case.block_table, case.page_size,
                              width=case.width, block_rows=case.block_rows, rows_per_request=case.rows_per_request)
    ew, ec = oracle.topk_words(case.logits, case.valid_len, 256, width=case.width)
    logits, valid, table = upload(case)
    for rep in range(REPEATS):
        flush.fill_(rep & 0xFF)
        tops = tk.tops(logits, valid, width=case.width)
        out, cnt, ids = tk.select_ordered(logits, valid, case.k, tops, table, case.page_size, width=case.width,
                                          block_rows=case.block_rows, rows_per_request=case.rows_per_request,
                                          ids=True)
        words, wcnt = tk.select_words(logits, valid, 256, tops, width=case.width)
        torch.cuda.synchronize()
        for g, e in zip((out, cnt, ids), exp):
            assert np.array_equal(g.cpu().numpy(), e), (library, "ordered", rep)
        assert np.array_equal(words.cpu().numpy(), ew) and np.array_equal(wcnt.cpu().numpy(), ec), \
            (library, "words", rep)
    assert tk.device_status() == 0, library
