"""The hold launch option (the kernel does not release the next grid on the
stream early). It changes launch order only. So every kernel must give the same
result with and without it. This holds for one launch, for launches back to back
on one stream (each launch then waits for the whole previous grid), and inside a
CUDA graph."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import exact_bf16_top_gb300 as tk
import oracle
import workloads as W
from gpu_util import assert_same_sets, run_gpu, run_oracle, upload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _setup():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    tk._build.build()
    oracle.build()
    tk.device_status(clear=True)
    yield
    assert tk.device_status(clear=True) == 0


def _cases():
    return [
        ("one-tile", W.config2(32, 9000, 512), {}),
        ("streamed", W.ragged_case(seed=71, rows=6, width=100003, row_stride=100008, k=512,
                                   mode=W.TOKEN, with_table=True), {"path": 1}),
        ("resident-keys", W.ragged_case(seed=72, rows=6, width=100003, row_stride=100008, k=300,
                                        mode=W.BLOCK8, with_table=True), {"path": 2}),
    ]


@pytest.mark.parametrize("name,case,opts", _cases(), ids=lambda x: x if isinstance(x, str) else "")
def test_hold_same_result(name, case, opts):
    exp = run_oracle(case)
    assert_same_sets(run_gpu(case, hold=True, **opts), exp, name + " hold")
    assert_same_sets(run_gpu(case, **opts), exp, name)


def test_hold_back_to_back_and_in_a_graph():
    # Alternate held and released launches of two different workloads on one
    # stream, eagerly and captured in a graph; every output must be exact.
    a, b = W.config2(128, 16384, 512, seed=3), W.ragged_case(seed=73, rows=5, width=70001,
                                                             row_stride=70008, k=512,
                                                             mode=W.TOKEN, with_table=True)
    ea, eb = run_oracle(a), run_oracle(b)
    la, va, ta = upload(a)
    lb, vb, tb = upload(b)
    oa = torch.empty((a.rows, a.k), dtype=torch.int32, device="cuda")
    ob = torch.empty((b.rows, b.k), dtype=torch.int32, device="cuda")
    s = torch.cuda.Stream()

    def step(i):
        tk.select(la, va, a.k, a.mode, ta, a.page_size, out=oa, width=a.width, stream=s, hold=i % 2 == 0)
        tk.select(lb, vb, b.k, b.mode, tb, b.page_size, out=ob, width=b.width, stream=s, hold=i % 3 == 0)

    for i in range(4):
        step(i)
    s.synchronize()
    assert_same_sets(oa.cpu().numpy(), ea, "eager a")
    assert_same_sets(ob.cpu().numpy(), eb, "eager b")
    oa.fill_(-7)
    ob.fill_(-7)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for i in range(4):
            step(i)
    g.replay()
    torch.cuda.synchronize()
    assert_same_sets(oa.cpu().numpy(), ea, "graph a")
    assert_same_sets(ob.cpu().numpy(), eb, "graph b")


def test_hold_ordered_and_words():
    case = W.paged_case(77, rows=20, width=40000, k=512, q=2, block_rows=2048)
    logits, valid, table = upload(case)
    tops = tk.tops(logits, valid, width=case.width)
    exp = oracle.topk_ordered(case.logits, case.valid_len, case.k, case.block_table, case.page_size,
                              width=case.width, threads=16, block_rows=case.block_rows,
                              rows_per_request=case.rows_per_request)
    for hold in (True, False):
        out, cnt, ids = tk.select_ordered(logits, valid, case.k, tops, table, case.page_size,
                                          width=case.width, block_rows=case.block_rows,
                                          rows_per_request=case.rows_per_request, ids=True, hold=hold)
        torch.cuda.synchronize()
        for g, e in zip((out, cnt, ids), exp):
            assert np.array_equal(g.cpu().numpy(), e), hold
    wexp = oracle.topk_words(case.logits, case.valid_len, 512, width=case.width)
    for hold in (True, False):
        out, cnt = tk.select_words(logits, valid, 512, tops, width=case.width, hold=hold)
        torch.cuda.synchronize()
        assert np.array_equal(cnt.cpu().numpy(), wexp[1]), hold
        assert np.array_equal(out.cpu().numpy(), wexp[0]), hold


@pytest.fixture(scope="module")
def early_consumer(tmp_path_factory):
    """The test helper tests/pdl_consumer.cu built with nvcc (sm_103a)."""
    import ctypes
    import os
    import subprocess
    src = os.path.join(os.path.dirname(os.path.abspath(__file__)), "pdl_consumer.cu")
    so = str(tmp_path_factory.mktemp("pdl") / "libpdl_consumer.so")
    nvcc = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    subprocess.run([nvcc if os.path.exists(nvcc) else "nvcc", "-gencode", "arch=compute_103a,code=sm_103a",
                    "-O2", "-shared", "-Xcompiler", "-fPIC", "-o", so, src], check=True, capture_output=True)
    lib = ctypes.CDLL(so)
    lib.launch_copy_early.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p]
    lib.launch_copy_early.restype = ctypes.c_int
    return lib


def test_hold_keeps_an_early_reader_from_stale_output(early_consumer):
    """A consumer that reads the output before waiting for the preceding grid
    (launched with programmatic stream serialization) must see the finished
    output when the select was launched with hold: the output is pre-filled
    with a marker before every select, and the early copy must equal the
    oracle's selection every time."""
    case = W.config2(32, 9000, 512, seed=4)
    ctas = tk.plan(case.rows, case.width, case.k, case.mode)["ctas"]
    assert ctas < torch.cuda.get_device_properties(0).multi_processor_count  # a spare-slot launch
    logits, valid, table = upload(case)
    exp = np.sort(run_oracle(case), 1)
    out = torch.empty((case.rows, case.k), dtype=torch.int32, device="cuda")
    copy = torch.empty_like(out)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        for _ in range(20):
            out.fill_(-7)
            tk.select(logits, valid, case.k, case.mode, table, case.page_size, out=out, hold=True, stream=s)
            assert early_consumer.launch_copy_early(out.data_ptr(), copy.data_ptr(), out.numel(),
                                                    s.cuda_stream) == 0
            s.synchronize()
            assert np.array_equal(np.sort(copy.cpu().numpy(), 1), exp)
