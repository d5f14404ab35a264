"""topk_bf16_select_static, the entry point that allocates nothing.

Some callers cannot allocate device memory: code recorded into a CUDA graph by
stream capture, where an allocation would be captured too; programs that hand
all device memory to one pool up front and leave no allocator to call; and
plug-ins whose host application owns every allocation. This entry point keeps
its per-row working table in a static array inside the library, so its callers
pass only inputs and outputs. Its results must match topk_bf16_select's exactly
(the selected index sets), on consecutive calls that share that table.

This file is collected last so that it also runs after every other test has
left the library's per-device state behind; it passes alone as well.
"""
from __future__ import annotations

import ctypes

import numpy as np
import pytest
import torch

import exact_bf16_top_gb300 as tk
import workloads as W
from gpu_util import assert_same_sets, upload

MAX_ROWS = 65536
MAX_WIDTH = 16384


@pytest.fixture(scope="module")
def lib():
    # The release library, whatever an earlier test left as the binding's default.
    tk._build.build()
    lib = tk.load(tk.library_path())
    saved, tk._lib = tk._lib, lib
    yield lib
    tk._lib = saved


def test_sizes_beyond_the_table_are_rejected_on_the_host(lib):
    # Fake, aligned device addresses: the call must refuse before it touches CUDA.
    def call(rows, width):
        return lib.topk_bf16_select_static(4096, width, rows, width, 8192, 8, tk.TOKEN, None, 0, 64,
                                           4096 * 16, None)

    assert call(MAX_ROWS + 1, MAX_WIDTH) == 6
    assert call(1, MAX_WIDTH + 8) == 6
    assert call(-1, MAX_WIDTH) == 1
    assert tk.status_string(6)


def _select_both(case, garbage_seed):
    logits, valid, table = upload(case)
    gen = torch.Generator(device="cpu").manual_seed(garbage_seed)
    fill = torch.randint(-5, 1 << 20, (case.logits.shape[0], case.k), generator=gen,
                         dtype=torch.int32).cuda()
    out_static = fill.clone()
    tk.select_static(logits, valid, case.k, out_static, case.mode, table, case.page_size,
                     width=case.width)
    out_ref = tk.select(logits, valid, case.k, case.mode, table, case.page_size, width=case.width)
    torch.cuda.synchronize()
    return out_static.cpu().numpy(), out_ref.cpu().numpy()


def _cases():
    # Two calls in a row per mode: the second call's rows start from the cuts
    # the first call left in the shared table, over different data.
    token = [W.config2(512, 9000, 512, seed=3), W.config2(512, 16384, 512, seed=4)]
    block = [W.config2(64, 16384, 256, seed=5), W.config2(64, 12000, 256, seed=6)]
    for c in block:
        c.mode = tk.BLOCK8
        c.block_table = None
        c.name = c.name.replace("consumer", "block")
    return token, block


@pytest.mark.gpu
def test_static_entry_matches_select_on_two_calls_in_a_row(lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    tk.device_status(clear=True)
    for pair in _cases():
        for i, case in enumerate(pair):
            got, exp = _select_both(case, garbage_seed=i)
            assert_same_sets(got, exp, f"{case.name} call {i + 1}")
    assert tk.device_status(clear=True) == 0, "device status flags set"


@pytest.mark.gpu
def test_static_entry_refuses_oversized_calls_on_a_device(lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    logits = torch.zeros((2, MAX_WIDTH * 2), dtype=torch.int16, device="cuda")
    valid = torch.full((2,), 8, dtype=torch.int32, device="cuda")
    out = torch.zeros((2, 8), dtype=torch.int32, device="cuda")
    with pytest.raises(tk.TopkError) as e:
        tk.select_static(logits, valid, 8, out)
    assert e.value.status == 6
    assert torch.count_nonzero(out).item() == 0
