"""Helpers for the GPU tests: upload a workloads.Case, run the CUDA path through
the C ABI, and compare with the oracle (sorted rows, bit-exact)."""
from __future__ import annotations

import os

import numpy as np
import torch

import exact_bf16_top_gb300 as tk
import oracle

THREADS = os.cpu_count() or 4


def upload(case, device="cuda"):
    logits = torch.from_numpy(np.ascontiguousarray(case.logits).view(np.int16)).to(device)
    valid = torch.from_numpy(np.ascontiguousarray(case.valid_len)).to(device)
    table = None if case.block_table is None else torch.from_numpy(case.block_table).to(device)
    return logits, valid, table


def run_gpu(case, **opts):
    logits, valid, table = upload(case)
    if case.block_rows is not None or case.rows_per_request != 1:
        opts = dict(opts, block_rows=case.block_rows, rows_per_request=case.rows_per_request)
    out = tk.select(logits, valid, case.k, case.mode, table, case.page_size, width=case.width, **opts)
    torch.cuda.synchronize()
    return out.cpu().numpy()


def run_oracle(case):
    return oracle.topk(case.logits, case.valid_len, case.k, case.mode, case.block_table,
                       case.page_size, width=case.width, threads=THREADS,
                       block_rows=case.block_rows, rows_per_request=case.rows_per_request)


def assert_same_sets(got, exp, name=""):
    g = np.sort(got, axis=1)
    e = np.sort(exp, axis=1)
    bad = np.flatnonzero((g != e).any(axis=1))
    if len(bad):
        r = int(bad[0])
        diff_g = sorted(set(g[r].tolist()) - set(e[r].tolist()))[:10]
        diff_e = sorted(set(e[r].tolist()) - set(g[r].tolist()))[:10]
        raise AssertionError(f"{name}: {len(bad)} rows differ; first row {r}: "
                             f"extra {diff_g}, missing {diff_e}")
