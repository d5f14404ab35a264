"""Pins for the CPU oracle (no GPU).

The oracle is checked against things other than itself: hand-derived cases
(tests/golden/hand_cases.json), a float-based brute force on tiny rows (which
never forms the 16-bit key), every one of the 65,536 BF16 bit patterns, the
invariants of an exact top-k, torch.topk on rows without NaN, closed-form
special rows, and the inverse of the block table. Finally, plausible mistakes
are planted in copies of the oracle's C source and each must be caught.
"""
from __future__ import annotations

import json
import os
import shutil
import tempfile

import numpy as np
import pytest
import torch

import oracle
import workloads
from bruteforce import topk_row

HERE = os.path.dirname(os.path.abspath(__file__))


# ------------------------------------------------------------------ helpers

def bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32)


def rank_values(bits: np.ndarray) -> np.ndarray:
    """Real-number order with -0 just below +0 (float64; NaN stays NaN)."""
    with np.errstate(invalid="ignore"):
        f = bits_to_f32(bits).astype(np.float64)
    zero = f == 0.0
    return np.where(zero, np.where(np.signbit(f), -1e-300, 1e-300), f)


def golden_cases():
    with open(os.path.join(HERE, "golden", "hand_cases.json")) as fh:
        data = json.load(fh)
    for c in data["cases"]:
        width = c["width"]
        if "logits" in c:
            row = np.array([int(h, 16) for h in c["logits"]], np.uint16)
        else:
            row = np.full(width, int(c["fill"], 16), np.uint16)
            for pos, h in c.get("set", {}).items():
                row[int(pos)] = int(h, 16)
        assert row.shape[0] == width, c["name"]
        table = np.array([c["table"]], np.int32) if "table" in c else None
        yield c, row, table


def check_golden(lib) -> list[str]:
    """Each row sits in a wider buffer whose columns past the row's width hold
    +inf, so a valid length that is not clamped to the width reads them (and
    selects them) instead of reading past the buffer."""
    bad = []
    for c, row, table in golden_cases():
        buf = np.full((1, row.shape[0] + 64), 0x7F80, np.uint16)
        buf[0, :row.shape[0]] = row
        got = oracle.topk(buf, [c["valid_len"]], c["k"], c["mode"], table, width=row.shape[0], lib=lib)
        if sorted(got[0].tolist()) != c["expected"]:
            bad.append(f"golden {c['name']}: {sorted(got[0].tolist())} != {c['expected']}")
    return bad + check_paged_golden(lib)


def check_paged_golden(lib) -> list[str]:
    """tests/golden/paged_cases.json: requests of several rows, block rows != page."""
    with open(os.path.join(HERE, "golden", "paged_cases.json")) as fh:
        data = json.load(fh)
    bad = []
    for c in data["cases"]:
        rows = []
        for r in c["rows"]:
            row = np.full(c["width"], int(r["fill"], 16), np.uint16)
            for pos, h in r.get("set", {}).items():
                row[int(pos)] = int(h, 16)
            rows.append(row)
        got = oracle.topk(np.stack(rows), [r["valid_len"] for r in c["rows"]], c["k"], c["mode"],
                          np.array(c["table"], np.int32), c["page_size"], lib=lib,
                          block_rows=c["block_rows"], rows_per_request=c["rows_per_request"])
        got = [sorted(g.tolist()) for g in got]
        if got != c["expected"]:
            bad.append(f"paged golden {c['name']}: {got} != {c['expected']}")
    return bad


def _tiny_rows(rng, n):
    """Tiny rows of several kinds: raw bit patterns, N(0,1), heavy ties, specials."""
    specials = np.array([0x0000, 0x8000, 0x7F80, 0xFF80, 0x7FC0, 0xFFC0, 0x0001, 0x8001,
                         0x3F80, 0xBF80, 0x7F7F, 0xFF7F], np.uint16)
    yield rng.integers(0, 1 << 16, size=n).astype(np.uint16)
    yield workloads.normal_bf16(rng, (n,))
    yield specials[rng.integers(0, len(specials), size=n)]
    yield np.array([0x3F80, 0x4000, 0x8000, 0x0000], np.uint16)[rng.integers(0, 4, size=n)]


def check_bruteforce(lib, seed: int = 1, trials: int = 3) -> list[str]:
    rng = workloads.rng_for(seed)
    bad = []
    for _ in range(trials):
        for width in (1, 5, 8, 13, 24, 40, 64):
            for row in _tiny_rows(rng, width):
                for mode in (0, 1):
                    L = int(rng.integers(0, width + 1))
                    n = L if mode == 0 else (L + 7) // 8
                    pages = max(1, -(-max(width, 1) // 4))
                    table = rng.permutation(pages * 3)[:pages].astype(np.int32)
                    for k in range(1, n + 3):
                        for tbl in (None, table):
                            exp = topk_row(row.tolist(), L, k, mode, tbl, page=4)
                            got = oracle.topk(row[None, :], [L], k, mode,
                                              None if tbl is None else tbl[None, :], page_size=4,
                                              lib=lib)[0].tolist()
                            if sorted(got) != sorted(exp):
                                bad.append(f"brute mode{mode} L{L} k{k} row={row.tolist()}: "
                                           f"{sorted(got)} != {sorted(exp)}")
                                return bad
    return bad


def check_all_patterns(lib, ks=(1, 2, 3, 255, 4096, 32767, 32768, 65000)) -> list[str]:
    """One row holding every BF16 bit pattern once, shuffled; several k."""
    rng = workloads.rng_for(7)
    row = rng.permutation(1 << 16).astype(np.uint16)
    bad = []
    for k in ks:
        exp = sorted(topk_row(row.tolist(), 1 << 16, k, 0))
        got = sorted(oracle.topk(row[None, :], [1 << 16], k, 0, lib=lib)[0].tolist())
        if got != exp:
            bad.append(f"all-patterns k{k}")
    return bad


# ------------------------------------------------------------------ pins

def test_golden_cases():
    assert check_golden(oracle.load()) == []


def test_bruteforce_tiny_rows():
    assert check_bruteforce(oracle.load()) == []


def test_every_bf16_pattern():
    assert check_all_patterns(oracle.load()) == []


def _check_invariants(bits, L, k, got):
    """Count, threshold and tie invariants of an exact top-k (token mode, no table)."""
    if L <= k:                      # short row: 0 .. L-1 whatever the values
        assert got.tolist() == list(range(L)) + [-1] * (k - L)
        return
    r = rank_values(bits[:L])
    nonnan = np.flatnonzero(~np.isnan(r))
    sel = got[got >= 0]
    assert len(set(sel.tolist())) == len(sel), "duplicate index"
    assert len(sel) == min(k, len(nonnan)), "count != min(k, #non-NaN)"
    assert np.all(sel < L)
    assert not np.any(np.isnan(r[sel])), "NaN selected"
    if len(sel) < k:
        return
    kth = r[sel].min()
    above = nonnan[r[nonnan] > kth]
    assert set(above.tolist()) <= set(sel.tolist()), "a value above the k-th is missing"
    ties = nonnan[r[nonnan] == kth]
    taken = np.sort(sel[r[sel] == kth])
    assert np.array_equal(taken, ties[: len(taken)]), "ties are not the lowest indices"


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_invariants_random_rows(seed):
    rng = workloads.rng_for(seed)
    width = 20011
    rows = [workloads.normal_bf16(rng, (width,)),
            rng.integers(0, 1 << 16, size=width).astype(np.uint16),
            np.array([0x3F80, 0x4000, 0x8000, 0x0000, 0x7FC0], np.uint16)[rng.integers(0, 5, width)]]
    logits = np.stack(rows)
    for k in (1, 511, 512, 2048, 19000):
        L = np.array([width, width - 7, 12345], np.int32)
        got = oracle.topk(logits, L, k, 0)
        for i in range(len(rows)):
            _check_invariants(logits[i], int(L[i]), k, got[i])


def test_against_torch_topk():
    """Value multiset equals torch.topk's on NaN-free rows; with distinct values
    the index sets are equal (sglang PR #39305, Accuracy: checked as a multiset
    against torch.topk)."""
    rng = workloads.rng_for(3)
    logits = workloads.normal_bf16(rng, (6, 16384))
    for k in (64, 512, 2048):
        got = oracle.topk(logits, np.full(6, 16384), k, 0)
        f = torch.from_numpy(bits_to_f32(logits))
        ref = torch.topk(f, k, dim=1)
        for r in range(6):
            vals = np.sort(bits_to_f32(logits[r])[got[r]])
            assert np.array_equal(vals, np.sort(ref.values[r].numpy()))
    distinct = np.stack([rng.permutation(np.arange(0x3C00, 0x3C00 + 8192)).astype(np.uint16)
                         for _ in range(3)])
    got = oracle.topk(distinct, np.full(3, 8192), 300, 0)
    ref = torch.topk(torch.from_numpy(bits_to_f32(distinct)), 300, dim=1).indices.numpy()
    for r in range(3):
        assert set(got[r].tolist()) == set(ref[r].tolist())


def test_special_rows():
    n, k = 4096, 100
    const = np.full((1, n), 0x3F80, np.uint16)
    assert sorted(oracle.topk(const, [n], k, 0)[0].tolist()) == list(range(k))
    inc = (0x3C00 + np.arange(n)).astype(np.uint16)[None, :]     # strictly increasing values
    assert sorted(oracle.topk(inc, [n], k, 0)[0].tolist()) == list(range(n - k, n))
    ninf = np.full((1, n), 0xFF80, np.uint16)
    assert sorted(oracle.topk(ninf, [n], k, 0)[0].tolist()) == list(range(k))
    got = oracle.topk(ninf, [n], k, 1)[0].tolist()           # block: only the newest block
    assert sorted(got) == [-1] * (k - 1) + [n // 8 - 1]
    for L in (0, 1, 50, 100):
        assert oracle.topk(const, [L], k, 0)[0].tolist() == list(range(L)) + [-1] * (k - L)


def test_transform_inverse():
    """Mapping physical ids back through the inverse table recovers the logical set."""
    case = workloads.config2(rows=8, valid=9000, k=512, seed=5)
    phys = oracle.topk(case.logits, case.valid_len, case.k, 0, case.block_table)
    logical = oracle.topk(case.logits, case.valid_len, case.k, 0)
    inv = {}
    for r in range(case.rows):
        for p, pid in enumerate(case.block_table[r]):
            inv[int(pid)] = (r, p)
    for r in range(case.rows):
        back = []
        for x in phys[r]:
            rr, p = inv[int(x) // 64]
            assert rr == r
            back.append(p * 64 + int(x) % 64)
        assert sorted(back) == sorted(logical[r].tolist())


def test_threads_give_same_result():
    case = workloads.ragged_case(4, rows=13, width=5000, row_stride=5008, k=300)
    a = oracle.topk(case.logits, case.valid_len, case.k, 0, width=case.width, threads=1)
    b = oracle.topk(case.logits, case.valid_len, case.k, 0, width=case.width, threads=4)
    assert np.array_equal(a, b)


# ------------------------------------------------- planted mistakes are caught

MUTANTS = [
    ("ties to the highest index",
     [("(uint64_t)(0xFFFFFFFFu - (uint32_t)i)", "(uint64_t)(uint32_t)i"),
      ("return (int32_t)(0xFFFFFFFFu - (uint32_t)w);", "return (int32_t)(uint32_t)w;")]),
    ("positive/negative key masks swapped", [("? 0xFFFFu : 0x8000u", "? 0x8000u : 0xFFFFu")]),
    ("negatives not reversed", [("? 0xFFFFu : 0x8000u", "? 0x7FFFu : 0x8000u")]),
    ("infinities taken for NaN", [("(x & 0x7FFFu) > 0x7F80u", "(x & 0x7FFFu) >= 0x7F80u")]),
    ("newest block not pinned", [("if (i == n - 1) { nan = 0; key = KEY_POS_INF; }", "")]),
    ("-inf blocks not written as -1", [("j->mode == ORACLE_BLOCK8 && key == KEY_NEG_INF", "0")]),
    ("bypass misses n == k", [("if (n <= j->k) {", "if (n < j->k) {")]),
    ("page offset dropped", [("page_id * j->block_rows + i % j->page", "page_id * j->block_rows")]),
    ("page size taken for block rows", [("page_id * j->block_rows + i % j->page", "page_id * j->page + i % j->page")]),
    ("request ignored", [("const int32_t request = r / j->rows_per_request;", "const int32_t request = r;")]),
    ("valid_len not clamped", [("if (L > j->width) L = j->width;", "")]),
    ("block minimum instead of maximum", [("order_key(row[t]) > key", "order_key(row[t]) < key")]),
    ("block NaN not propagated", [("if (is_nan_bf16(row[t])) nan = 1;", "if (0) nan = 1;")]),
    ("one too few selected", [("int32_t sel = m < j->k ? m : j->k;", "int32_t sel = (m < j->k ? m : j->k) - 1;")]),
    ("ascending sort", [("return x < y ? 1 : (x > y ? -1 : 0);", "return x < y ? -1 : (x > y ? 1 : 0);")]),
    ("last block group short by one", [("int32_t end = 8 * i + 8 < L ? 8 * i + 8 : L;",
                                        "int32_t end = 8 * i + 7 < L ? 8 * i + 7 : L;")]),
]


@pytest.mark.parametrize("name,edits", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_is_caught(name, edits):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "topk_oracle.c")).read()
    for old, new in edits:
        assert src.count(old) == 1, f"mutation anchor not found once: {old!r}"
        src = src.replace(old, new)
    tmp = tempfile.mkdtemp(prefix="oracle_mutant_")
    try:
        path = os.path.join(tmp, "m.c")
        with open(path, "w") as fh:
            fh.write(src)
        lib = oracle.load(oracle.build(force=True, src=path, out=os.path.join(tmp, "libm.so")))
        caught = check_golden(lib) or check_bruteforce(lib, trials=1) or check_all_patterns(lib)
        assert caught, f"planted mistake not caught: {name}"
    finally:
        shutil.rmtree(tmp, ignore_errors=True)
