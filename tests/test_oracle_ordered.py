"""Pins for the oracle's ordered select and per-8 maxima ("tops"), no GPU.

The ordered variant (vLLM kimi_k3 "dsa/indexer", IndexerSelect) writes the same
selection as the plain one in ascending element-index order, with per-row
counts and the untransformed indices. It is pinned by hand-derived cases
(tests/golden/ordered_cases.json), by the float brute force on tiny rows (its
selection, then sorted by index), by invariants on random rows, and by planted
mistakes. The tops are pinned without the key formula: they must rank the
values exactly as real numbers do (every BF16 pattern, -0 below +0), and each
group's top must be the top of its largest element alone.
"""
from __future__ import annotations

import json
import math
import os
import shutil
import tempfile

import numpy as np
import pytest

import oracle
import workloads
from bruteforce import bf16_value, topk_row

HERE = os.path.dirname(os.path.abspath(__file__))


def _golden():
    with open(os.path.join(HERE, "golden", "ordered_cases.json")) as fh:
        return json.load(fh)["cases"]


def check_ordered_golden(lib) -> list[str]:
    bad = []
    for c in _golden():
        row = np.array([int(h, 16) for h in c["logits"]], np.uint16)[None, :]
        table = np.array([c["table"]], np.int32) if "table" in c else None
        out, valid, ids = oracle.topk_ordered(row, [c["valid_len"]], c["k"], table, c["page_size"],
                                              block_rows=c["block_rows"], lib=lib)
        got = (out[0].tolist(), int(valid[0]), ids[0].tolist())
        exp = (c["expected_out"], c["expected_valid"], c["expected_ids"])
        if got != exp:
            bad.append(f"ordered golden {c['name']}: {got} != {exp}")
        tops = oracle.tops(row, [c["valid_len"]], lib=lib)[0].tolist()
        if tops != [int(h, 16) for h in c["expected_tops"]]:
            bad.append(f"tops golden {c['name']}: {[hex(t) for t in tops]}")
    return bad


def check_ordered_bruteforce(lib, seed: int = 3, trials: int = 2) -> list[str]:
    """The float brute force's selection (logical indices), sorted ascending,
    then transformed; counts and ids alongside."""
    rng = workloads.rng_for(seed)
    specials = np.array([0x0000, 0x8000, 0x7F80, 0xFF80, 0x7FC0, 0x3F80, 0xBF80, 0x4000], np.uint16)
    for _ in range(trials):
        for width in (1, 7, 8, 9, 24, 40):
            rows = [rng.integers(0, 1 << 16, size=width).astype(np.uint16),
                    workloads.normal_bf16(rng, (width,)),
                    specials[rng.integers(0, len(specials), size=width)]]
            for row in rows:
                L = int(rng.integers(0, width + 1))
                pages = max(1, -(-width // 4))
                table = rng.permutation(pages * 3)[:pages].astype(np.int32)
                for k in range(1, L + 3):
                    sel = sorted(i for i in topk_row(row.tolist(), L, k, 0) if i >= 0)
                    exp_ids = sel + [-1] * (k - len(sel))
                    exp_out = [int(table[i // 4]) * 4 + i % 4 for i in sel] + [-1] * (k - len(sel))
                    out, valid, ids = oracle.topk_ordered(row[None, :], [L], k, table[None, :], 4, lib=lib)
                    if (out[0].tolist(), int(valid[0]), ids[0].tolist()) != (exp_out, len(sel), exp_ids):
                        return [f"ordered brute L{L} k{k} row={row.tolist()}: "
                                f"{out[0].tolist()} {int(valid[0])} {ids[0].tolist()}"]
    return []


def _real_rank(bits: int):
    v = bf16_value(bits)
    return (v, 0 if (v == 0.0 and math.copysign(1.0, v) < 0) else 1)


def check_tops_order(lib) -> list[str]:
    """Every non-NaN pattern alone in a row: its top ranks as its value does,
    distinct values get distinct tops, and every top is nonzero; NaN gets 0."""
    pats = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    logits = np.zeros((1 << 16, 8), np.uint16)
    logits[:, 0] = pats
    t = oracle.tops(logits, np.ones(1 << 16, np.int32), lib=lib)[:, 0].astype(np.int64)
    bad = []
    real = [p for p in range(1 << 16) if not math.isnan(bf16_value(p))]
    real.sort(key=_real_rank)
    seq = [int(t[p]) for p in real]
    if any(b <= a for a, b in zip(seq, seq[1:])) or seq[0] == 0:
        bad.append("tops do not rank the values strictly")
    if any(int(t[p]) != 0 for p in range(1 << 16) if math.isnan(bf16_value(p))):
        bad.append("a NaN has a nonzero top")
    return bad


def check_tops_groups(lib, seed: int = 5) -> list[str]:
    """A group's top is the top of its largest eligible element (by real value)
    on its own; groups past the valid length, or of NaN only, are 0."""
    rng = workloads.rng_for(seed)
    rows, width = 40, 37
    logits = np.where(rng.random((rows, width)) < 0.1, np.uint16(0x7FC0),
                      workloads.normal_bf16(rng, (rows, width))).astype(np.uint16)
    lens = rng.integers(0, width + 1, size=rows).astype(np.int32)
    got = oracle.tops(logits, lens, lib=lib)
    alone = np.zeros((1, 8), np.uint16)
    for r in range(rows):
        for g in range(got.shape[1]):
            elems = [int(x) for x in logits[r, 8 * g: min(8 * g + 8, int(lens[r]))]
                     if not math.isnan(bf16_value(int(x)))]
            if not elems:
                exp = 0
            else:
                alone[0, 0] = max(elems, key=_real_rank)
                exp = int(oracle.tops(alone, [1], lib=lib)[0, 0])
            if int(got[r, g]) != exp:
                return [f"tops row {r} group {g}: {int(got[r, g])} != {exp}"]
    return []


def test_ordered_golden():
    assert check_ordered_golden(oracle.load()) == []


def test_ordered_bruteforce():
    assert check_ordered_bruteforce(oracle.load()) == []


def test_tops_rank_every_pattern():
    assert check_tops_order(oracle.load()) == []


def test_tops_are_group_maxima():
    assert check_tops_groups(oracle.load()) == []


@pytest.mark.parametrize("seed", [0, 1])
def test_ordered_invariants(seed):
    """Same set as the plain select; ascending ids; out = transform(ids);
    counts = selected entries; -1 exactly past the count."""
    case = workloads.paged_case(70 + seed, rows=23, width=3000, k=300, q=2, block_rows=2048)
    plain = oracle.topk(case.logits, case.valid_len, case.k, 0, case.block_table, case.page_size,
                        width=case.width, block_rows=case.block_rows, rows_per_request=2)
    out, valid, ids = oracle.topk_ordered(case.logits, case.valid_len, case.k, case.block_table,
                                          case.page_size, width=case.width,
                                          block_rows=case.block_rows, rows_per_request=2)
    for r in range(case.rows):
        n = int(valid[r])
        assert (out[r, n:] == -1).all() and (ids[r, n:] == -1).all()
        assert (np.diff(ids[r, :n]) > 0).all()
        assert sorted(out[r, :n].tolist()) == sorted(x for x in plain[r].tolist() if x >= 0)
        trow = case.block_table[r // 2]
        assert out[r, :n].tolist() == [int(trow[i // 64]) * 2048 + i % 64 for i in ids[r, :n].tolist()]


MUTANTS = [
    ("descending index order", [("return x < y ? -1 : (x > y ? 1 : 0);", "return x < y ? 1 : (x > y ? -1 : 0);")]),
    ("ids past the count not -1", [("j->ids[(int64_t)r * j->k + s] = s < sel ? sel_idx[s] : -1;",
                                    "j->ids[(int64_t)r * j->k + s] = s < sel ? sel_idx[s] : 0;")]),
    ("count one short", [("j->valid[r] = sel;", "j->valid[r] = sel - 1;")]),
    ("tops read past the valid length", [("for (int32_t t = 8 * g; t < 8 * g + 8 && t < L; ++t)",
                                          "for (int32_t t = 8 * g; t < 8 * g + 8 && t < width; ++t)")]),
    ("tops keep NaN", [("if (!is_nan_bf16(row[t]) && order_key(row[t]) > top)", "if (order_key(row[t]) > top)")]),
    ("tops take the minimum", [("order_key(row[t]) > top) top = order_key(row[t]);",
                                "(top == 0 || order_key(row[t]) < top)) top = order_key(row[t]);")]),
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
        caught = check_ordered_golden(lib) or check_ordered_bruteforce(lib, trials=1) \
            or check_tops_groups(lib)
        assert caught, f"planted mistake not caught: {name}"
    finally:
        shutil.rmtree(tmp, ignore_errors=True)
