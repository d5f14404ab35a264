"""Pins for the oracle's local top-n words (IndexerLocalTopk on the vLLM kimi_k3
"dsa/indexer" page), no GPU: hand-derived cases (tests/golden/words_cases.json),
the float brute force's selection arranged as the page orders it (above the
threshold, then the ties, each in index order), word keys checked against the
pinned per-8 maxima of single elements, and planted mistakes."""
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


def _rank(bits: int):
    v = bf16_value(bits)
    return (v, 0 if (v == 0.0 and math.copysign(1.0, v) < 0) else 1)


def decode(words: np.ndarray, n: int):
    """(key, index) of each nonzero word of one row."""
    w = words.view(np.uint32).astype(np.int64)
    out = []
    for j in range(n):
        if w[j] == 0:
            out.append(None)
            continue
        hi = (w[n + j // 32] >> (j % 32)) & 1
        out.append((int(w[j] >> 16), int(0xFFFF - (w[j] & 0xFFFF)) | (int(hi) << 16)))
    return out


def check_words_golden(lib) -> list[str]:
    with open(os.path.join(HERE, "golden", "words_cases.json")) as fh:
        cases = json.load(fh)["cases"]
    bad = []
    for c in cases:
        row = np.full(c["width"], int(c["fill"], 16), np.uint16)
        for pos, h in c["set"].items():
            row[int(pos)] = int(h, 16)
        n = c["n"]
        out, valid = oracle.topk_words(row[None, :], [c["valid_len"]], n, lib=lib)
        exp = np.zeros(n + n // 32, np.uint32)
        for j, h in c["expected_words"].items():
            exp[int(j)] = int(h, 16)
        if not np.array_equal(out[0].view(np.uint32), exp) or int(valid[0]) != c["expected_valid"]:
            bad.append(f"words golden {c['name']}")
    return bad


def check_words_bruteforce(lib, seed: int = 11) -> list[str]:
    rng = workloads.rng_for(seed)
    specials = np.array([0x0000, 0x8000, 0x7F80, 0xFF80, 0x7FC0, 0x3F80, 0xBF80], np.uint16)
    one = np.zeros((1, 8), np.uint16)
    for width in (5, 31, 32, 33, 70, 200):
        for row in (workloads.normal_bf16(rng, (width,)), specials[rng.integers(0, len(specials), width)],
                    rng.integers(0, 1 << 16, size=width).astype(np.uint16)):
            L = int(rng.integers(0, width + 1))
            for n in (32, 64):
                out, valid = oracle.topk_words(row[None, :], [L], n, lib=lib)
                got = decode(out[0], n)
                if L <= n:
                    order = list(range(L))
                else:
                    sel = [i for i in topk_row(row.tolist(), L, n, 0) if i >= 0]
                    if len(sel) < n:
                        order = sorted(sel)
                    else:
                        t = min((_rank(int(row[i])) for i in sel))
                        order = sorted(i for i in sel if _rank(int(row[i])) > t) + \
                            sorted(i for i in sel if _rank(int(row[i])) == t)
                exp = []
                for i in order:
                    one[0, 0] = row[i]
                    key = int(oracle.tops(one, [1], lib=lib)[0, 0]) if not math.isnan(bf16_value(int(row[i]))) \
                        else None
                    exp.append((key, i))
                got_real = [g for g in got if g is not None]
                if int(valid[0]) != len(order) or [g[1] for g in got_real] != order or \
                        any(e[0] is not None and g[0] != e[0] for g, e in zip(got_real, exp)) or \
                        any(g is not None for g in got[len(order):]):
                    return [f"words brute L{L} n{n} row={row.tolist()}: {got_real[:6]} vs {exp[:6]}"]
    return []


def test_words_golden():
    assert check_words_golden(oracle.load()) == []


def test_words_bruteforce():
    assert check_words_bruteforce(oracle.load()) == []


MUTANTS = [
    ("ties before the keys above", [("if ((pass == 0) == (sel < n || key > T))", "if ((pass == 1) == (sel < n || key > T))")]),
    ("index not inverted", [("(0xFFFFu - ((uint32_t)l & 0xFFFFu))", "((uint32_t)l & 0xFFFFu)")]),
    ("plane bit dropped", [("if ((l >> 16) & 1) orow[n + j / 32]", "if (0) orow[n + j / 32]")]),
    ("short rows only below n", [("if (L <= n) { /* every element, in index order */", "if (L < n) { /* every element, in index order */")]),
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
        assert check_words_golden(lib) or check_words_bruteforce(lib), f"planted mistake not caught: {name}"
    finally:
        shutil.rmtree(tmp, ignore_errors=True)
