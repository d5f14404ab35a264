"""Brute-force top-k on tiny rows, written from the definition with Python floats.

It never forms the 16-bit order key: values are ordered as real numbers, with
-0 below +0 and NaN removed, and ties are broken by the lower index. It pins the
oracle (which sorts packed key words in C) from an independent direction.
Definition: vLLM "decode_topk_cute" module docstring ("What this module
computes"); sglang PR #39305 Modifications (-0 below +0; NaN never selected);
vLLM kimi_k3 "dsa/indexer" (lowest-index ties; IndexerSelect.emit transform).
"""
from __future__ import annotations

import math
import struct


def bf16_value(bits: int) -> float:
    return struct.unpack("<f", struct.pack("<I", (int(bits) & 0xFFFF) << 16))[0]


def _rank(v: float):
    """Sort key for 'larger first': the value, then +0 above -0."""
    return (v, 0 if (v == 0.0 and math.copysign(1.0, v) < 0) else 1)


def topk_row(bits, valid_len: int, k: int, mode: int, table_row=None, page: int = 64):
    width = len(bits)
    L = max(0, min(int(valid_len), width))
    n = L if mode == 0 else (L + 7) // 8

    def phys(i):
        return i if table_row is None else int(table_row[i // page]) * page + i % page

    if n <= k:
        return [phys(i) for i in range(n)] + [-1] * (k - n)

    cands = []          # (value, index)
    for i in range(n):
        if mode == 0:
            v = bf16_value(bits[i])
            if math.isnan(v):
                continue
        else:
            group = [bf16_value(b) for b in bits[8 * i: min(8 * i + 8, L)]]
            if i == n - 1:
                v = math.inf                               # newest block pinned
            elif any(math.isnan(g) for g in group):
                continue
            else:
                v = max(group, key=_rank)
        cands.append((v, i))
    cands.sort(key=lambda c: (tuple(-x for x in _rank(c[0])), c[1]))
    chosen = cands[:k]
    out = []
    for v, i in chosen:
        out.append(-1 if (mode == 1 and v == -math.inf) else phys(i))
    return out + [-1] * (k - len(out))
