"""Seeded synthetic inputs for exact BF16 top-k.

Shared by the tests, the benchmark and the smoke check; it feeds the CUDA path
and the CPU oracle the same bits. It holds none of the selection's arithmetic:
only value distributions, valid lengths and block tables.

Every generator is deterministic in its seed (numpy PCG64). N(0,1) draws are
made in float32 and rounded to BF16 (round to nearest even) by torch.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

TOKEN = 0
BLOCK8 = 1
PAGE = 64

BF16_POS_INF = 0x7F80
BF16_NEG_INF = 0xFF80
BF16_ONE = 0x3F80
BF16_POS_ZERO = 0x0000
BF16_NEG_ZERO = 0x8000
NAN_PATTERNS = (0x7FC0, 0xFFC0, 0x7F81, 0xFF81, 0x7FFF, 0xFFFF)


@dataclass
class Case:
    """One launch's worth of input: logits [rows, row_stride] as BF16 bits."""
    name: str
    logits: np.ndarray            # uint16 [rows, row_stride]
    width: int
    valid_len: np.ndarray         # int32 [rows]
    k: int
    mode: int = TOKEN
    block_table: np.ndarray | None = None   # int32 [ceil(rows / rows_per_request), pages] or None
    page_size: int = PAGE
    notes: dict = field(default_factory=dict)
    block_rows: int | None = None           # physical rows per page (None: page_size)
    rows_per_request: int = 1               # rows sharing one table row

    @property
    def rows(self) -> int:
        return int(self.logits.shape[0])

    def logit_bytes(self) -> int:
        """Bytes of logits a launch must read: every valid logit of rows with n > k."""
        L = np.clip(self.valid_len.astype(np.int64), 0, self.width)
        n = L if self.mode == TOKEN else (L + 7) // 8
        return int(2 * L[n > self.k].sum())


def rng_for(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> BF16 bits (round to nearest even), as uint16."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def normal_bf16(rng: np.random.Generator, shape) -> np.ndarray:
    return to_bf16_bits(rng.standard_normal(size=shape, dtype=np.float32))


def identity_table(rows: int, width: int, page: int = PAGE) -> np.ndarray:
    pages = -(-width // page)
    return np.tile(np.arange(pages, dtype=np.int32), (rows, 1))


def permuted_table(rng: np.random.Generator, rows: int, width: int, page: int = PAGE) -> np.ndarray:
    """Each row's pages map to distinct physical pages: a seeded permutation of
    [0, rows * pages) laid out row-major."""
    pages = -(-width // page)
    return rng.permutation(rows * pages).astype(np.int32).reshape(rows, pages)


# ---------------------------------------------------------------- the configs

def config1(seed: int = 0) -> Case:
    """Token mode, 4 rows x 4096 N(0,1) logits (all valid), k=512, identity table."""
    rng = rng_for(seed)
    logits = normal_bf16(rng, (4, 4096))
    return Case("token 4x4096 k512 identity-table", logits, 4096,
                np.full(4, 4096, np.int32), 512, TOKEN, identity_table(4, 4096))


def config2(rows: int, valid: int, k: int = 512, seed: int = 0, width: int = 16384) -> Case:
    """Consumer top-k: rows x 16384 N(0,1) logits, every row `valid` long, and a
    per-row table of randomly permuted 64-token pages."""
    rng = rng_for(seed)
    logits = normal_bf16(rng, (rows, width))
    table = permuted_table(rng, rows, width)
    return Case(f"consumer {rows}x{width} valid{valid} k{k}", logits, width,
                np.full(rows, valid, np.int32), k, TOKEN, table)


CONFIG2_ROWS = (1, 32, 128, 512, 2048)
CONFIG2_VALID = (16384, 9000, 4096)
CONFIG2_K = (512, 2048)


def _zipf_values(rng: np.random.Generator, count: int = 200) -> np.ndarray:
    """`count` distinct finite BF16 values (N(0,1) draws, deduplicated), sorted ascending."""
    vals = np.unique(normal_bf16(rng, (4 * count,)).astype(np.int32))
    vals = vals[(vals & 0x7FFF) != 0]                      # no zeros: keep them distinct
    f = torch.from_numpy(vals.astype(np.uint16).view(np.int16)).view(torch.bfloat16).float().numpy()
    order = np.argsort(f, kind="stable")
    vals = vals[order]
    pick = np.sort(rng.choice(len(vals), size=count, replace=False))
    return vals[pick].astype(np.uint16)


def config3(seed: int = 0, rows: int = 64, width: int = 150000, k: int = 512) -> Case:
    """Crowded bins: 200 distinct values, Zipf(1)-weighted.

    Rows 0-31: random rank -> value map. Rows 32-47: the heaviest ranks on the
    largest values (the k-th largest sits inside a bin of tens of thousands of
    ties). Rows 48-55: the largest values only at element positions 1..7 mod 8
    (position 0 mod 8 holds the smallest value). Rows 56-63: ascending rows (the
    largest values all at the end). Valid lengths uniform in [2/3 width, width]
    ([100000, 150000] at the default width).
    """
    rng = rng_for(seed)
    vals = _zipf_values(rng)                       # ascending by value
    nv = len(vals)
    w = 1.0 / np.arange(1, nv + 1)
    w /= w.sum()
    logits = np.empty((rows, width), np.uint16)
    for r in range(rows):
        ranks = rng.choice(nv, size=width, p=w)     # rank 0 = heaviest
        if r < 32 or r >= 48:
            perm = rng.permutation(nv)               # rank -> value index
        else:
            perm = np.arange(nv)[::-1]               # heaviest rank -> largest value
        idx = perm[ranks]
        if 48 <= r < 56:
            lane0 = (np.arange(width) % 8) == 0
            idx[lane0] = 0
        elif r >= 56:
            idx = np.sort(idx)
        logits[r] = vals[idx]
    valid = rng.integers((2 * width) // 3, width + 1, size=rows).astype(np.int32)
    return Case(f"crowded {rows}x{width} k{k}", logits, width, valid, k, TOKEN)


def config4(seed: int = 0, rows: int = 32, width: int = 1 << 20, k: int = 2048) -> Case:
    """Block mode: N(0,1), 5% of aligned 8-logit blocks all -inf, 0.1% NaN logits
    (random sign and payload), valid lengths uniform in [width/2, width], k=2048."""
    rng = rng_for(seed)
    logits = normal_bf16(rng, (rows, width))
    blocks = logits.reshape(rows, width // 8, 8)
    ninf = rng.random((rows, width // 8)) < 0.05
    blocks[ninf] = BF16_NEG_INF
    nan = rng.random((rows, width)) < 0.001
    logits[nan] = np.asarray(NAN_PATTERNS, np.uint16)[rng.integers(0, len(NAN_PATTERNS), int(nan.sum()))]
    valid = rng.integers(width // 2, width + 1, size=rows).astype(np.int32)
    return Case(f"block {rows}x{width} k{k}", logits, width, valid, k, BLOCK8)


def config5a(seed: int = 0, rows: int = 256, width: int = 524288, k: int = 512) -> Case:
    """Wide token rows: 256 x 524288 N(0,1), all valid, k=512."""
    rng = rng_for(seed)
    return Case(f"wide {rows}x{width} k{k}", normal_bf16(rng, (rows, width)), width,
                np.full(rows, width, np.int32), k, TOKEN)


def config5b(seed: int = 0, rows: int = 64, width: int = 1 << 20, k: int = 512) -> Case:
    """Wide token rows: 64 x 1048576 N(0,1), all valid, k=512."""
    return config5a(seed, rows, width, k)


# ------------------------------------------------------------------ edge rows

def _edge_token_rows(rng: np.random.Generator, width: int, k: int):
    rows, lens = [], []

    def add(row, L=width):
        rows.append(np.asarray(row, np.uint16))
        lens.append(L)

    for L in (0, 1, 7, 8, 9, 511, 512, 513, 8999, 9001, width - 1):
        add(normal_bf16(rng, (width,)), L)
    add(np.full(width, BF16_ONE))                        # constant rows
    add(np.full(width, BF16_POS_ZERO))
    add(np.full(width, BF16_NEG_INF))                    # all -inf
    add(np.full(width, BF16_POS_INF))                    # all +inf
    r = np.where(rng.random(width) < 0.5, BF16_POS_ZERO, BF16_NEG_ZERO).astype(np.uint16)
    pos = rng.choice(width, size=k // 2, replace=False)
    r[pos] = to_bf16_bits(np.abs(rng.standard_normal(k // 2, dtype=np.float32)) + 0.5)
    add(r)                                               # +/-0 pivot: fewer than k positives
    r = np.where(rng.random(width) < 0.5, BF16_POS_ZERO, BF16_NEG_ZERO).astype(np.uint16)
    r[rng.choice(width, size=k - 3, replace=False)] = BF16_ONE
    add(r)                                               # k-3 ones, then the zeros decide
    den = rng.integers(1, 0x80, size=width).astype(np.uint16)
    add(den | np.where(rng.random(width) < 0.5, 0, 0x8000).astype(np.uint16))   # denormals only
    r = den.copy()
    r[rng.choice(width, size=k - 40, replace=False)] = BF16_ONE
    add(r)                                               # denormals at the pivot
    add(rng.integers(0, 1 << 16, size=width).astype(np.uint16))                  # full range
    for count in (1, k - 1, k, 600):                     # +NaN counts
        r = normal_bf16(rng, (width,))
        r[rng.choice(width, size=count, replace=False)] = 0x7FC0
        add(r)
    r = normal_bf16(rng, (width,))
    r[rng.choice(width, size=2000, replace=False)] = 0xFFC0
    add(r)                                               # -NaN
    r = np.full(width, 0x7FC0, np.uint16)
    r[rng.choice(width, size=k // 2, replace=False)] = normal_bf16(rng, (k // 2,))
    add(r)                                               # mostly +NaN: fewer than k non-NaN
    r = np.full(width, 0xFFC1, np.uint16)
    r[rng.choice(width, size=k + 10, replace=False)] = normal_bf16(rng, (k + 10,))
    add(r)                                               # mostly -NaN: just above k non-NaN
    four = to_bf16_bits(np.array([-1.5, 0.25, 1.0, 2.0], np.float32))
    add(four[rng.integers(0, 4, size=width)])            # 4-value heavy ties
    add(np.arange(width, dtype=np.uint16) % 0x7F00)      # ascending, then wraps
    return rows, lens


def _edge_block_rows(rng: np.random.Generator, width: int, k: int):
    rows, lens = [], []

    def add(row, L=width):
        rows.append(np.asarray(row, np.uint16))
        lens.append(L)

    add(np.full(width, BF16_NEG_INF))                    # all -inf: only the newest block
    r = normal_bf16(rng, (width,))
    r[width - 3] = 0x7FC0
    add(r)                                               # NaN in the newest block
    r = np.where(rng.random(width) < 0.5, BF16_POS_ZERO, BF16_NEG_ZERO).astype(np.uint16)
    add(r)                                               # +/-0 blocks
    for L in (8 * k - 5, 8 * k, 8 * k + 1, 8 * k + 9, width - 3):
        add(normal_bf16(rng, (width,)), L)               # around n == k, partial newest block
    r = normal_bf16(rng, (width,))
    b = r.reshape(-1, 8)
    b[rng.random(b.shape[0]) < 0.97] = BF16_NEG_INF
    add(r)                                               # fewer than k blocks above -inf
    r = normal_bf16(rng, (width,))
    r[rng.random(width) < 0.05] = 0x7FC0
    add(r)                                               # many NaN blocks
    add(rng.integers(0, 1 << 16, size=width).astype(np.uint16))                  # full range
    add(np.full(width, BF16_ONE))                        # constant
    return rows, lens


def resident_cut_rows(seed: int = 0, width: int = 1 << 20, k: int = 2048) -> Case:
    """Block rows for the resident-keys selection's branches (every row full).

    Row 0: N(0,1). Row 1: N(0,1) with one aligned run of 2048 blocks near 200
    (far above the rest: the k-th largest block sits far above the k-th largest
    per-thread maximum). Row 2: the first 16384 blocks N(3, 0.25), the rest
    N(0,1) (thousands of blocks of one CTA's share at or above the cut). Row 3:
    N(0,1) sorted ascending. Row 4: constant 1.0 (ties everywhere).
    """
    rng = rng_for(seed)
    nb = width // 8
    logits = normal_bf16(rng, (5, width))
    run = 2048 * int(rng.integers(0, nb // 2048))
    logits[1, 8 * run:8 * (run + 2048)] = to_bf16_bits(200.0 + rng.standard_normal(8 * 2048, dtype=np.float32))
    logits[2, :8 * 16384] = to_bf16_bits(3.0 + 0.25 * rng.standard_normal(8 * 16384, dtype=np.float32))
    logits[3] = to_bf16_bits(np.sort(rng.standard_normal(width, dtype=np.float32)))
    logits[4] = BF16_ONE
    valid = np.full(5, width, np.int32)
    return Case(f"resident-cut rows 5x{width} k{k}", logits, width, valid, k, BLOCK8)


def ordered_wide(seed: int = 0, rows: int = 64, width: int = 1 << 20, k: int = 2048) -> Case:
    """Long token rows for the ordered select bounded by per-8 maxima (the
    indexer's decode step: top-2048 of up to 1M keys per row): N(0,1) scores,
    valid lengths uniform in [width/2, width], a seeded-permuted table of 64-token
    pages."""
    rng = rng_for(seed)
    logits = normal_bf16(rng, (rows, width))
    valid = rng.integers(width // 2, width + 1, size=rows).astype(np.int32)
    table = permuted_table(rng, rows, width)
    return Case(f"ordered {rows}x{width} k{k}", logits, width, valid, k, TOKEN, table)


def local_rows(seed: int = 0, rows: int = 128, width: int = 16384, n: int = 2048) -> Case:
    """One GPU's part of a context split over several (DCP): rows of up to 16384
    keys (a 128K context over 8 GPUs) whose local top-n (n 2048) goes out as
    B' words; N(0,1), valid lengths uniform in [width/2, width], no table."""
    rng = rng_for(seed)
    logits = normal_bf16(rng, (rows, width))
    valid = rng.integers(width // 2, width + 1, size=rows).astype(np.int32)
    return Case(f"local {rows}x{width} n{n}", logits, width, valid, n, TOKEN)


def edge_cases(seed: int = 0, width: int = 16384, k: int = 512) -> list[Case]:
    """Edge rows in token and block mode (one Case per mode)."""
    rng = rng_for(seed)
    out = []
    for mode, maker, name in ((TOKEN, _edge_token_rows, "edge token"),
                              (BLOCK8, _edge_block_rows, "edge block")):
        kk = k if mode == TOKEN else max(1, k // 4)
        rows, lens = maker(rng, width, kk)
        logits = np.stack(rows)
        table = permuted_table(rng, len(rows), width if mode == TOKEN else -(-width // 8))
        out.append(Case(f"{name} {len(rows)}x{width} k{kk}", logits, width,
                        np.asarray(lens, np.int32), kk, mode, table))
    return out


def ragged_case(seed: int, rows: int, width: int, row_stride: int, k: int, mode: int = TOKEN,
                min_valid: int = 0, with_table: bool = False) -> Case:
    """Random rows with ragged valid lengths in [min_valid, width], N(0,1) values."""
    rng = rng_for(seed)
    logits = normal_bf16(rng, (rows, row_stride))
    valid = rng.integers(min_valid, width + 1, size=rows).astype(np.int32)
    table = None
    if with_table:
        n_width = width if mode == TOKEN else -(-width // 8)
        table = permuted_table(rng, rows, n_width)
    return Case(f"ragged {rows}x{width}/{row_stride} k{k} mode{mode}", logits, width, valid, k,
                mode, table)


def shifting_rows(seed: int, rows: int = 3000, width: int = 8192, k: int = 512,
                  mode: int = TOKEN, run: int = 700) -> Case:
    """Runs of `run` rows that share a value distribution, the distribution
    changing from run to run: N(0,1); 4 N(0,1) - 20 (every value negative);
    N(0,1) / 4; N(0,1) with every 13th row a short one (valid length k / 2 in
    token mode, 4k logits in block mode); then around again. A CTA that walks
    rows in a fixed stride meets long runs of alike rows and the changes
    between them."""
    rng = rng_for(seed)
    x = rng.standard_normal(size=(rows, width), dtype=np.float32)
    kind = (np.arange(rows) // run) % 4
    x[kind == 1] = 4.0 * x[kind == 1] - 20.0
    x[kind == 2] *= 0.25
    valid = np.full(rows, width, np.int32)
    short = (kind == 3) & (np.arange(rows) % 13 == 0)
    valid[short] = k // 2 if mode == TOKEN else 4 * k
    n_width = width if mode == TOKEN else -(-width // 8)
    return Case(f"shifting {rows}x{width} k{k} mode{mode}", to_bf16_bits(x), width, valid, k,
                mode, permuted_table(rng, rows, n_width))


def paged_case(seed: int, rows: int, width: int, k: int, mode: int = TOKEN, q: int = 2,
               block_rows: int = 2048, page: int = PAGE) -> Case:
    """N(0,1) rows with ragged valid lengths, in requests of q rows that share a
    table row of seeded-permuted page ids, block_rows physical rows per page."""
    rng = rng_for(seed)
    stride = -(-width // 8) * 8
    logits = normal_bf16(rng, (rows, stride))
    valid = rng.integers(0, width + 1, size=rows).astype(np.int32)
    n_width = width if mode == TOKEN else -(-width // 8)
    table = permuted_table(rng, -(-rows // q), n_width, page)
    return Case(f"paged {rows}x{width} k{k} mode{mode} q{q} block_rows{block_rows}", logits, width,
                valid, k, mode, table, page, block_rows=block_rows, rows_per_request=q)


def fallback_rows(seed: int = 0, rows: int = 8, width: int = 16384, k: int = 512) -> Case:
    """Token rows built so that a sample-style cut cannot serve them and the
    exact fallbacks must run (the DecodeTopK page's direct path: the sample
    misjudges the row). Even rows: N(0,1) where seven of every eight 16-byte
    vectors are all NaN, so most groups of logits hold no usable representative
    (fewer than k of them) while more than k logits are eligible. Odd rows:
    every vector's eight logits equal (one N(0,1) draw per vector), so any cut
    taken from group maxima lets whole vectors through, several times k
    logits. Valid lengths = width; no table."""
    rng = rng_for(seed)
    vecs = -(-width // 8)
    out = np.empty((rows, vecs * 8), np.uint16)
    for r in range(rows):
        if r % 2 == 0:
            row = normal_bf16(rng, (vecs * 8,))
            nan_vec = rng.random(vecs) < 7.0 / 8.0
            row.reshape(vecs, 8)[nan_vec] = 0x7FC0
        else:
            row = np.repeat(normal_bf16(rng, (vecs,)), 8)
        out[r] = row
    return Case(f"fallback {rows}x{width} k{k}", out[:, :width].copy() if width % 8 else out, width,
                np.full(rows, width, np.int32), k, TOKEN, None)
