"""Host-side figures of bench.py: the algorithmic bytes behind every roofline
fraction, checked against closed forms worked out by hand for each workload."""
import os
import sys

import numpy as np

import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_headline_bytes_closed_form():
    # 2048 full rows of 16384 logits, k 512, 64-logit pages (256 per row):
    # logits 2048*16384*2, valid lengths 2048*4, output 2048*512*4, and
    # min(512, 256) = 256 table entries of 4 bytes per row.
    c = W.config2(2048, 16384, 512)
    want = 2048 * 16384 * 2 + 2048 * 4 + 2048 * 512 * 4 + 2048 * 256 * 4
    assert want == 73_408_512
    assert bench.algorithmic_bytes(c) == want


def test_bytes_with_partial_rows_and_k2048():
    # valid 4096, k 2048: 64 pages per row hold the row, min(2048, 64) entries.
    c = W.config2(32, 4096, 2048)
    assert bench.algorithmic_bytes(c) == 32 * (4096 * 2 + 4 + 2048 * 4 + 64 * 4)
    # valid 9000: ceil(9000 / 64) = 141 pages.
    c = W.config2(128, 9000, 512)
    assert bench.algorithmic_bytes(c) == 128 * (9000 * 2 + 4 + 512 * 4 + 141 * 4)


def test_bypass_rows_read_no_logits():
    # Rows with at most k elements are answered from valid_len alone.
    c = W.config2(4, 16384, 512)
    c.valid_len = np.array([0, 100, 512, 513], dtype=np.int32)
    pages = [0, 2, 8, 9]  # ceil(L / 64), each below k
    want = 513 * 2 + 4 * 4 + 4 * 512 * 4 + 4 * sum(pages)
    assert bench.algorithmic_bytes(c) == want


def test_block_mode_bytes_count_every_logit():
    # Block rows read all their logits (the maximum of 8 needs them all);
    # no table here, so no page term.
    c = W.config4(0)
    L = np.clip(c.valid_len.astype(np.int64), 0, c.width)
    assert ((L + 7) // 8 > c.k).all()
    want = int(2 * L.sum()) + 4 * c.rows + 4 * c.rows * c.k
    assert bench.algorithmic_bytes(c) == want


def test_ordered_bytes_closed_form():
    # Ordered select: the per-8 maxima, at least k 16-byte vectors, valid
    # lengths, output, valid counts, and the page term; words add k / 32 words
    # of planes per row and read short rows whole.
    c = W.config2(2, 16384, 512)
    c.valid_len = np.array([16384, 300], dtype=np.int32)
    pages = min(512, 16384 // 64) + min(300, 512, -(-300 // 64))
    base = 4 * 2 + 4 * 2 * 512 + 4 * 2
    want = (2 * 2048 + 16 * 512) + base + 4 * pages
    assert bench.ordered_bytes(c) == want
    c.block_table = None
    want_words = (2 * 2048 + 16 * 512) + 2 * 300 + 4 * 2 + 4 * 2 * (512 + 16) + 4 * 2
    assert bench.ordered_bytes(c, words=True) == want_words
