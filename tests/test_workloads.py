"""The seeded input generators: shapes, determinism and the stated structure."""
import numpy as np

import workloads as W


def test_config1_shape_and_seed():
    a, b = W.config1(0), W.config1(0)
    assert a.logits.shape == (4, 4096) and a.k == 512 and a.mode == W.TOKEN
    assert np.array_equal(a.logits, b.logits)
    assert np.array_equal(a.block_table, np.tile(np.arange(64), (4, 1)))


def test_config2_permuted_pages():
    c = W.config2(rows=32, valid=9000, k=512)
    assert c.logits.shape == (32, 16384) and (c.valid_len == 9000).all()
    flat = np.sort(c.block_table.reshape(-1))
    assert np.array_equal(flat, np.arange(32 * 256))


def test_config3_crowded_values():
    c = W.config3(rows=8, width=20000)
    assert len(np.unique(c.logits)) <= 200
    assert ((c.valid_len >= 13333) & (c.valid_len <= 20000)).all()
    assert len(np.unique(W.config3(rows=1).logits)) > 50


def test_config4_block_structure():
    c = W.config4(rows=2, width=1 << 16)
    blocks = c.logits.reshape(2, -1, 8)
    all_ninf = (blocks == W.BF16_NEG_INF).all(axis=2).mean()
    assert 0.03 < all_ninf < 0.07
    nan = ((c.logits & 0x7FFF) > 0x7F80).mean()
    assert 0.0003 < nan < 0.003
    assert (c.valid_len >= 1 << 15).all() and (c.valid_len <= 1 << 16).all()


def test_edge_cases_build():
    cases = W.edge_cases()
    assert [c.mode for c in cases] == [W.TOKEN, W.BLOCK8]
    for c in cases:
        assert c.logits.shape[0] == len(c.valid_len) == c.block_table.shape[0]
