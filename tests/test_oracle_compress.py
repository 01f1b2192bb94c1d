"""Pins for the oracle's token-level cache compression (the DeepSeek page's "KV cache
compression" section: blocks of m consecutive tokens merge into one row, a component-wise
weighted sum with weights from a softmax over the block's tokens of each component of
z = W^Z x), checked against closed forms, limits and a pure-Python twin.  CPU only."""
import math

import numpy as np
import pytest

import oracle
from oracle import twin


def _rng(seed):
    return np.random.default_rng(seed)


def _bf16_like(x):
    a = np.asarray(x, dtype=np.float32)
    u = a.view(np.uint32).astype(np.uint64)
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16) << 16
    return r.astype(np.uint32).view(np.float32)


def test_equal_weights_give_the_block_mean():
    rows = _rng(0).standard_normal((12, 7))
    for z in (np.zeros((12, 7)), np.full((12, 7), 3.5), np.repeat(_rng(1).standard_normal((3, 7)), 4, axis=0)):
        np.testing.assert_allclose(oracle.compress(rows, z, 4), rows.reshape(3, 4, 7).mean(axis=1), rtol=1e-13,
                                   atol=1e-14)


def test_a_dominant_token_is_copied_per_component():
    """Component k takes the row of the token whose z[k] dominates, a different token for each
    component (a softmax over components instead of tokens would not)."""
    rows = _rng(2).standard_normal((4, 8))
    z = np.zeros((4, 8))
    winner = np.array([0, 1, 2, 3, 3, 2, 1, 0])
    z[winner, np.arange(8)] = 80.0
    np.testing.assert_allclose(oracle.compress(rows, z, 4)[0], rows[winner, np.arange(8)], rtol=1e-12, atol=1e-12)


def test_merging_identical_rows_returns_the_row():
    row = _rng(3).standard_normal(9)
    rows = np.tile(row, (5, 1))
    z = _rng(4).standard_normal((5, 9)) * 10
    np.testing.assert_allclose(oracle.compress(rows, z, 5)[0], row, rtol=1e-13, atol=1e-13)


def test_one_token_blocks_change_nothing():
    rows = _rng(5).standard_normal((6, 4))
    z = _rng(6).standard_normal((6, 4)) * 5
    np.testing.assert_array_equal(oracle.compress(rows, z, 1), rows)


def test_shift_of_z_per_component_changes_nothing():
    rows = _rng(7).standard_normal((8, 6))
    z = _rng(8).standard_normal((8, 6))
    shift = _rng(9).standard_normal(6) * 100
    np.testing.assert_allclose(oracle.compress(rows, z + shift, 4), oracle.compress(rows, z, 4), rtol=1e-12,
                               atol=1e-12)


def test_matches_twin():
    rng = _rng(10)
    rows = rng.standard_normal((16, 5))
    z = rng.standard_normal((16, 5)) * 3
    got = oracle.compress(rows, z, 4)
    for g in range(4):
        np.testing.assert_allclose(got[g], twin.compress_block(rows[4 * g:4 * g + 4].tolist(),
                                                               z[4 * g:4 * g + 4].tolist()), rtol=1e-12, atol=1e-13)


def _inputs(seed, B, nb, m, d_model, d_c=8, d_r=4):
    rng = _rng(seed)
    h = _bf16_like(rng.standard_normal((B * nb * m, d_model)))
    w_dkv = _bf16_like(rng.standard_normal((d_c, d_model)) / 4)
    w_kr = _bf16_like(rng.standard_normal((d_r, d_model)) / 4)
    w_z = _bf16_like(rng.standard_normal((d_c + d_r, d_model)) / 4)
    return h, w_dkv, w_kr, w_z


def test_compressed_write_with_m1_is_the_plain_cache_write():
    h, w_dkv, w_kr, w_z = _inputs(11, 2, 3, 1, 16)
    bt = np.array([[3, 0], [1, 2]], dtype=np.int32)
    sl = np.array([5, 7], dtype=np.int32)
    rows, slot = oracle.cache_append_compressed(h, w_dkv, w_kr, w_z, bt, sl, 3, 1, num_pages=4, page=4)
    ref, ref_slot = oracle.cache_append(h, w_dkv, w_kr, bt, sl, 3, num_pages=4, page=4)
    np.testing.assert_array_equal(slot, ref_slot)
    np.testing.assert_allclose(rows, ref, rtol=1e-13, atol=1e-13)


def test_compressed_write_rotates_each_token_at_its_own_position():
    """With W^Z = 0 a block is the mean of its tokens' rows, each rotated at its own position
    P*m + i; the merged row goes to compressed position P."""
    h, w_dkv, w_kr, w_z = _inputs(12, 1, 2, 4, 16)
    w_z[:] = 0
    bt = np.array([[2, 1]], dtype=np.int32)
    sl = np.array([6], dtype=np.int32)          # compressed positions 4 and 5: tokens 16-19 and 20-23
    rows, slot = oracle.cache_append_compressed(h, w_dkv, w_kr, w_z, bt, sl, 2, 4, num_pages=3, page=4)
    assert slot.tolist() == [1 * 4 + 0, 1 * 4 + 1]
    for j, P in enumerate((4, 5)):
        toks = []
        for i in range(4):
            x = h[(j * 4 + i)].astype(np.float64)
            c = w_dkv.astype(np.float64) @ x
            kr = oracle.rope(w_kr.astype(np.float64) @ x, P * 4 + i)
            toks.append(np.concatenate([c, kr]))
        np.testing.assert_allclose(rows[j], np.mean(toks, axis=0), rtol=1e-12, atol=1e-12)


def test_compressed_write_matches_twin():
    B, nb, m, d_model, d_c, d_r = 2, 2, 4, 12, 6, 4
    h, w_dkv, w_kr, w_z = _inputs(13, B, nb, m, d_model, d_c, d_r)
    bt = np.array([[0, 1], [2, 3]], dtype=np.int32)
    sl = np.array([3, 8], dtype=np.int32)
    rows, slot = oracle.cache_append_compressed(h, w_dkv, w_kr, w_z, bt, sl, nb, m, num_pages=4, page=4,
                                                rope_base=50.0)
    H = h.astype(np.float64).tolist()
    for b in range(B):
        for j in range(nb):
            P = int(sl[b]) - nb + j
            toks, zs = [], []
            for i in range(m):
                x = H[(b * nb + j) * m + i]
                c = [math.fsum(wr * xv for wr, xv in zip(row, x)) for row in w_dkv.astype(np.float64).tolist()]
                kr = [math.fsum(wr * xv for wr, xv in zip(row, x)) for row in w_kr.astype(np.float64).tolist()]
                toks.append(c + twin.rope_phasor(kr, P * m + i, 50.0))
                zs.append([math.fsum(wr * xv for wr, xv in zip(row, x)) for row in w_z.astype(np.float64).tolist()])
            np.testing.assert_allclose(rows[b * nb + j], twin.compress_block(toks, zs), rtol=1e-11, atol=1e-12)
            assert slot[b * nb + j] == bt[b, P // 4] * 4 + P % 4


def test_pins_catch_planted_mistakes():
    """Slips planted in a copy of the merge, on the CPU: a softmax taken over the components
    instead of the tokens, and weights from the rows instead of z, each fail a pin above."""
    rows = _rng(2).standard_normal((4, 8))
    z = np.zeros((4, 8))
    winner = np.array([0, 1, 2, 3, 3, 2, 1, 0])
    z[winner, np.arange(8)] = 80.0

    def over_components(rows, z):
        w = np.exp(z - z.max(axis=1, keepdims=True))
        w /= w.sum(axis=1, keepdims=True)
        return (w * rows).sum(axis=0)

    def weights_from_rows(rows, z):
        w = np.exp(rows - rows.max(axis=0))
        return (w * rows).sum(axis=0) / w.sum(axis=0)
    want = rows[winner, np.arange(8)]
    assert not np.allclose(over_components(rows, z), want, atol=1e-3)
    assert not np.allclose(weights_from_rows(rows, z), want, atol=1e-3)
