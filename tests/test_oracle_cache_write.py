"""Pins for the oracle's cache write (the step before the decode): the down-projection
c = W^DKV h of the "DeepSeek-V2" explainer's Step 5 (equation 9), the rotated position key
k^R = RoPE(W^KR h) of Step 7, and where each new token's row lands in the paged pool.
Checked against closed forms, the property Step 7 states (a rotated query-key score depends
only on the distance), hand-computed slot numbers and the pure-Python twin.  CPU only."""
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


# ---------------------------------------------------------------------------
# RoPE (Step 7)
# ---------------------------------------------------------------------------
def test_rope_position_zero_is_identity():
    x = _rng(0).standard_normal(64)
    assert np.array_equal(oracle.rope(x, 0.0), x)


def test_rope_keeps_every_pair_length():
    x = _rng(1).standard_normal(64)
    y = oracle.rope(x, 1234.0)
    np.testing.assert_allclose(np.hypot(y[0::2], y[1::2]), np.hypot(x[0::2], x[1::2]), rtol=1e-13)
    assert not np.allclose(y, x)


def test_rope_score_depends_only_on_distance():
    """Step 7: after rotation, a query-key score is a function of j - t alone."""
    rng = _rng(2)
    q, k = rng.standard_normal(64), rng.standard_normal(64)
    for t, j in [(0, 5), (17, 3), (100000, 131071)]:
        ref = oracle.rope(q, t) @ oracle.rope(k, j)
        for shift in (1, 64, 4099):
            got = oracle.rope(q, t + shift) @ oracle.rope(k, j + shift)
            assert got == pytest.approx(ref, rel=1e-9, abs=1e-9)
    # ... and it does depend on the distance
    assert abs(oracle.rope(q, 0) @ oracle.rope(k, 0) - oracle.rope(q, 0) @ oracle.rope(k, 7)) > 1e-3


def test_rope_rotations_compose():
    x = _rng(3).standard_normal(64)
    np.testing.assert_allclose(oracle.rope(oracle.rope(x, 300.0), 4000.0), oracle.rope(x, 4300.0),
                               rtol=1e-9, atol=1e-9)


@pytest.mark.parametrize("i", [0, 1, 5, 31])
def test_rope_pair_i_has_period_two_pi_over_theta_i(i):
    """Pair i turns at theta_i = base^(-2i/d): one period later it is back where it started,
    while a pair with another frequency is not."""
    x = _rng(4).standard_normal(64)
    period = 2.0 * math.pi * 10000.0 ** (2.0 * i / 64)
    y = oracle.rope(x, period)
    np.testing.assert_allclose(y[2 * i:2 * i + 2], x[2 * i:2 * i + 2], rtol=1e-9, atol=1e-9)
    j = 2 if i != 2 else 3
    assert not np.allclose(y[2 * j:2 * j + 2], x[2 * j:2 * j + 2], atol=1e-3)


def test_rope_turns_counter_clockwise():
    """Reading: a quarter turn of pair 0 takes (1, 0) to (0, 1)."""
    e0 = np.zeros(64)
    e0[0] = 1.0
    y = oracle.rope(e0, math.pi / 2)
    assert y[0] == pytest.approx(0.0, abs=1e-15) and y[1] == pytest.approx(1.0, abs=1e-15)


def test_rope_matches_phasor_twin():
    rng = _rng(5)
    for pos in (0.0, 1.0, 77.0, 8195.0, 131071.0):
        x = rng.standard_normal(64)
        np.testing.assert_allclose(oracle.rope(x, pos), twin.rope_phasor(list(x), pos, 10000.0),
                                   rtol=1e-9, atol=1e-9)


# ---------------------------------------------------------------------------
# Projection and slot (Step 5 equation 9, Step 7, the paged pool)
# ---------------------------------------------------------------------------
def _layout(lens, page, max_pages, num_pages, seed):
    rng = _rng(seed)
    perm = rng.permutation(num_pages)
    bt = -np.ones((len(lens), max_pages), dtype=np.int32)
    cur = 0
    for b, L in enumerate(lens):
        n = (L + page - 1) // page
        bt[b, :n] = perm[cur:cur + n]
        cur += n
    return bt


def test_basis_inputs_select_weight_columns():
    """h = e_k gives c = column k of W^DKV (a transposed W would give row k) and
    k^R = RoPE(column k of W^KR) at the token's position."""
    rng = _rng(6)
    d_model, d_c, d_r = 12, 6, 4
    w_dkv = _bf16_like(rng.standard_normal((d_c, d_model)))
    w_kr = _bf16_like(rng.standard_normal((d_r, d_model)))
    bt = np.array([[2, 0]], dtype=np.int32)
    for k in (0, 5, 11):
        h = np.zeros((1, d_model), dtype=np.float32)
        h[0, k] = 1.0
        rows, slot = oracle.cache_append(h, w_dkv, w_kr, bt, np.array([3]), 1, num_pages=3, page=4)
        np.testing.assert_array_equal(rows[0, :d_c], w_dkv[:, k].astype(np.float64))
        np.testing.assert_allclose(rows[0, d_c:], oracle.rope(w_kr[:, k], 2.0), rtol=1e-15, atol=1e-15)
        assert slot[0] == 2 * 4 + 2


def test_slots_computed_by_hand():
    """Page 4; sequence 0 has 5 tokens in pages [7, 2], sequence 1 has 3 in page [4];
    2 new tokens each: positions 3, 4 and 1, 2."""
    bt = np.array([[7, 2], [4, -1]], dtype=np.int32)
    h = np.ones((4, 3), dtype=np.float32)
    w = np.ones((2, 3), dtype=np.float32)
    _, slot = oracle.cache_append(h, w, w, bt, np.array([5, 3]), 2, num_pages=8, page=4)
    assert slot.tolist() == [7 * 4 + 3, 2 * 4 + 0, 4 * 4 + 1, 4 * 4 + 2]


def test_tokens_without_a_valid_slot_get_minus_one():
    bt = np.array([[1, 9], [0, -1], [2, 3]], dtype=np.int32)
    h = np.ones((3, 2), dtype=np.float32)
    w = np.ones((2, 2), dtype=np.float32)
    # seq 0: position 4 -> logical page 1 -> physical 9, beyond 4 pages; seq 1: length 0 -> position -1;
    # seq 2: position 8 -> logical page 2, beyond the table
    _, slot = oracle.cache_append(h, w, w, bt, np.array([5, 0, 9]), 1, num_pages=4, page=4)
    assert slot.tolist() == [-1, -1, -1]


@pytest.mark.parametrize("seed,Tq,lens", [(7, 1, (5, 9, 1)), (8, 3, (3, 8, 6)), (9, 4, (16, 4))])
def test_cache_write_matches_twin(seed, Tq, lens):
    rng = _rng(seed)
    d_model, d_c, d_r, page = 16, 8, 4, 4
    max_pages = max((L + page - 1) // page for L in lens)
    num_pages = sum((L + page - 1) // page for L in lens) + 2
    bt = _layout(lens, page, max_pages, num_pages, seed)
    h = _bf16_like(rng.standard_normal((len(lens), Tq, d_model)))
    w_dkv = _bf16_like(rng.standard_normal((d_c, d_model)) / 4)
    w_kr = _bf16_like(rng.standard_normal((d_r, d_model)) / 4)
    rows, slot = oracle.cache_append(h, w_dkv, w_kr, bt, np.array(lens), Tq, num_pages=num_pages, page=page,
                                     rope_base=100.0)
    ref = twin.cache_rows(h.astype(np.float64).tolist(), w_dkv.astype(np.float64).tolist(),
                          w_kr.astype(np.float64).tolist(), bt.tolist(), list(lens), Tq, page, num_pages, 100.0)
    got = {int(s): rows[n] for n, s in enumerate(slot) if s >= 0}
    assert sorted(got) == sorted(ref)
    for s, r in ref.items():
        np.testing.assert_allclose(got[s], r, rtol=1e-12, atol=1e-12)


def test_written_row_is_what_the_decode_reads():
    """A one-token context written by the cache write decodes to its own latent (o = c, and
    lse = scale * q . [c | k^R]): the write's position convention matches the decode's."""
    rng = _rng(10)
    d_model, d_c, d_r, page = 16, 8, 4, 4
    h = _bf16_like(rng.standard_normal((1, d_model)))
    w_dkv = _bf16_like(rng.standard_normal((d_c, d_model)))
    w_kr = _bf16_like(rng.standard_normal((d_r, d_model)))
    bt = np.array([[1]], dtype=np.int32)
    rows, slot = oracle.cache_append(h, w_dkv, w_kr, bt, np.array([1]), 1, num_pages=2, page=page)
    assert slot[0] == 4
    # position 0: k^R is W^KR h unrotated
    np.testing.assert_array_equal(rows[0, d_c:], (w_kr.astype(np.float64) @ h[0].astype(np.float64)))
    pool = np.zeros((2, page, d_c + d_r), dtype=np.float64)
    pool.reshape(-1, d_c + d_r)[slot[0]] = rows[0]
    q = rng.standard_normal((1, 1, 1, d_c + d_r))
    o, lse = oracle.decode_absorbed(q, pool.astype(np.float32), bt, np.array([1], dtype=np.int32), 0.5, d_c=d_c)
    np.testing.assert_allclose(o[0, 0, 0], pool.astype(np.float32).reshape(-1, d_c + d_r)[4, :d_c], rtol=1e-12)
    assert lse[0, 0, 0] == pytest.approx(0.5 * float(q[0, 0, 0] @ pool.astype(np.float32).reshape(-1, d_c + d_r)[4]),
                                         rel=1e-12)


def test_pins_catch_planted_rope_mistakes():
    """Plausible slips in the rotation, planted in a copy of the oracle's arithmetic on the CPU,
    each fail one of the pins above."""
    def rope_variant(x, pos, sign=1.0, expo=2.0, pair_stride=False):
        d = len(x)
        out = np.zeros(d)
        for i in range(d // 2):
            a = pos * 10000.0 ** (-expo * i / d)
            c, s = math.cos(a), sign * math.sin(a)
            i0, i1 = (i, i + d // 2) if pair_stride else (2 * i, 2 * i + 1)
            out[i0] = x[i0] * c - x[i1] * s
            out[i1] = x[i0] * s + x[i1] * c
        return out
    x = _rng(11).standard_normal(64)
    ok = rope_variant(x, 8195.0)
    np.testing.assert_allclose(ok, oracle.rope(x, 8195.0), rtol=1e-9, atol=1e-9)
    # clockwise turn: the quarter-turn pin sees (0, -1)
    e0 = np.zeros(64)
    e0[0] = 1.0
    assert rope_variant(e0, math.pi / 2, sign=-1.0)[1] == pytest.approx(-1.0)
    # frequencies base^(-i/d): pair 5's period pin fails
    period = 2.0 * math.pi * 10000.0 ** (2.0 * 5 / 64)
    assert not np.allclose(rope_variant(x, period, expo=1.0)[10:12], x[10:12], atol=1e-3)
    # half-split pairs (i, i + d/2) instead of adjacent ones: the phasor twin disagrees
    assert not np.allclose(rope_variant(x, 77.0, pair_stride=True), twin.rope_phasor(list(x), 77.0, 10000.0),
                           atol=1e-6)
    # a sine-only mistake in one component (x0 sin + x1 sin): lengths are not kept
    y = ok.copy()
    a = 8195.0
    y[1] = x[0] * math.sin(a) + x[1] * math.sin(a)
    assert not np.isclose(np.hypot(y[0], y[1]), np.hypot(x[0], x[1]))
