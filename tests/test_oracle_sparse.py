"""Pins for the oracle's indexer path (the DeepSeek page's "KV cache data movement
minimization" section: every cached token also keeps a small index vector; a decoding
token scores all of them, keeps the k best, and attends over those tokens only).

The index scores are checked against dot products written out in pure Python, the top-k
against Python's own sort with the tie rule spelled as a key, and the sparse decode against
its limits: k >= L is the dense decode, k = 1 is a closed form, and the result is the dense
decode over a pool that holds only the selected tokens.  A mistake planted in a copy of the
selection (ties to the higher index) is caught.  CPU only."""
import math

import numpy as np
import pytest

import oracle


def _rng(seed):
    return np.random.default_rng(seed)


def _paged(rows_per_seq, page, rng, width):
    """Random rows laid out in a shuffled page pool; returns (pool, block_table, lens, dense)."""
    B = len(rows_per_seq)
    max_pages = max(1, max((L + page - 1) // page for L in rows_per_seq))
    n_pages = B * max_pages
    perm = rng.permutation(n_pages).astype(np.int32)
    bt = perm.reshape(B, max_pages)
    pool = rng.standard_normal((n_pages, page, width)).astype(np.float32)
    dense = [np.stack([pool[bt[b, t // page], t % page] for t in range(L)]) if L else np.zeros((0, width), np.float32)
             for b, L in enumerate(rows_per_seq)]
    return pool, bt, np.array(rows_per_seq, dtype=np.int32), dense


def test_index_scores_are_the_dot_products():
    rng = _rng(0)
    lens = [5, 0, 70, 64]
    ipool, bt, sl, dense = _paged(lens, 16, rng, 8)
    q = rng.standard_normal((4, 8)).astype(np.float32)
    s = oracle.index_scores(q, ipool, bt, sl)
    assert s.shape == (4, 70)
    for b, L in enumerate(lens):
        for t in range(L):
            want = sum(float(q[b, d]) * float(dense[b][t, d]) for d in range(8))
            assert abs(s[b, t] - want) <= 1e-12 * (1 + abs(want))
        assert np.all(np.isnan(s[b, L:]))


def test_index_scores_follow_the_block_table():
    """A basis query picks one coordinate of each token's index vector, page by page."""
    rng = _rng(1)
    ipool, bt, sl, dense = _paged([130], 64, rng, 16)
    for d in (0, 7, 15):
        q = np.zeros((1, 16), np.float32)
        q[0, d] = 1.0
        np.testing.assert_array_equal(oracle.index_scores(q, ipool, bt, sl)[0], dense[0][:, d].astype(np.float64))


def _sorted_topk(s, k):
    # Python's sort on the key (NaN last, larger first, lower index first) as an independent statement of the rule
    order = sorted(range(len(s)), key=lambda t: (math.isnan(s[t]), -s[t] if not math.isnan(s[t]) else 0.0, t))
    return sorted(order[:max(0, min(k, len(s)))])


@pytest.mark.parametrize("seed", range(6))
def test_topk_matches_a_sort(seed):
    rng = _rng(10 + seed)
    n = int(rng.integers(1, 300))
    s = np.round(rng.standard_normal(n) * 3) / 2  # many exact ties
    if seed % 2:
        s[rng.integers(0, n, 5)] = -np.inf
        s[rng.integers(0, n, 3)] = np.nan
    for k in (0, 1, 2, 7, n // 2, n - 1, n, n + 5):
        got = oracle.topk_row(s, k)
        assert list(got) == _sorted_topk(list(s), k), (n, k)


def test_topk_ties_take_the_lower_index():
    s = np.array([1.0, 3.0, 3.0, 3.0, 2.0, 3.0])
    assert list(oracle.topk_row(s, 2)) == [1, 2]
    assert list(oracle.topk_row(s, 4)) == [1, 2, 3, 5]
    assert list(oracle.topk_row(s, 5)) == [1, 2, 3, 4, 5]


def test_topk_ranks_nan_below_minus_infinity():
    s = np.array([np.nan, -np.inf, np.nan, -1e300])
    assert list(oracle.topk_row(s, 1)) == [3]
    assert list(oracle.topk_row(s, 2)) == [1, 3]
    assert list(oracle.topk_row(s, 3)) == [0, 1, 3]


def test_a_planted_tie_mistake_is_caught():
    """A selection that breaks ties toward the higher index disagrees with the sort."""
    def wrong(s, k):
        order = sorted(range(len(s)), key=lambda t: (-s[t], -t))
        return sorted(order[:k])
    s = list(np.round(_rng(3).standard_normal(50)))
    assert any(wrong(s, k) != list(oracle.topk_row(np.array(s), k)) for k in range(1, 50))


def _sparse_case(lens, seed, H=4, d_c=32, d_r=8, d_idx=8, page=16):
    rng = _rng(seed)
    D = d_c + d_r
    pool, bt, sl, dense = _paged(lens, page, rng, D)
    ipool = rng.standard_normal(pool.shape[:2] + (d_idx,)).astype(np.float32)
    q_abs = rng.standard_normal((len(lens), 1, H, D)) * 0.3
    q_idx = rng.standard_normal((len(lens), d_idx)).astype(np.float32)
    return q_abs, q_idx, pool, ipool, bt, sl, dense


def test_sparse_decode_with_k_at_least_the_length_is_the_dense_decode():
    q, qi, pool, ipool, bt, sl, _ = _sparse_case([40, 17, 33], 20)
    o_d, lse_d = oracle.decode_absorbed(q, pool, bt, sl, 0.25, d_c=32)
    for k in (40, 64):
        o, lse, sel = oracle.decode_sparse(q, qi, pool, ipool, bt, sl, k, 0.25, d_c=32)
        np.testing.assert_allclose(o, o_d, rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(lse, lse_d, rtol=1e-12, atol=1e-13)
        assert [list(x) for x in sel] == [list(range(L)) for L in (40, 17, 33)]


def test_sparse_decode_with_k_one_returns_the_best_token():
    q, qi, pool, ipool, bt, sl, dense = _sparse_case([50, 9], 21)
    o, lse, sel = oracle.decode_sparse(q, qi, pool, ipool, bt, sl, 1, 0.5, d_c=32)
    for b in range(2):
        idx = oracle.index_scores(qi, ipool, bt, sl)[b, :sl[b]]
        t = int(np.argmax(idx))
        assert list(sel[b]) == [t]
        row = dense[b][t].astype(np.float64)
        np.testing.assert_allclose(o[b, 0], np.tile(row[:32], (4, 1)), rtol=1e-13, atol=1e-13)
        np.testing.assert_allclose(lse[b, 0], 0.5 * (q[b, 0] @ row), rtol=1e-12, atol=1e-12)


def test_sparse_decode_is_the_dense_decode_over_the_selected_tokens():
    lens = [45, 30]
    q, qi, pool, ipool, bt, sl, dense = _sparse_case(lens, 22)
    k = 11
    o, lse, sel = oracle.decode_sparse(q, qi, pool, ipool, bt, sl, k, 0.3, d_c=32)
    for b in range(2):
        kept = dense[b][sel[b]]
        # brute force over the kept rows, one head at a time
        for h in range(4):
            s = 0.3 * (kept.astype(np.float64) @ q[b, 0, h])
            m = s.max()
            w = np.exp(s - m)
            np.testing.assert_allclose(lse[b, 0, h], m + math.log(w.sum()), rtol=1e-12, atol=1e-12)
            np.testing.assert_allclose(o[b, 0, h], (w / w.sum()) @ kept[:, :32].astype(np.float64), rtol=1e-11,
                                       atol=1e-12)


def test_sparse_decode_of_an_empty_sequence_is_empty():
    q, qi, pool, ipool, bt, sl, _ = _sparse_case([0, 5], 23)
    o, lse, sel = oracle.decode_sparse(q, qi, pool, ipool, bt, sl, 3, 0.3, d_c=32)
    assert sel[0].size == 0 and np.all(o[0] == 0) and np.all(np.isneginf(lse[0]))
    assert sel[1].size == 3


# ---------------------------------------------------------------------------------------------
# E4M3 index cache (index vectors held in 8 bits with one scale per token)
# ---------------------------------------------------------------------------------------------

def test_e4m3_values_from_the_format_definition():
    """Hand-computed codes: sign, 4 exponent bits (bias 7), 3 mantissa bits, subnormals at
    exponent 0, S.1111.111 the only NaN, no infinity."""
    cases = {0x00: 0.0, 0x38: 1.0, 0x3C: 1.5, 0x40: 2.0, 0xC0: -2.0, 0x7E: 448.0, 0xFE: -448.0,
             0x08: 2.0 ** -6, 0x07: 7 / 8 * 2.0 ** -6, 0x01: 2.0 ** -9, 0x30: 0.5, 0x77: 240.0, 0x7F: None,
             0xFF: None}
    for code, want in cases.items():
        got = oracle.e4m3_value(code)
        if want is None:
            assert math.isnan(got), hex(code)
        else:
            assert got == want, (hex(code), got, want)
    assert math.copysign(1.0, oracle.e4m3_value(0x80)) == -1.0


def test_e4m3_values_match_an_independent_conversion():
    """Every one of the 256 codes against torch's float8_e4m3fn conversion (written elsewhere)."""
    import torch
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).float().numpy()
    got = np.array([oracle.e4m3_value(c) for c in range(256)])
    both_nan = np.isnan(ref) & np.isnan(got)
    assert np.array_equal(got[~both_nan], ref[~both_nan].astype(np.float64))
    assert np.array_equal(np.isnan(ref), np.isnan(got))


def test_e4m3_codes_are_monotone_in_magnitude():
    vals = [oracle.e4m3_value(c) for c in range(0x7F)]
    assert all(a < b for a, b in zip(vals, vals[1:]))


def test_e4m3_index_scores_are_scaled_dot_products():
    rng = _rng(40)
    lens = [30, 3, 0]
    P, page, d = 8, 16, 8
    codes = rng.integers(0, 256, (P, page, d), dtype=np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x3A  # no NaN codes
    scale = rng.uniform(0.01, 2.0, (P, page)).astype(np.float32)
    bt = rng.permutation(P).astype(np.int32)[:6].reshape(3, 2)
    q = rng.standard_normal((3, d)).astype(np.float32)
    s = oracle.index_scores_e4m3(q, codes, scale, bt, np.array(lens, np.int32))
    for b, L in enumerate(lens):
        for t in range(L):
            pg, sl = bt[b, t // page], t % page
            want = float(scale[pg, sl]) * sum(float(q[b, i]) * oracle.e4m3_value(codes[pg, sl, i]) for i in range(d))
            assert abs(s[b, t] - want) <= 1e-12 * (1 + abs(want))


def test_e4m3_index_scores_equal_the_bf16_scores_of_the_decoded_vectors():
    """Decoding the codes, multiplying by the scales and scoring as a float index cache gives the
    same numbers (scale 1 and e4m3 values are exact in float32)."""
    rng = _rng(41)
    codes = rng.integers(0, 0x7E, (4, 16, 32), dtype=np.uint8)
    table = np.array([oracle.e4m3_value(c) for c in range(256)], dtype=np.float32)
    bt = np.arange(4, dtype=np.int32).reshape(2, 2)
    sl = np.array([32, 20], np.int32)
    q = rng.standard_normal((2, 32)).astype(np.float32)
    a = oracle.index_scores_e4m3(q, codes, np.ones((4, 16), np.float32), bt, sl)
    b = oracle.index_scores(q, table[codes], bt, sl)
    np.testing.assert_allclose(a, b, rtol=1e-13, atol=1e-13)
