"""Pins for the fp64 oracle, checked against things other than the oracle itself:
values printed on the pages (tests/golden), closed forms, invariants, and a
separately written pure-Python twin on tiny shapes.  CPU only."""
import json
import math
import os

import numpy as np
import pytest

import oracle
from oracle import cache_math, twin

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _rng(seed):
    return np.random.default_rng(seed)


def _bf16_like(x):
    """Round float64 values to bf16-representable float32 (RNE), so f32 storage is exact."""
    a = np.asarray(x, dtype=np.float32)
    u = a.view(np.uint32).astype(np.uint64)
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16) << 16
    return r.astype(np.uint32).view(np.float32)


def _small_problem(seed=0, B=2, Tq=1, H=3, d_h=5, d_c=8, d_r=3, page=4, lens=(7, 10),
                   shuffle=True, spare=2):
    rng = _rng(seed)
    pages_per = [(L + page - 1) // page for L in lens]
    P = sum(pages_per) + spare
    pool = _bf16_like(rng.standard_normal((P, page, d_c + d_r)) * 0.5)
    perm = rng.permutation(P) if shuffle else np.arange(P)
    maxp = max(pages_per)
    bt = -np.ones((B, maxp), dtype=np.int32)
    cur = 0
    for b in range(B):
        bt[b, :pages_per[b]] = perm[cur:cur + pages_per[b]]
        cur += pages_per[b]
    q_nope = _bf16_like(rng.standard_normal((B, Tq, H, d_h)) * 0.5)
    q_rope = _bf16_like(rng.standard_normal((B, Tq, H, d_r)) * 0.5)
    w_uk = _bf16_like(rng.standard_normal((H, d_h, d_c)) / math.sqrt(d_c))
    w_uv = _bf16_like(rng.standard_normal((H, d_h, d_c)) / math.sqrt(d_c))
    return dict(pool=pool, bt=bt, lens=np.array(lens, dtype=np.int32), q_nope=q_nope,
                q_rope=q_rope, w_uk=w_uk, w_uv=w_uv, d_c=d_c, page=page)


# ---------------------------------------------------------------------------
# Step 6 toy example (golden values printed on the page)
# ---------------------------------------------------------------------------
def test_toy_absorption_matches_printed_values():
    g = _golden("toy_absorption.json")
    W_uk = np.array(g["W_UK"], dtype=np.float32)[None]          # one head, d_h = d_c = 2
    q = np.array(g["q"], dtype=np.float32).reshape(1, 1, 2)     # the page's q = W_Q h
    c = np.array(g["c"], dtype=np.float32)
    q_abs = oracle.absorb_q(q, np.zeros((1, 1, 0), np.float32), W_uk)
    assert float(q_abs[0, 0] @ c) == g["score"]
    # Absorbing the columns of W_Q gives the rows of M = W_Q^T W_UK.
    WQ = np.array(g["W_Q"], dtype=np.float32)
    cols = WQ.T.reshape(2, 1, 2)
    M = oracle.absorb_q(cols, np.zeros((2, 1, 0), np.float32), W_uk)[:, 0, :]
    assert M.tolist() == g["M"]
    assert (M @ c).tolist() == g["Mc"]
    assert float(np.array(g["h"]) @ (M @ c)) == g["score"]


def test_toy_decode_one_token_both_forms():
    """A one-token context returns that token (absorbed: c; naive: W_UV c) and lse = its score."""
    g = _golden("toy_absorption.json")
    W_uk = np.array(g["W_UK"], dtype=np.float32)[None]
    W_uv = np.eye(2, dtype=np.float32)[None]
    pool = np.array(g["c"], dtype=np.float32).reshape(1, 1, 2)  # one page of one token, d_r = 0
    bt = np.zeros((1, 1), np.int32)
    lens = np.ones(1, np.int32)
    q = np.array(g["q"], dtype=np.float32).reshape(1, 1, 1, 2)
    q_abs = oracle.absorb_q(q, np.zeros((1, 1, 1, 0), np.float32), W_uk)
    o, lse = oracle.decode_absorbed(q_abs, pool, bt, lens, scale=1.0, d_c=2)
    assert o[0, 0, 0].tolist() == g["c"] and lse[0, 0, 0] == g["score"]
    out, lse2 = oracle.decode_naive(q, np.zeros((1, 1, 1, 0), np.float32), W_uk, W_uv, pool, bt,
                                    lens, scale=1.0)
    assert out[0, 0, 0].tolist() == g["c"] and lse2[0, 0, 0] == g["score"]


def test_two_channels_add_inside_softmax():
    """Step 7: per head the content score and the RoPE score add.  Integer toy: content 13
    (Step 6) plus q^R . k^R = (1,2).(3,4) = 11 gives a one-token lse of exactly 24."""
    g = _golden("toy_absorption.json")
    W_uk = np.array(g["W_UK"], dtype=np.float32)[None]
    W_uv = np.eye(2, dtype=np.float32)[None]
    row = np.array(g["c"] + [3, 4], dtype=np.float32).reshape(1, 1, 4)
    bt = np.zeros((1, 1), np.int32)
    lens = np.ones(1, np.int32)
    q = np.array(g["q"], dtype=np.float32).reshape(1, 1, 1, 2)
    qr = np.array([1, 2], dtype=np.float32).reshape(1, 1, 1, 2)
    q_abs = oracle.absorb_q(q, qr, W_uk)
    _, lse = oracle.decode_absorbed(q_abs, row, bt, lens, scale=1.0, d_c=2)
    _, lse_n = oracle.decode_naive(q, qr, W_uk, W_uv, row, bt, lens, scale=1.0)
    assert lse[0, 0, 0] == 24.0 and lse_n[0, 0, 0] == 24.0
    # and with two tokens the softmax mixes them: scores 24 and 0 (second token all zero)
    pool2 = np.concatenate([row, np.zeros((1, 1, 4), np.float32)], axis=1)
    lens2 = np.array([2], np.int32)
    o2, lse2 = oracle.decode_absorbed(q_abs, pool2, bt, lens2, scale=1.0, d_c=2)
    assert abs(lse2[0, 0, 0] - math.log(math.exp(24.0) + 1.0)) < 1e-12
    p0 = 1.0 / (1.0 + math.exp(-24.0))
    assert np.allclose(o2[0, 0, 0], p0 * np.array(g["c"]), rtol=1e-15, atol=0)


# ---------------------------------------------------------------------------
# Associativity (Step 6): naive == absorbed, fp64
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("causal,Tq", [(False, 1), (True, 3), (False, 2)])
def test_naive_equals_absorbed(causal, Tq):
    p = _small_problem(seed=1, Tq=Tq)
    scale = 1.0 / math.sqrt(5 + 3)
    out_n, lse_n = oracle.decode_naive(p["q_nope"], p["q_rope"], p["w_uk"], p["w_uv"], p["pool"],
                                       p["bt"], p["lens"], scale, causal)
    q_abs = oracle.absorb_q(p["q_nope"], p["q_rope"], p["w_uk"])
    o_lat, lse_a = oracle.decode_absorbed(q_abs, p["pool"], p["bt"], p["lens"], scale, causal,
                                          d_c=p["d_c"])
    out_a = oracle.up_proj(o_lat, p["w_uv"])
    assert np.allclose(out_a, out_n, rtol=1e-12, atol=1e-14)
    assert np.allclose(lse_a, lse_n, rtol=1e-13, atol=1e-13)


def test_naive_equals_absorbed_full_width_heads():
    """Same identity at the real widths (d_c=512, d_r=64, d_h=128), two heads, 70 tokens."""
    rng = _rng(5)
    H, d_h, d_c, d_r, page = 2, 128, 512, 64, 64
    pool = _bf16_like(rng.standard_normal((2, page, d_c + d_r)) * 0.5)
    bt = np.array([[1, 0]], np.int32)
    lens = np.array([70], np.int32)
    qn = _bf16_like(rng.standard_normal((1, 1, H, d_h)) * 0.5)
    qr = _bf16_like(rng.standard_normal((1, 1, H, d_r)) * 0.5)
    wk = _bf16_like(rng.standard_normal((H, d_h, d_c)) / math.sqrt(d_c))
    wv = _bf16_like(rng.standard_normal((H, d_h, d_c)) / math.sqrt(d_c))
    s = 1.0 / math.sqrt(192)
    out_n, lse_n = oracle.decode_naive(qn, qr, wk, wv, pool, bt, lens, s)
    o_lat, lse_a = oracle.decode_absorbed(oracle.absorb_q(qn, qr, wk), pool, bt, lens, s)
    assert np.allclose(oracle.up_proj(o_lat, wv), out_n, rtol=1e-11, atol=1e-14)
    assert np.allclose(lse_a, lse_n, rtol=1e-13, atol=1e-13)


# ---------------------------------------------------------------------------
# Closed forms and invariants of the softmax
# ---------------------------------------------------------------------------
def test_weights_sum_to_one():
    """Constant latent c_j = 1 for every token: o = sum_j p_j * 1 = 1 exactly iff sum p = 1."""
    p = _small_problem(seed=2)
    pool = p["pool"].copy()
    pool[..., :p["d_c"]] = 1.0
    q_abs = oracle.absorb_q(p["q_nope"], p["q_rope"], p["w_uk"])
    o, _ = oracle.decode_absorbed(q_abs, pool, p["bt"], p["lens"], 0.3, d_c=p["d_c"])
    assert np.allclose(o, 1.0, rtol=0, atol=1e-14)


def test_zero_query_gives_mean_and_log_n():
    p = _small_problem(seed=3)
    q_abs = np.zeros((2, 1, 3, p["d_c"] + 3), np.float32)
    o, lse = oracle.decode_absorbed(q_abs, p["pool"], p["bt"], p["lens"], 0.7, d_c=p["d_c"])
    for b, L in enumerate(p["lens"]):
        rows = twin.gather_rows(p["pool"], p["bt"][b], int(L), p["page"])
        mean = np.mean(np.array(rows)[:, :p["d_c"]].astype(np.float64), axis=0)
        assert np.allclose(o[b, 0], mean[None], rtol=1e-13, atol=1e-15)
        assert np.allclose(lse[b, 0], math.log(L), rtol=0, atol=1e-14)


def test_identical_rows_closed_form():
    p = _small_problem(seed=4)
    row = p["pool"][0, 0].copy()
    pool = np.broadcast_to(row, p["pool"].shape).copy()
    q_abs = _bf16_like(_rng(9).standard_normal((2, 1, 3, row.size)))
    s = 0.25
    o, lse = oracle.decode_absorbed(q_abs, pool, p["bt"], p["lens"], s, d_c=p["d_c"])
    for b, L in enumerate(p["lens"]):
        assert np.allclose(o[b, 0], row[:p["d_c"]].astype(np.float64)[None], rtol=1e-13, atol=1e-15)
        expect = s * (q_abs[b, 0].astype(np.float64) @ row.astype(np.float64)) + math.log(L)
        assert np.allclose(lse[b, 0], expect, rtol=1e-13, atol=1e-13)


def test_one_token_context_returns_its_latent():
    p = _small_problem(seed=6, lens=(1, 1))
    q_abs = oracle.absorb_q(p["q_nope"], p["q_rope"], p["w_uk"])
    o, lse = oracle.decode_absorbed(q_abs, p["pool"], p["bt"], p["lens"], 0.4, d_c=p["d_c"])
    for b in range(2):
        row = p["pool"][p["bt"][b, 0], 0].astype(np.float64)
        assert np.array_equal(o[b, 0], np.broadcast_to(row[:p["d_c"]], o[b, 0].shape))
        assert np.allclose(lse[b, 0], 0.4 * (q_abs[b, 0] @ row), rtol=1e-14, atol=1e-14)


def test_empty_sequence():
    p = _small_problem(seed=7, lens=(0, 5))
    q_abs = oracle.absorb_q(p["q_nope"], p["q_rope"], p["w_uk"])
    o, lse = oracle.decode_absorbed(q_abs, p["pool"], p["bt"], p["lens"], 0.4, d_c=p["d_c"])
    assert np.all(o[0] == 0.0) and np.all(np.isneginf(lse[0]))
    assert np.all(np.isfinite(lse[1]))


def test_block_table_permutation_invariance():
    a = _small_problem(seed=8, shuffle=False, spare=0)
    rng = _rng(10)
    P = a["pool"].shape[0]
    perm = rng.permutation(P)            # physical page perm[i] holds what page i held
    pool2 = np.empty_like(a["pool"])
    pool2[perm] = a["pool"]
    bt2 = np.where(a["bt"] >= 0, perm[np.maximum(a["bt"], 0)], -1).astype(np.int32)
    q_abs = oracle.absorb_q(a["q_nope"], a["q_rope"], a["w_uk"])
    o1, l1 = oracle.decode_absorbed(q_abs, a["pool"], a["bt"], a["lens"], 0.4, d_c=a["d_c"])
    o2, l2 = oracle.decode_absorbed(q_abs, pool2, bt2, a["lens"], 0.4, d_c=a["d_c"])
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_causal_equals_truncated_context():
    p = _small_problem(seed=11, Tq=3)
    q_abs = oracle.absorb_q(p["q_nope"], p["q_rope"], p["w_uk"])
    o, lse = oracle.decode_absorbed(q_abs, p["pool"], p["bt"], p["lens"], 0.4, True, d_c=p["d_c"])
    for t in range(3):
        lens_t = np.maximum(p["lens"] - (3 - 1 - t), 0).astype(np.int32)
        ot, lt = oracle.decode_absorbed(q_abs[:, t:t + 1].copy(), p["pool"], p["bt"], lens_t, 0.4,
                                        False, d_c=p["d_c"])
        assert np.array_equal(o[:, t], ot[:, 0]) and np.array_equal(lse[:, t], lt[:, 0])


def test_combine_of_page_splits_equals_whole():
    """Attention over disjoint token ranges, merged by log-sum-exp, equals the whole."""
    p = _small_problem(seed=12, lens=(13, 16), page=2)
    q_abs = oracle.absorb_q(p["q_nope"], p["q_rope"], p["w_uk"])
    o, lse = oracle.decode_absorbed(q_abs, p["pool"], p["bt"], p["lens"], 0.6, d_c=p["d_c"])
    parts_o, parts_l = [], []
    for lo, hi in [(0, 2), (2, 3), (3, 8)]:  # page ranges
        bt = np.full_like(p["bt"], -1)
        lens = np.zeros(2, np.int32)
        for b, L in enumerate(p["lens"]):
            npg = (int(L) + 1) // 2
            a, z = min(lo, npg), min(hi, npg)
            bt[b, :z - a] = p["bt"][b, a:z]
            lens[b] = max(0, min(int(L), z * 2) - a * 2)
        oo, ll = oracle.decode_absorbed(q_abs, p["pool"], bt, lens, 0.6, d_c=p["d_c"])
        parts_o.append(oo)
        parts_l.append(ll)
    oc, lc = oracle.combine(np.stack(parts_o), np.stack(parts_l))
    assert np.allclose(oc, o, rtol=1e-13, atol=1e-15)
    assert np.allclose(lc, lse, rtol=1e-14, atol=1e-14)


# ---------------------------------------------------------------------------
# Brute force: the independent pure-Python twin on tiny shapes
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("seed,causal", [(20, False), (21, True), (22, True)])
def test_oracle_matches_python_twin(seed, causal):
    p = _small_problem(seed=seed, B=2, Tq=2, H=2, d_h=3, d_c=4, d_r=2, page=2, lens=(5, 3))
    s = 0.8
    out_n, lse_n = oracle.decode_naive(p["q_nope"], p["q_rope"], p["w_uk"], p["w_uv"], p["pool"],
                                       p["bt"], p["lens"], s, causal)
    q_abs = oracle.absorb_q(p["q_nope"], p["q_rope"], p["w_uk"])
    o_lat, lse_a = oracle.decode_absorbed(q_abs, p["pool"], p["bt"], p["lens"], s, causal,
                                          d_c=p["d_c"])
    out_a = oracle.up_proj(o_lat, p["w_uv"])
    f = lambda a: np.asarray(a, dtype=np.float64).tolist()
    out_t, lse_t = twin.decode(f(p["q_nope"]), f(p["q_rope"]), f(p["w_uk"]), f(p["w_uv"]),
                               f(p["pool"]), p["bt"].tolist(), p["lens"].tolist(), s, causal)
    assert np.allclose(out_n, np.array(out_t), rtol=1e-12, atol=1e-15)
    assert np.allclose(out_a, np.array(out_t), rtol=1e-12, atol=1e-15)
    assert np.allclose(lse_n, np.array(lse_t), rtol=1e-13, atol=1e-14)
    assert np.allclose(lse_a, np.array(lse_t), rtol=1e-13, atol=1e-14)


def test_oracle_matches_twin_at_real_width_sampled_heads():
    """Real widths (576-wide rows, d_h=128), two heads, a ragged 67-token context."""
    rng = _rng(30)
    d_h, d_c, d_r, page = 128, 512, 64, 64
    pool = _bf16_like(rng.standard_normal((3, page, d_c + d_r)) * 0.5)
    bt = np.array([[2, 0]], np.int32)
    lens = np.array([67], np.int32)
    qa = _bf16_like(rng.standard_normal((1, 1, 2, d_c + d_r)) * 0.5)
    s = 1.0 / math.sqrt(192)
    o, lse = oracle.decode_absorbed(qa, pool, bt, lens, s)
    rows = twin.gather_rows(pool.astype(np.float64).tolist(), [2, 0], 67, page)
    for h in range(2):
        ot, lt = twin.attend_latent(qa[0, 0, h].astype(np.float64).tolist(), rows, d_c, s)
        assert np.allclose(o[0, 0, h], ot, rtol=1e-12, atol=1e-15)
        assert abs(lse[0, 0, h] - lt) < 1e-12


# ---------------------------------------------------------------------------
# Planted mistakes: the pins above must catch plausible slips (planted in the twin)
# ---------------------------------------------------------------------------
def test_pins_catch_planted_mistakes():
    g = _golden("toy_absorption.json")
    W_uk = [[float(x) for x in r] for r in g["W_UK"]]
    c = [float(x) for x in g["c"]]
    q = [float(x) for x in g["q"]]
    eye = [[1.0, 0.0], [0.0, 1.0]]
    # correct twin reproduces the printed score (and the two-channel toy 24)
    _, l = twin.attend_naive(q, [], W_uk, eye, [c], 2, 1.0)
    assert l == g["score"]
    _, l = twin.attend_naive(q, [1.0, 2.0], W_uk, eye, [c + [3.0, 4.0]], 2, 1.0)
    assert l == 24.0
    # transposed W_UK: k = W^T c = (3, 7) -> score 27, the toy pin fails
    WT = [list(r) for r in zip(*W_uk)]
    _, l = twin.attend_naive(q, [], WT, eye, [c], 2, 1.0)
    assert l != g["score"]
    # dropped RoPE channel: 13 instead of 24, the two-channel pin fails
    _, l = twin.attend_naive(q, [0.0, 0.0], W_uk, eye, [c + [3.0, 4.0]], 2, 1.0)
    assert l != 24.0
    # off-by-one causal window: the truncated-context pin would see a different row count
    rows = [[1.0, 0.0], [0.0, 1.0], [5.0, 5.0]]
    o_ok, _ = twin.attend_latent([0.0, 0.0], rows[:2], 2, 1.0)
    o_bad, _ = twin.attend_latent([0.0, 0.0], rows[:3], 2, 1.0)
    assert o_ok != o_bad


# ---------------------------------------------------------------------------
# Cache arithmetic (Steps 2, 4, 8) against the printed numbers
# ---------------------------------------------------------------------------
def test_cache_arithmetic_matches_printed_numbers():
    g = _golden("cache_arithmetic.json")
    s, pr = g["shapes"], g["printed"]
    mha = cache_math.mha_numbers_per_token(s["heads"], s["d_head"], s["layers"])
    mla = cache_math.mla_numbers_per_token(s["d_c"], s["d_r"], s["layers"])
    assert mha == pr["mha_numbers_per_token"]["value"]
    assert mla == pr["mla_numbers_per_token"]["value"]
    assert s["d_c"] + s["d_r"] == pr["mla_numbers_per_token_layer"]["value"]
    mb = cache_math.cache_bytes(mha, 1) / 1e6
    assert abs(mb - pr["mha_mb_per_token"]["value"]) <= pr["mha_mb_per_token"]["rounding"]
    gb = cache_math.cache_bytes(mha, s["report_tokens"]) / 1e9
    assert abs(gb - pr["mha_gb_report"]["value"]) <= pr["mha_gb_report"]["rounding"]
    assert gb < pr["node_gb"]["value"]
    assert abs(mha / mla - pr["ratio"]["value"]) <= pr["ratio"]["rounding"]
    gb2 = cache_math.cache_bytes(mla, s["report_tokens"]) / 1e9
    assert abs(gb2 - pr["mla_gb_report"]["value"]) <= pr["mla_gb_report"]["rounding"]
    pct = 100 * cache_math.reduction_fraction(mla, mha)
    assert abs(pct - pr["same_precision_saving_pct"]["value"]) <= pr["same_precision_saving_pct"]["rounding"]
    assert cache_math.gqa_equivalent_groups(s["d_c"], s["d_r"], s["d_head"]) == pr["gqa_equivalent_groups"]["value"]
    assert cache_math.gqa_reduction(s["heads"], 8) == pr["gqa8_cut"]["value"]
    assert cache_math.gqa_reduction(s["heads"], 1) == pr["mqa_cut"]["value"]
    pct2 = 100 * cache_math.reduction_fraction(pr["v2_deployed_kb"]["value"], pr["served_67b_kb"]["value"])
    assert abs(pct2 - pr["abstract_saving_pct"]["value"]) <= pr["abstract_saving_pct"]["rounding"]
