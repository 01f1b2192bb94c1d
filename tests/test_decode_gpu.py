"""GPU parity: the CUDA path through the C ABI against the fp64 oracle, element by
element, on seeded synthetic inputs; plus gather bit-exactness, split invariance,
edge cases and the device-side guards."""
import math

import numpy as np
import pytest
import torch

import mla_latent_kv_77_b300 as mla
from mla_latent_kv_77_b300 import workloads
import oracle
from helpers import check_lse, check_out, oracle_decode

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _gpu(case):
    return (case.q_abs.to(DEV) if case.q_abs is not None else None, case.pool.to(DEV),
            case.block_table.to(DEV), case.seq_lens.to(DEV))


def _clear_status():
    mla.get_device_status()


# small versions of the workloads: several tiles, ragged tails, the degenerate cases
SMALL = {
    "contiguous_b1_l512": dict(seq_lens=[512]),
    "paged_inorder_ragged": dict(seq_lens=[300, 64, 1000]),
    "shuffled_pool_nan_garbage": dict(seq_lens=[700, 1, 129, 64 * 9 + 5, 33], shuffle=True, spare_pages=5,
                                      garbage="nan"),
    "peaked_rows": dict(seq_lens=[3000, 1500], peaked_frac=0.01),
    "causal_tq4": dict(seq_lens=[516, 260, 4], Tq=4, causal=True),
    "causal_shorter_than_queries": dict(seq_lens=[2, 70], Tq=3, causal=True),
    "empty_and_single_token": dict(seq_lens=[0, 1, 65]),
    "noncausal_tq2": dict(seq_lens=[130, 77], Tq=2),
    "many_short": dict(seq_lens=[(17 * i) % 200 + 1 for i in range(40)], shuffle=True),
}


@pytest.mark.parametrize("name", sorted(SMALL))
def test_decode_matches_oracle_small(name):
    case = workloads.make_case(name, seed=3, **SMALL[name])
    _clear_status()
    q, pool, bt, sl = _gpu(case)
    o, lse = mla.decode(q, pool, bt, sl, case.scale, causal=case.causal)
    st, word = mla.get_device_status()
    assert st == 0 and word == 0
    ref_o, ref_lse = oracle_decode(case)
    check_out(o, ref_o)
    check_lse(lse, ref_lse)


@pytest.mark.parametrize("splits", [1, 2, 7, 1000])
def test_split_count_does_not_change_the_result(splits):
    case = workloads.make_case("splits", [64 * 20 + 9, 64 * 7, 3], shuffle=True, seed=5)
    q, pool, bt, sl = _gpu(case)
    o, lse = mla.decode(q, pool, bt, sl, case.scale, num_splits=splits)
    ref_o, ref_lse = oracle_decode(case)
    check_out(o, ref_o)
    check_lse(lse, ref_lse)
    o1, l1 = mla.decode(q, pool, bt, sl, case.scale, num_splits=1)
    d = (o.float() - o1.float()).abs().max().item()
    assert d <= 2e-2 and (lse - l1).abs().max().item() <= 1e-3


def test_gather_is_bit_exact_under_page_permutation():
    """The same logical cache laid out in order, or shuffled in a larger pool whose spare
    pages and tail slots hold NaN, gives bit-identical o_lat and lse."""
    lens = [64 * 11 + 3, 64 * 4, 200]
    a = workloads.make_case("inorder", lens, seed=9)
    b = workloads.make_case("shuffled", lens, shuffle=True, spare_pages=6, garbage="nan", seed=9)
    # place a's pages where b's table points
    for i, L in enumerate(lens):
        n = (L + 63) // 64
        b.pool[b.block_table[i, :n].long()] = a.pool[a.block_table[i, :n].long()]
        # and NaN in the unused tail of the last page
        tail = L - (n - 1) * 64
        b.pool[b.block_table[i, n - 1].long(), tail:] = float("nan")
    qa, pa, ba, sa = _gpu(a)
    o1, l1 = mla.decode(qa, pa, ba, sa, a.scale)
    o2, l2 = mla.decode(qa, b.pool.to(DEV), b.block_table.to(DEV), sa, a.scale)
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    assert torch.equal(l1.view(torch.int32), l2.view(torch.int32))


def test_absorb_q_matches_oracle_ragged_tokens():
    case = workloads.make_case("absorb", [1], Tq=1, q_mode="both", seed=11)
    g = torch.Generator().manual_seed(12)
    n = 130  # two token tiles, ragged
    q_nope = (torch.randn(n, 128, 128, generator=g) * 0.5).bfloat16()
    q_rope = (torch.randn(n, 128, 64, generator=g) * 0.5).bfloat16()
    q_abs = mla.absorb_q(q_nope.to(DEV), q_rope.to(DEV), case.w_uk.to(DEV))
    ref = oracle.absorb_q(q_nope, q_rope, case.w_uk)
    check_out(q_abs, ref, "q_abs")
    assert torch.equal(q_abs[..., 512:].cpu(), q_rope)  # RoPE part copied unchanged


def test_up_proj_matches_oracle_ragged_tokens():
    case = workloads.make_case("upproj", [1], Tq=1, q_mode="both", seed=13)
    g = torch.Generator().manual_seed(14)
    n = 200
    o_lat = (torch.randn(n, 128, 512, generator=g) * 0.05).bfloat16()
    out = mla.up_proj(o_lat.to(DEV), case.w_uv.to(DEV))
    ref = oracle.up_proj(o_lat.double().numpy(), case.w_uv)
    check_out(out, ref, "out")


def test_fused_path_matches_naive_oracle():
    """absorb -> decode -> up-proj against the naive form (per-head K, V rebuilt)."""
    case = workloads.make_case("fused", [300, 70], Tq=4, causal=True, q_mode="both", seed=15)
    qn, qr, wk, wv = (t.to(DEV) for t in (case.q_nope, case.q_rope, case.w_uk, case.w_uv))
    q_abs = mla.absorb_q(qn, qr, wk)
    o, lse = mla.decode(q_abs, case.pool.to(DEV), case.block_table.to(DEV), case.seq_lens.to(DEV), case.scale,
                        causal=True)
    out = mla.up_proj(o, wv)
    ref_out, ref_lse = oracle.decode_naive(case.q_nope, case.q_rope, case.w_uk, case.w_uv, case.pool,
                                           case.block_table, case.seq_lens, case.scale, causal=True)
    check_out(out, ref_out, "out")
    check_lse(lse, ref_lse)


def test_combine_matches_oracle():
    g = torch.Generator().manual_seed(16)
    R, rows = 5, 37
    o = torch.randn(R, rows, 512, generator=g) * 0.1
    l = torch.randn(R, rows, generator=g) * 3
    l[1, 3] = -math.inf
    l[:, 7] = -math.inf          # a row with no tokens at all
    o_out, l_out = mla.combine(o.to(DEV), l.to(DEV))
    ref_o, ref_l = oracle.combine(o.double().numpy(), l.double().numpy())
    check_out(o_out, ref_o, "combine")
    check_lse(l_out, ref_l)
    assert torch.all(o_out[7] == 0)


def test_bad_block_table_entry_sets_status_without_trapping():
    case = workloads.make_case("bad", [300], seed=17)
    q, pool, bt, sl = _gpu(case)
    bt_bad = bt.clone()
    bt_bad[0, 2] = case.num_pages + 1000
    _clear_status()
    mla.decode(q, pool, bt_bad, sl, case.scale)
    st, word = mla.get_device_status()
    assert st == mla.Status.DEVICE_FAULT and word & mla.DEV_BAD_BLOCK_TABLE
    # the context is still usable
    o, lse = mla.decode(q, pool, bt, sl, case.scale)
    assert mla.get_device_status() == (0, 0)
    ref_o, ref_lse = oracle_decode(case)
    check_out(o, ref_o)


def test_bad_sequence_length_sets_status():
    case = workloads.make_case("badlen", [100, 64], seed=18)
    q, pool, bt, sl = _gpu(case)
    _clear_status()
    mla.decode(q, pool, bt, torch.tensor([100, 64 * 50], dtype=torch.int32, device=DEV), case.scale)
    st, word = mla.get_device_status()
    assert st == mla.Status.DEVICE_FAULT and word & mla.DEV_BAD_SEQ_LEN


def test_bounded_wait_gives_up_and_context_survives():
    _clear_status()
    mla.test_bounded_wait(50)
    st, word = mla.get_device_status()
    assert st == mla.Status.DEVICE_FAULT and word == mla.DEV_WAIT_TIMEOUT
    case = workloads.make_case("after", [128], seed=19)
    q, pool, bt, sl = _gpu(case)
    o, lse = mla.decode(q, pool, bt, sl, case.scale)
    assert mla.get_device_status() == (0, 0)
    check_out(o, oracle_decode(case)[0])


@pytest.mark.parametrize("batch,q_len,causal", [(1100, 1, False), (700, 3, True)])
def test_large_batches_of_short_sequences(batch, q_len, causal):
    """Batches whose query count passes the planner's one-query-per-thread limit (1024: the
    queries are no longer sorted) and its shared-memory limit (2048: the planner's arrays move to
    the workspace), with short ragged sequences over a shuffled pool, against the oracle on every
    query."""
    g = torch.Generator().manual_seed(41 + batch)
    lens = [int(x) for x in torch.randint(1, 160, (batch,), generator=g)]
    if causal:
        lens = [max(L, q_len) for L in lens]
    case = workloads.make_case("many", lens, Tq=q_len, causal=causal, shuffle=True, spare_pages=7,
                               garbage="nan", seed=43)
    assert case.B * case.Tq > (2048 if q_len > 1 else 1024)
    _clear_status()
    q, pool, bt, sl = _gpu(case)
    o, lse = mla.decode(q, pool, bt, sl, case.scale, causal=causal)
    assert mla.get_device_status() == (0, 0)
    ref_o, ref_lse = oracle_decode(case)
    check_out(o, ref_o)
    check_lse(lse, ref_lse)


def test_b1_l512_fused_chain_matches_naive_oracle():
    """The single-sequence, 512-token workload at its own shape (contiguous cache as 8 identity
    pages) through absorb -> decode -> up-projection, against the naive form that rebuilds every
    head's keys and values (explainer Steps 5-7)."""
    case = workloads.make_workload("b1_l512", seed=0)
    qn, qr, wk, wv = (t.to(DEV) for t in (case.q_nope, case.q_rope, case.w_uk, case.w_uv))
    q_abs = mla.absorb_q(qn, qr, wk)
    o, lse = mla.decode(q_abs, case.pool.to(DEV), case.block_table.to(DEV), case.seq_lens.to(DEV), case.scale)
    out = mla.up_proj(o, wv)
    assert mla.get_device_status() == (0, 0)
    ref_out, ref_lse = oracle.decode_naive(case.q_nope, case.q_rope, case.w_uk, case.w_uv, case.pool,
                                           case.block_table, case.seq_lens, case.scale, causal=False)
    check_out(out, ref_out, "out")
    check_lse(lse, ref_lse)
