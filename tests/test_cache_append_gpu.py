"""GPU parity of the cache write (mla_cache_append, the step before the decode: c = W^DKV h and
k^R = RoPE(W^KR h) of the "DeepSeek-V2" explainer's Steps 5 and 7, scattered into the paged pool)
against the fp64 oracle: each written number is the bf16 rounding of the oracle's exact value
(a one-step difference allowed where fp32 accumulation lands next to a rounding midpoint), the
slot choice and every other pool byte are bit-exact, and a decode over the written cache matches
the oracle's decode over the oracle's rows."""
import math

import numpy as np
import pytest
import torch

import mla_latent_kv_77_b300 as mla
from mla_latent_kv_77_b300 import workloads
import oracle
from helpers import bf16_ulp, check_lse, check_out

pytestmark = pytest.mark.gpu

DEV = "cuda"
# at most this share of written numbers may sit one bf16 step from the rounded oracle value
FLIP_SHARE = 0.01


def _bf16_bits_of(x64: np.ndarray) -> np.ndarray:
    """Round float64 values to bf16 (nearest even, through float32) and return the 16-bit patterns."""
    u = np.asarray(x64, dtype=np.float32).view(np.uint32).astype(np.uint64)
    return (((u + 0x7FFF + ((u >> 16) & 1)) >> 16) & 0xFFFF).astype(np.uint16)


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def _run(ac, rope_base=mla.ROPE_BASE):
    c = ac.case
    pool = c.pool.to(DEV)
    before = _bits(pool).reshape(-1, workloads.D)
    mla.get_device_status()
    mla.cache_append(ac.h.to(DEV), ac.w_dkv.to(DEV), ac.w_kr.to(DEV), c.block_table.to(DEV), c.seq_lens.to(DEV),
                     pool, q_len=c.Tq, rope_base=rope_base)
    st, word = mla.get_device_status()
    return before, pool, st, word


def _magnitudes(ac, token_ids=None):
    """M[n, col] = sum_k |h[n, k]| |W[col, k]|, the scale of fp32 accumulation error in row n's
    column col (a RoPE pair mixes both of its columns, so those take the pair's larger M)."""
    h = np.abs(ac.h.float().numpy().astype(np.float64))
    if token_ids is not None:
        h = h[token_ids]
    w = np.abs(np.concatenate([ac.w_dkv.float().numpy(), ac.w_kr.float().numpy()]).astype(np.float64))
    m = h @ w.T
    r = m[:, workloads.D_C:]
    pair = np.maximum(r[:, 0::2], r[:, 1::2])
    m[:, workloads.D_C::2] = pair
    m[:, workloads.D_C + 1::2] = pair
    return m


def _check_written(ac, before, pool, rows, slot, token_ids=None):
    """rows/slot from the oracle for the tokens token_ids (all tokens when None).  Each written
    number must be the bf16 rounding of the exact value, or one bf16 step from it, give or take
    the fp32 accumulation error 2^-16 * sum_k |h_k W_k| (which decides the rounding of values near
    zero); at most FLIP_SHARE of them may take the neighbouring step."""
    after = _bits(pool).reshape(-1, workloads.D)
    ok = slot >= 0
    written = slot[ok]
    assert len(np.unique(written)) == len(written)
    if token_ids is None:
        # every row the oracle does not write is byte-for-byte what it was
        keep = np.ones(after.shape[0], dtype=bool)
        keep[written] = False
        assert np.array_equal(after[keep], before[keep]), "rows outside the new tokens' slots changed"
    got_bits = after[written]
    ref = rows[ok]
    acc = 2.0 ** -16 * _magnitudes(ac, token_ids)[ok]
    want_bits = _bf16_bits_of(ref)
    same = got_bits == want_bits
    got = (got_bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    assert np.all(np.isfinite(got))
    err = np.abs(got - ref)
    step = bf16_ulp(np.maximum(np.abs(ref), np.abs(got)))
    bad = ~same & (err > step + acc)
    if bad.any():
        i, j = np.argwhere(bad)[0]
        raise AssertionError(f"{int(bad.sum())} numbers off by more than one bf16 step: first at token row {i}, "
                             f"column {j}: got {got[i, j]!r}, exact {ref[i, j]!r}, step {step[i, j]:.3e}, "
                             f"accumulation bound {acc[i, j]:.3e}")
    flips = float((~same).mean())
    assert flips <= FLIP_SHARE, f"{flips:.4f} of the numbers differ from the rounded oracle value"
    return flips


def _small_case(lens, Tq, d_model, shuffle=True, spare_pages=3, garbage="nan", seed=0):
    return workloads.make_append_case("t", lens, Tq=Tq, d_model=d_model, shuffle=shuffle, spare_pages=spare_pages,
                                      garbage=garbage, seed=seed, device="cpu")


CASES = {
    # 64 new tokens of width 5120 after 4095 cached (one token tile, K split over a cluster of 8)
    "decode_step_b64": dict(lens=[4096] * 64, Tq=1, d_model=5120, shuffle=False, spare_pages=0, garbage=None),
    # 128 new tokens (4 per sequence), pages shuffled
    "causal_step_b32_tq4": dict(lens=[8192 + 4] * 32, Tq=4, d_model=5120),
    # 185 tokens: two token tiles (ragged second), 4 splits, NaN in every slot nobody owns
    "ragged_b5_tq37": dict(lens=[37, 100, 64 * 7 + 3, 1000, 2999], Tq=37, d_model=5120),
    # 17 K blocks over 8 splits (uneven)
    "uneven_split_d1088": dict(lens=[70, 5, 64, 130], Tq=5, d_model=1088),
    # one K block: no split at all
    "single_k_block_d64": dict(lens=[3, 64, 65], Tq=2, d_model=64),
    # a 1300-token prompt: 11 token tiles of 64-column tiles, no split
    "prefill_l1300": dict(lens=[1300], Tq=1300, d_model=1024),
    # two 1000-token prompts (one after 1000 cached tokens): 16 token tiles of 144-column tiles
    # (the prompt shape), ragged last tile
    "prefill_2x1000": dict(lens=[2000, 1000], Tq=1000, d_model=512),
}


@pytest.mark.parametrize("name", list(CASES))
def test_cache_write_matches_oracle(name):
    ac = _small_case(**CASES[name])
    before, pool, st, word = _run(ac)
    assert st == 0 and word == 0, (st, word)
    c = ac.case
    rows, slot = oracle.cache_append(ac.h, ac.w_dkv, ac.w_kr, c.block_table, c.seq_lens, c.Tq, c.num_pages)
    assert (slot >= 0).all()
    _check_written(ac, before, pool, rows, slot)


def test_other_rope_base():
    ac = _small_case([200, 90], 6, 512)
    before, pool, st, word = _run(ac, rope_base=500000.0)
    assert st == 0
    c = ac.case
    rows, slot = oracle.cache_append(ac.h, ac.w_dkv, ac.w_kr, c.block_table, c.seq_lens, c.Tq, c.num_pages,
                                     rope_base=500000.0)
    _check_written(ac, before, pool, rows, slot)


def test_full_size_prefill_sampled_tokens():
    """The 4096-token prompt at d_model 5120 (the prefill workload), checked on 48 sampled tokens."""
    ac = workloads.make_append_workload("prefill_l4096", device="cpu")
    before, pool, st, word = _run(ac)
    assert st == 0
    c = ac.case
    rng = np.random.default_rng(5)
    toks = np.sort(np.concatenate([[0, 1, 4095, 128, 127], rng.choice(4096, 43, replace=False)]))
    toks = np.unique(toks)
    # token t of the one sequence is at position t: as a batch of one-token sequences of length t + 1
    bt = c.block_table.numpy()[np.zeros(len(toks), dtype=np.int64)]
    rows, slot = oracle.cache_append(ac.h.float().numpy()[toks], ac.w_dkv, ac.w_kr, bt, toks + 1, 1, c.num_pages)
    assert slot.tolist() == (c.block_table.numpy()[0, toks // 64].astype(np.int64) * 64 + toks % 64).tolist()
    _check_written(ac, before, pool, rows, slot, token_ids=toks)
    # and nothing but the prompt's rows changed
    after = _bits(pool).reshape(-1, workloads.D)
    pages = c.block_table.numpy()[0]
    mask = np.ones(after.shape[0], dtype=bool)
    for p in pages[pages >= 0]:
        mask[p * 64:(p + 1) * 64] = False
    assert np.array_equal(after[mask], before[mask])


def test_rows_do_not_depend_on_where_they_go():
    """The same tokens through two different block tables: bit-identical rows."""
    lens, Tq, d = [300, 70, 129], 3, 2048
    a = _small_case(lens, Tq, d, shuffle=False, spare_pages=0, seed=3)
    b = _small_case(lens, Tq, d, shuffle=True, spare_pages=9, seed=3)
    assert torch.equal(a.h, b.h) and not torch.equal(a.case.block_table, b.case.block_table)
    _, pa, st_a, _ = _run(a)
    _, pb, st_b, _ = _run(b)
    assert st_a == 0 and st_b == 0
    _, sa = oracle.cache_append(a.h, a.w_dkv, a.w_kr, a.case.block_table, a.case.seq_lens, Tq, a.case.num_pages)
    _, sb = oracle.cache_append(b.h, b.w_dkv, b.w_kr, b.case.block_table, b.case.seq_lens, Tq, b.case.num_pages)
    ra = _bits(pa).reshape(-1, workloads.D)[sa]
    rb = _bits(pb).reshape(-1, workloads.D)[sb]
    assert np.array_equal(ra, rb)


def test_bad_lengths_and_pages_are_flagged_and_skipped():
    ac = _small_case([40, 2, 130, 66], 3, 256, spare_pages=2)
    c = ac.case
    c.seq_lens[1] = 2                      # shorter than its 3 new tokens: the first has position -1
    c.block_table[2, 2] = c.num_pages + 5   # sequence 2's last two new tokens (positions 128, 129)
    #                                         land on a page outside the pool; position 127 does not
    before, pool, st, word = _run(ac)
    assert st == mla.Status.DEVICE_FAULT
    assert word == (mla.DEV_BAD_SEQ_LEN | mla.DEV_BAD_BLOCK_TABLE)
    rows, slot = oracle.cache_append(ac.h, ac.w_dkv, ac.w_kr, c.block_table, c.seq_lens, c.Tq, c.num_pages)
    assert np.flatnonzero(slot < 0).tolist() == [3, 7, 8]
    _check_written(ac, before, pool, rows, slot)


def test_one_launch_per_call():
    for lens, Tq, d in (([4096] * 64, 1, 5120), ([1300], 1300, 1024), ([4096], 4096, 256)):
        ac = _small_case(lens, Tq, d, shuffle=False, spare_pages=0, garbage=None)
        _run(ac)
        n0 = mla.launch_count()
        _run(ac)
        assert mla.launch_count() - n0 == 1


def test_write_then_decode_matches_oracle_chain():
    """Four new tokens per sequence written by the cache write, then the causal decode of those
    tokens' queries over the whole cache: against the oracle's decode over the oracle's rows."""
    lens = [300, 1000, 64 * 5 + 4, 2000]
    Tq = 4
    ac = _small_case(lens, Tq, 5120, spare_pages=4, seed=7)
    c = ac.case
    pool = c.pool.to(DEV)
    mla.get_device_status()
    mla.cache_append(ac.h.to(DEV), ac.w_dkv.to(DEV), ac.w_kr.to(DEV), c.block_table.to(DEV), c.seq_lens.to(DEV),
                     pool, q_len=Tq)
    q = workloads._randn_bf16((len(lens), Tq, workloads.H, workloads.D), 0.5, 7, 2, "cpu")
    o_lat, lse = mla.decode(q.to(DEV), pool, c.block_table.to(DEV), c.seq_lens.to(DEV), causal=True)
    st, word = mla.get_device_status()
    assert st == 0, word
    rows, slot = oracle.cache_append(ac.h, ac.w_dkv, ac.w_kr, c.block_table, c.seq_lens, Tq, c.num_pages)
    ref_pool = c.pool.float().numpy().astype(np.float64).reshape(-1, workloads.D)
    ref_pool[slot] = rows
    ref_pool = ref_pool.reshape(c.pool.shape)
    ref_o, ref_lse = oracle.decode_absorbed(q, ref_pool.astype(np.float32), c.block_table, c.seq_lens,
                                            workloads.SCALE, causal=True)
    check_out(o_lat, ref_o)
    check_lse(lse, ref_lse)
