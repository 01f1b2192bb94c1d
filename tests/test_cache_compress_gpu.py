"""GPU parity of the compressed cache write (mla_cache_append_compressed: blocks of m new
tokens merged into one cache row, component-wise, with softmax weights over the block from
z = W^Z h -- the DeepSeek page's "KV cache compression" section) against the fp64 oracle: each
written number within one bf16 step of the exact merge (plus the fp32 arithmetic's share), at
most a few numbers a step away from the rounded exact value, every other pool byte unchanged,
and a decode over the compressed cache matching the oracle's decode over the oracle's rows."""
import numpy as np
import pytest
import torch

import mla_latent_kv_77_b300 as mla
from mla_latent_kv_77_b300 import workloads
import oracle
from helpers import bf16_ulp, check_lse, check_out

pytestmark = pytest.mark.gpu

DEV = "cuda"
FLIP_SHARE = 0.02


def _bits(t):
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def _bf16_bits_of(x64):
    u = np.asarray(x64, dtype=np.float32).view(np.uint32).astype(np.uint64)
    return (((u + 0x7FFF + ((u >> 16) & 1)) >> 16) & 0xFFFF).astype(np.uint16)


def _case(lens, nb, m, d_model, seed=0, shuffle=True):
    """lens: compressed lengths (the nb new rows included)."""
    case = workloads.make_case("c", lens, Tq=nb, causal=True, shuffle=shuffle, spare_pages=2, garbage="nan",
                               q_mode="none", seed=seed, device="cpu")
    h, w_dkv, w_kr = workloads.append_inputs(len(lens) * nb * m, d_model, seed=seed)
    w_z = workloads._randn_bf16((workloads.D, d_model), 1.0 / np.sqrt(d_model), seed, 12, "cpu")
    return case, h, w_dkv, w_kr, w_z


def _run(case, h, w_dkv, w_kr, w_z, nb, m, rope_base=mla.ROPE_BASE):
    pool = case.pool.to(DEV)
    before = _bits(pool).reshape(-1, workloads.D)
    mla.get_device_status()
    mla.cache_append_compressed(h.to(DEV), w_dkv.to(DEV), w_kr.to(DEV), w_z.to(DEV), case.block_table.to(DEV),
                                case.seq_lens.to(DEV), pool, n_blocks=nb, m=m, rope_base=rope_base)
    st, word = mla.get_device_status()
    return before, pool, st, word


def _check(case, before, pool, rows, slot):
    after = _bits(pool).reshape(-1, workloads.D)
    ok = slot >= 0
    written = slot[ok]
    keep = np.ones(after.shape[0], dtype=bool)
    keep[written] = False
    assert np.array_equal(after[keep], before[keep]), "rows outside the new rows' slots changed"
    got_bits = after[written]
    ref = rows[ok]
    got = (got_bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    assert np.all(np.isfinite(got))
    err = np.abs(got - ref)
    step = bf16_ulp(np.maximum(np.abs(ref), np.abs(got)))
    slack = 1e-3 * (1.0 + np.abs(ref).max(axis=1, keepdims=True))
    bad = err > step + slack
    if bad.any():
        i, j = np.argwhere(bad)[0]
        raise AssertionError(f"{int(bad.sum())} numbers off: row {i} column {j}: got {got[i, j]!r}, "
                             f"exact {ref[i, j]!r}")
    flips = float((got_bits != _bf16_bits_of(ref)).mean())
    assert flips <= FLIP_SHARE, f"{flips:.4f} of the numbers differ from the rounded exact merge"


CASES = {
    # 16 sequences x one block of 4 (CSA's m): 64 tokens, K split over clusters of 4
    "b16_m4": dict(lens=[40, 9, 300] + [70] * 13, nb=1, m=4, d_model=5120),
    # 8 sequences x two blocks of 4
    "b8_nb2_m4": dict(lens=[2, 65, 128, 7, 300, 64, 33, 90], nb=2, m=4, d_model=5120),
    # blocks of 32 over 128 tokens
    "b4_m32": dict(lens=[5, 100, 64, 3], nb=1, m=32, d_model=1024),
    # one block of 128 (HCA's m): the whole token tile is one block
    "b1_m128": dict(lens=[77], nb=1, m=128, d_model=512),
    # 120 tokens in blocks of 8, three sequences x five blocks, ragged token tile
    "b3_nb5_m8": dict(lens=[5, 129, 66], nb=5, m=8, d_model=2048),
    # m = 1: the plain cache write through the merge path
    "b5_m1": dict(lens=[10, 64, 65, 3, 200], nb=2, m=1, d_model=768),
}


@pytest.mark.parametrize("name", list(CASES))
def test_compressed_write_matches_oracle(name):
    c = CASES[name]
    case, h, w_dkv, w_kr, w_z = _case(c["lens"], c["nb"], c["m"], c["d_model"])
    before, pool, st, word = _run(case, h, w_dkv, w_kr, w_z, c["nb"], c["m"])
    assert st == 0 and word == 0, (st, word)
    rows, slot = oracle.cache_append_compressed(h, w_dkv, w_kr, w_z, case.block_table, case.seq_lens, c["nb"],
                                                c["m"], case.num_pages)
    assert (slot >= 0).all()
    _check(case, before, pool, rows, slot)


def test_decode_over_the_compressed_cache():
    """Two new blocks of 4 per sequence, then a causal decode of two queries per sequence over
    the compressed rows, against the oracle's decode over the oracle's merged rows (in the
    cache's bf16 format)."""
    lens, nb, m = [300, 66, 129, 2], 2, 4
    case, h, w_dkv, w_kr, w_z = _case(lens, nb, m, 5120, seed=5)
    _, pool, st, _ = _run(case, h, w_dkv, w_kr, w_z, nb, m)
    assert st == 0
    q = workloads._randn_bf16((len(lens), nb, workloads.H, workloads.D), 0.5, 5, 2, "cpu")
    o, lse = mla.decode(q.to(DEV), pool, case.block_table.to(DEV), case.seq_lens.to(DEV), causal=True)
    st, word = mla.get_device_status()
    assert st == 0, word
    rows, slot = oracle.cache_append_compressed(h, w_dkv, w_kr, w_z, case.block_table, case.seq_lens, nb, m,
                                                case.num_pages)
    # the cache stores bf16: the oracle's merged rows, rounded to the format (nearest even), are
    # the rows its decode reads (short sequences here consist mostly of new rows)
    ref_pool = case.pool.float().numpy().astype(np.float64).reshape(-1, workloads.D)
    ref_pool[slot] = (_bf16_bits_of(rows).astype(np.uint32) << 16).view(np.float32)
    ref_o, ref_l = oracle.decode_absorbed(q, ref_pool.reshape(case.pool.shape).astype(np.float32),
                                          case.block_table, case.seq_lens, workloads.SCALE, causal=True)
    check_out(o, ref_o)
    check_lse(lse, ref_l)
