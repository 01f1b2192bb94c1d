"""GPU parity of the indexer decode path (the DeepSeek page's "KV cache data movement
minimization": index scores over every cached token, the top k, attention over the selected
tokens only) against the fp64 oracle.

  * index scores: every written score within the fp32 summation bound of the exact dot product,
    and entries past each length left untouched;
  * top-k: the selection is integer work decided by fp32 scores, so the oracle's selection is
    taken on the kernel's own scores and must match exactly (positions, order, -1 padding,
    lengths), for tie-heavy, NaN, -inf and signed-zero scores as well; the gathered rows are
    bit-for-bit the pool's rows and the rest of the compact pool is zero;
  * against the oracle's selection from its own fp64 scores, positions may differ only where
    two scores are within the fp32 bound of each other;
  * the sparse decode's o_lat / lse against the oracle's decode over the selected rows, and the
    k >= L case against the oracle's dense decode;
  * at the full 128K size, the scores of sampled sequences and the selection of all of them.
"""
import numpy as np
import pytest
import torch

import mla_latent_kv_77_b300 as mla
from mla_latent_kv_77_b300 import workloads
import oracle
from helpers import check_lse, check_out

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _to_dev(sc):
    c = sc.case
    return dict(q_abs=c.q_abs.to(DEV), pool=c.pool.to(DEV), bt=c.block_table.to(DEV), sl=c.seq_lens.to(DEV),
                idx=sc.idx_pool.to(DEV), q_idx=sc.q_idx.to(DEV))


def _np(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def _score_bound(sc):
    """fp32 summation bound per token: d_idx * 2^-24 * sum_i |q_i k_i| (products are exact)."""
    c = sc.case
    q = np.abs(_np(sc.q_idx))
    ip = np.abs(_np(sc.idx_pool))
    bt, sl = c.block_table.numpy(), c.seq_lens.numpy()
    L = int(sl.max()) if sl.size else 0
    out = np.zeros((c.B, max(1, L)))
    for b in range(c.B):
        for t0 in range(0, int(sl[b]), 64):
            n = min(64, int(sl[b]) - t0)
            out[b, t0:t0 + n] = ip[bt[b, t0 // 64], :n] @ q[b]
    return out * sc.d_idx * 2.0 ** -24 + 1e-30


def _check_scores(sc, got):
    c = sc.case
    ref = oracle.index_scores(_np(sc.q_idx), _np(sc.idx_pool), c.block_table.numpy(), c.seq_lens.numpy())
    bound = _score_bound(sc)
    g = got.cpu().numpy().astype(np.float64)
    for b in range(c.B):
        L = int(c.seq_lens[b])
        err = np.abs(g[b, :L] - ref[b, :L])
        assert np.all(err <= bound[b, :L]), (b, float((err / bound[b, :L]).max()))
    return ref


@pytest.mark.parametrize("d_idx", [32, 64, 128, 256])
def test_index_scores_match_oracle(d_idx):
    sc = workloads.make_sparse_case("s", [1, 63, 64, 65, 700, 0, 1500], k=8, d_idx=d_idx, shuffle=True,
                                    spare_pages=3, garbage="nan", seed=d_idx)
    d = _to_dev(sc)
    sentinel = torch.full((sc.case.B, sc.case.max_pages * 64), 12345.0, device=DEV)
    got = mla.index_scores(d["q_idx"], d["idx"], d["bt"], d["sl"], scores=sentinel)
    torch.cuda.synchronize()
    _check_scores(sc, got)
    for b in range(sc.case.B):
        assert torch.all(got[b, int(sc.case.seq_lens[b]):] == 12345.0), "entries past the length were written"
    assert mla.get_device_status() == (0, 0)


def _check_selection(scores_cpu, sl, k, sel_index, sel_lens, sel_bt, sel_pool=None, pool=None, bt=None):
    B = scores_cpu.shape[0]
    npk = (k + 63) // 64
    si, sn = sel_index.cpu().numpy(), sel_lens.cpu().numpy()
    assert np.array_equal(sel_bt.cpu().numpy(), np.arange(B * npk, dtype=np.int32).reshape(B, npk))
    for b in range(B):
        L = int(sl[b])
        want = oracle.topk_row(scores_cpu[b, :L].astype(np.float64), k) if L else np.zeros(0, np.int64)
        n = len(want)
        assert sn[b] == n
        assert np.array_equal(si[b, :n], want), (b, np.setdiff1d(si[b, :n], want)[:5], np.setdiff1d(want, si[b, :n])[:5])
        assert np.all(si[b, n:] == -1)
        if sel_pool is not None:
            rows = sel_pool[b * npk:(b + 1) * npk].reshape(npk * 64, -1)
            if n:
                t = torch.as_tensor(want, device=pool.device)
                src = pool[bt[b, t // 64].long(), t % 64]
                assert torch.equal(rows[:n].view(torch.int16), src.view(torch.int16)), b
            assert torch.all(rows[n:].view(torch.int16) == 0), b


@pytest.mark.parametrize("k", [1, 7, 64, 100, 512, 5000])
def test_topk_gather_matches_oracle_on_the_kernels_scores(k):
    sc = workloads.make_sparse_case("s", [0, 5, 64, 700, 4097, 20000, 1], k=k, shuffle=True, spare_pages=2, seed=k)
    d = _to_dev(sc)
    scores = mla.index_scores(d["q_idx"], d["idx"], d["bt"], d["sl"])
    si, sp, sbt, sn = mla.topk_gather(scores, d["sl"], d["pool"], d["bt"], k)
    torch.cuda.synchronize()
    _check_selection(scores.cpu().numpy(), sc.case.seq_lens.numpy(), k, si, sn, sbt, sp, d["pool"], d["bt"])
    assert mla.get_device_status() == (0, 0)


@pytest.mark.parametrize("seed", range(4))
def test_topk_ties_nan_inf_and_signed_zeros(seed):
    """Crafted scores: small integers (thousands of exact ties), -inf, NaN, -0.0 beside +0.0."""
    g = torch.Generator().manual_seed(seed)
    lens = [3000, 1, 130, 9000]
    B, max_pages = len(lens), (max(lens) + 63) // 64
    s = torch.randint(-3, 4, (B, max_pages * 64), generator=g).float()
    s[s == 0] = torch.where(torch.rand(int((s == 0).sum()), generator=g) < 0.5, -0.0, 0.0)
    m = torch.rand(s.shape, generator=g)
    s[m < 0.05] = float("-inf")
    s[(m >= 0.05) & (m < 0.08)] = float("nan")
    if seed == 3:
        s[0, :] = float("nan")  # a sequence of NaN only: the lowest positions win
    case = workloads.make_case("t", lens, shuffle=True, q_mode="none", seed=seed)
    pool, bt, sl = case.pool.to(DEV), case.block_table.to(DEV), case.seq_lens.to(DEV)
    for k in (1, 2, 100, 1000, 2999, 3000, 8999):
        si, sp, sbt, sn = mla.topk_gather(s.to(DEV), sl, pool, bt, k)
        torch.cuda.synchronize()
        _check_selection(s.numpy(), case.seq_lens.numpy(), k, si, sn, sbt, sp, pool, bt)


@pytest.mark.parametrize("k", [1, 1000, 30000])
def test_topk_long_tie_heavy_slices(k):
    """70000 integer scores: every warp's share of the candidates overflows its list, so the
    kernel takes its full-scan path; and one sequence of distinct scores beside it."""
    g = torch.Generator().manual_seed(k)
    lens = [70000, 70000]
    max_pages = (max(lens) + 63) // 64
    s = torch.randint(-3, 4, (2, max_pages * 64), generator=g).float()
    s[1] = torch.randn(max_pages * 64, generator=g)
    case = workloads.make_case("t", lens, shuffle=True, q_mode="none", seed=k)
    pool, bt, sl = case.pool.to(DEV), case.block_table.to(DEV), case.seq_lens.to(DEV)
    si, sp, sbt, sn = mla.topk_gather(s.to(DEV), sl, pool, bt, k)
    torch.cuda.synchronize()
    _check_selection(s.numpy(), case.seq_lens.numpy(), k, si, sn, sbt, sp, pool, bt)
    assert mla.get_device_status() == (0, 0)


@pytest.mark.parametrize("k", [1, 700, 5000])
def test_topk_past_the_shared_memory_copy(k):
    """409600 positions: each CTA's slice (51200) is longer than the shared-memory key copy holds,
    so every pass reads the scores from global memory.  The block table aliases 8 physical pages
    (reads only), and a second sequence of integer scores (ties) rides along."""
    g = torch.Generator().manual_seed(100 + k)
    max_pages = 6400
    lens = [max_pages * 64, 300000]
    s = torch.randn(2, max_pages * 64, generator=g)
    s[1] = torch.randint(-3, 4, (max_pages * 64,), generator=g).float()
    pool = workloads._randn_bf16((8, 64, workloads.D), 0.5, k, 1, DEV)
    bt = (torch.arange(max_pages, dtype=torch.int32) % 8).repeat(2, 1).contiguous()
    sl = torch.tensor(lens, dtype=torch.int32)
    si, sp, sbt, sn = mla.topk_gather(s.to(DEV), sl.to(DEV), pool, bt.to(DEV), k)
    torch.cuda.synchronize()
    _check_selection(s.numpy(), lens, k, si, sn, sbt, sp, pool, bt.to(DEV))
    assert mla.get_device_status() == (0, 0)


def test_sparse_decode_many_clusters():
    """64 sequences: 512 top-k CTAs run in several waves; checked on four of them."""
    k = 100
    lens = [2000 + 37 * i for i in range(64)]
    sc = workloads.make_sparse_case("s", lens, k=k, shuffle=True, seed=70)
    d = _to_dev(sc)
    o, lse, si = mla.decode_sparse(d["q_abs"], d["q_idx"], d["pool"], d["idx"], d["bt"], d["sl"], k)
    scores = mla.index_scores(d["q_idx"], d["idx"], d["bt"], d["sl"])
    torch.cuda.synchronize()
    assert mla.get_device_status() == (0, 0)
    s_np, sel = scores.cpu().numpy(), si.cpu().numpy()
    for b in range(64):
        assert np.array_equal(sel[b], oracle.topk_row(s_np[b, :lens[b]].astype(np.float64), k)), b
    seqs = [0, 21, 42, 63]
    o_ref, l_ref, extra = _oracle_over_selection(sc, sel, np.full(64, k), seqs)
    _check_sparse_out(o[seqs], o_ref, extra)
    check_lse(lse[seqs], l_ref)


def test_selection_agrees_with_the_oracles_own_scores_up_to_near_ties():
    sc = workloads.make_sparse_case("s", [30000, 12000], k=300, shuffle=True, seed=5)
    d = _to_dev(sc)
    scores = mla.index_scores(d["q_idx"], d["idx"], d["bt"], d["sl"])
    si, _, _, sn = mla.topk_gather(scores, d["sl"], d["pool"], d["bt"], 300)
    ref = oracle.index_scores(_np(sc.q_idx), _np(sc.idx_pool), sc.case.block_table.numpy(), sc.case.seq_lens.numpy())
    bound = _score_bound(sc)
    for b in range(2):
        L = int(sc.case.seq_lens[b])
        want = oracle.topk_row(ref[b, :L], 300)
        got = si[b, :int(sn[b])].cpu().numpy()
        kth = np.sort(ref[b, :L])[::-1][299]
        for t in np.setxor1d(got, want):
            assert abs(ref[b, t] - kth) <= 2 * bound[b, t] + 2 * bound[b].max(), (b, t)


def _p_rounding_bound(q_abs, rows, scale, d_c=512):
    """|o| error the kernel's arithmetic allows beyond the final bf16 rounding (q_abs [H, 576], rows
    [n, 576], float64 copies of the bf16 inputs; returns [H, d_c]):
      * P is rounded to bf16 (relative 2^-9) before the PV product: up to 2^-9 sum_t p_t |v_t|;
      * each score is an fp32 sum of 576 exact products, off by at most
        ds_t = 576 * 2^-24 * scale * sum_i |q_i r_ti| (twice that, for the tensor pipe's own
        accumulation order), which moves p_t by p_t ds_t and o by sum_t p_t ds_t |v_t - o|
        <= sum_t p_t ds_t (|v_t| + |o|)."""
    if rows.shape[0] == 0:
        return np.zeros((q_abs.shape[0], d_c))
    s = scale * (q_abs @ rows.T)
    p = np.exp(s - s.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    v = np.abs(rows[:, :d_c])
    ds = 2.0 * 576 * 2.0 ** -24 * scale * (np.abs(q_abs) @ np.abs(rows).T)
    o = np.abs(p @ rows[:, :d_c])
    pds = p * ds
    return 2.0 ** -9 * (p @ v) + pds @ v + pds.sum(axis=1, keepdims=True) * o


def _check_sparse_out(o, o_ref, extra):
    """Elementwise: the shared bound max(2e-2, 1 bf16 ulp), or half an ulp of the final rounding
    plus the P-rounding term when that is larger (outputs made of a few peaked rows), plus 1e-3 of
    fp32 slack; and the shared relative-L2 bound."""
    from helpers import bf16_ulp
    g = o.detach().float().cpu().numpy().astype(np.float64)
    ref = np.asarray(o_ref, dtype=np.float64)
    assert np.all(np.isfinite(g))
    bound = np.maximum(np.maximum(2e-2, bf16_ulp(ref)), 0.5 * bf16_ulp(ref) + extra + 1e-3)
    err = np.abs(g - ref)
    assert np.all(err <= bound), float((err / bound).max())
    check_out(o, o_ref, atol=np.inf)  # the relative-L2 part


def _oracle_over_selection(sc, sel_index, sel_lens, seqs):
    c = sc.case
    pool = c.pool.float().numpy()
    bt = c.block_table.numpy()
    o_all, l_all, x_all = [], [], []
    for b in seqs:
        n = int(sel_lens[b])
        t = sel_index[b, :n]
        rows = pool[bt[b, t // 64], t % 64] if n else np.zeros((0, workloads.D), np.float32)
        npg = max(1, (n + 63) // 64)
        comp = np.zeros((npg, 64, workloads.D), np.float32)
        comp.reshape(-1, workloads.D)[:n] = rows
        o, l = oracle.decode_absorbed(c.q_abs[b:b + 1].float().numpy(), comp, np.arange(npg, dtype=np.int32)[None],
                                      np.array([n], np.int32), c.scale)
        o_all.append(o[0])
        l_all.append(l[0])
        x_all.append(_p_rounding_bound(c.q_abs[b, 0].double().numpy(), rows.astype(np.float64), c.scale)[None])
    return np.stack(o_all), np.stack(l_all), np.stack(x_all)


@pytest.mark.parametrize("k", [1, 100, 512, 2000])
def test_decode_sparse_matches_oracle(k):
    """k <= 1024 decodes each sequence's selection whole; k = 2000 goes through the split plan."""
    sc = workloads.make_sparse_case("s", [0, 40, 700, 5000, 20000], k=k, shuffle=True, spare_pages=2, garbage="nan",
                                    peaked_frac=0.01, seed=10 + k)
    d = _to_dev(sc)
    o, lse, si = mla.decode_sparse(d["q_abs"], d["q_idx"], d["pool"], d["idx"], d["bt"], d["sl"], k)
    torch.cuda.synchronize()
    assert mla.get_device_status() == (0, 0)
    sel = si.cpu().numpy()
    lens = np.minimum(sc.case.seq_lens.numpy(), k)
    # the selection is the oracle's on the kernel's scores
    scores = mla.index_scores(d["q_idx"], d["idx"], d["bt"], d["sl"]).cpu().numpy()
    for b in range(sc.case.B):
        L = int(sc.case.seq_lens[b])
        want = oracle.topk_row(scores[b, :L].astype(np.float64), k) if L else np.zeros(0)
        assert np.array_equal(sel[b, :lens[b]], want)
    o_ref, l_ref, extra = _oracle_over_selection(sc, sel, lens, range(sc.case.B))
    _check_sparse_out(o, o_ref, extra)
    check_lse(lse, l_ref)


def test_decode_sparse_with_k_above_every_length_is_the_dense_decode():
    sc = workloads.make_sparse_case("s", [1, 64, 300, 999], k=1000, shuffle=True, seed=3)
    d = _to_dev(sc)
    o, lse, si = mla.decode_sparse(d["q_abs"], d["q_idx"], d["pool"], d["idx"], d["bt"], d["sl"], 1000)
    torch.cuda.synchronize()
    o_ref, l_ref = oracle.decode_absorbed(sc.case.q_abs.float().numpy(), sc.case.pool.float().numpy(),
                                          sc.case.block_table.numpy(), sc.case.seq_lens.numpy(), sc.case.scale)
    check_out(o, o_ref)
    check_lse(lse, l_ref)
    sel = si.cpu().numpy()
    for b, L in enumerate(sc.case.seq_lens.tolist()):
        assert np.array_equal(sel[b, :L], np.arange(L)) and np.all(sel[b, L:] == -1)


def _check_scores_e4m3(sc, got):
    """Each score within (d_idx + 1) * 2^-24 * scale * sum |q_i v_i| of the oracle's: the products
    of a bf16 coordinate and an E4M3 value are exact in fp32, the sum and the scale round."""
    c = sc.case
    codes, scale = sc.idx_codes.cpu().numpy(), sc.idx_scale.cpu().numpy()
    ref = oracle.index_scores_e4m3(_np(sc.q_idx), codes, scale, c.block_table.numpy(), c.seq_lens.numpy())
    table = np.array([oracle.e4m3_value(x) for x in range(256)])
    absv = np.abs(table[codes]) * scale[..., None]
    q = np.abs(_np(sc.q_idx))
    g = got.cpu().numpy().astype(np.float64)
    bt = c.block_table.numpy()
    for b in range(c.B):
        L = int(c.seq_lens[b])
        if L == 0:
            continue
        t = np.arange(L)
        mag = absv[bt[b, t // 64], t % 64] @ q[b]
        bound = (sc.d_idx + 1) * 2.0 ** -24 * mag + 1e-30
        err = np.abs(g[b, :L] - ref[b, :L])
        assert np.all(err <= bound), (b, float((err / bound).max()))
    return ref


@pytest.mark.parametrize("d_idx", [32, 64, 128, 256])
def test_index_scores_e4m3_match_oracle(d_idx):
    sc = workloads.make_sparse_case("s", [1, 63, 64, 65, 700, 0, 1500], k=8, d_idx=d_idx, shuffle=True,
                                    spare_pages=3, e4m3=True, seed=50 + d_idx)
    d = _to_dev(sc)
    codes, scale = sc.idx_codes.to(DEV), sc.idx_scale.to(DEV)
    sentinel = torch.full((sc.case.B, sc.case.max_pages * 64), 12345.0, device=DEV)
    got = mla.index_scores_e4m3(d["q_idx"], codes, scale, d["bt"], d["sl"], scores=sentinel)
    torch.cuda.synchronize()
    _check_scores_e4m3(sc, got)
    for b in range(sc.case.B):
        assert torch.all(got[b, int(sc.case.seq_lens[b]):] == 12345.0)
    assert mla.get_device_status() == (0, 0)


def test_e4m3_nan_codes_give_nan_scores_that_rank_last():
    """A token whose codes include S.1111.111 (NaN) scores NaN, as the oracle's decoding says,
    and is picked only after every other token."""
    sc = workloads.make_sparse_case("s", [200], k=8, d_idx=64, e4m3=True, seed=80)
    codes = sc.idx_codes.clone()
    bt = sc.case.block_table
    bad = [3, 64, 150]
    for t, c in zip(bad, (0x7F, 0xFF, 0x7F)):
        codes[bt[0, t // 64], t % 64, 5] = c
    d = _to_dev(sc)
    scores = mla.index_scores_e4m3(d["q_idx"], codes.to(DEV), sc.idx_scale.to(DEV), d["bt"], d["sl"])
    torch.cuda.synchronize()
    g = scores.cpu().numpy()[0, :200]
    ref = oracle.index_scores_e4m3(_np(sc.q_idx), codes.numpy(), sc.idx_scale.numpy(), bt.numpy(),
                                   sc.case.seq_lens.numpy())[0]
    assert np.array_equal(np.isnan(g), np.isnan(ref)) and sorted(np.where(np.isnan(g))[0]) == bad
    si, _, _, sn = mla.topk_gather(scores, d["sl"], d["pool"], d["bt"], 199)
    sel = si.cpu().numpy()[0, :int(sn[0])]
    assert np.array_equal(sel, oracle.topk_row(g.astype(np.float64), 199))
    assert set(bad) - set(sel.tolist()) == {150}  # of the three NaN tokens the two lowest are taken last


def test_decode_sparse_with_an_e4m3_index_cache():
    k = 300
    sc = workloads.make_sparse_case("s", [0, 40, 700, 5000, 20000], k=k, shuffle=True, spare_pages=2, garbage="nan",
                                    e4m3=True, seed=60)
    d = _to_dev(sc)
    codes, scale = sc.idx_codes.to(DEV), sc.idx_scale.to(DEV)
    o, lse, si = mla.decode_sparse(d["q_abs"], d["q_idx"], d["pool"], codes, d["bt"], d["sl"], k, idx_scale=scale)
    torch.cuda.synchronize()
    assert mla.get_device_status() == (0, 0)
    scores = mla.index_scores_e4m3(d["q_idx"], codes, scale, d["bt"], d["sl"])
    _check_scores_e4m3(sc, scores)
    s_np = scores.cpu().numpy()
    sel = si.cpu().numpy()
    lens = np.minimum(sc.case.seq_lens.numpy(), k)
    for b in range(sc.case.B):
        L = int(sc.case.seq_lens[b])
        want = oracle.topk_row(s_np[b, :L].astype(np.float64), k) if L else np.zeros(0)
        assert np.array_equal(sel[b, :lens[b]], want)
    o_ref, l_ref, extra = _oracle_over_selection(sc, sel, lens, range(sc.case.B))
    _check_sparse_out(o, o_ref, extra)
    check_lse(lse, l_ref)


def test_bad_block_table_and_length_are_reported_not_faulted():
    sc = workloads.make_sparse_case("s", [200, 100], k=16, seed=4)
    d = _to_dev(sc)
    bt = d["bt"].clone()
    bt[0, 1] = 10 ** 6  # tokens 64..127 of sequence 0 on a page outside the pool
    scores = mla.index_scores(d["q_idx"], d["idx"], bt, d["sl"])
    torch.cuda.synchronize()
    assert mla.get_device_status()[1] == mla.DEV_BAD_BLOCK_TABLE
    s = scores.cpu()
    assert torch.all(torch.isnan(s[0, 64:128])) and not torch.any(torch.isnan(s[0, :64]))
    sl = d["sl"].clone()
    sl[1] = 10 ** 6  # clamped to the block table's 4 pages, whose unused entries are -1
    mla.index_scores(d["q_idx"], d["idx"], d["bt"], sl)
    torch.cuda.synchronize()
    assert mla.get_device_status()[1] == mla.DEV_BAD_SEQ_LEN | mla.DEV_BAD_BLOCK_TABLE
    sl[1] = -5
    si, _, _, sn = mla.topk_gather(torch.zeros(2, 256, device=DEV), sl, d["pool"], d["bt"], 16)
    torch.cuda.synchronize()
    assert mla.get_device_status()[1] == mla.DEV_BAD_SEQ_LEN
    assert int(sn[1]) == 0 and torch.all(si[1] == -1)


def test_full_size_128k_sampled():
    name = "sparse_b8_l128k_k512"
    sc = workloads.make_sparse_workload(name, device=DEV)
    c = sc.case
    bt, sl = c.block_table.to(DEV), c.seq_lens.to(DEV)
    o, lse, si = mla.decode_sparse(c.q_abs, sc.q_idx, c.pool, sc.idx_pool, bt, sl, sc.k)
    scores = mla.index_scores(sc.q_idx, sc.idx_pool, bt, sl)
    torch.cuda.synchronize()
    assert mla.get_device_status() == (0, 0)
    s = scores.cpu().numpy()
    sel = si.cpu().numpy()
    # scores of two whole sequences against the oracle
    for b in (0, 5):
        q = _np(sc.q_idx[b:b + 1])
        pages = c.block_table[b:b + 1]
        ip = sc.idx_pool.index_select(0, pages[0].to(DEV).long()).float().cpu().numpy()
        ref = oracle.index_scores(q, ip, np.arange(pages.shape[1], dtype=np.int32)[None], c.seq_lens[b:b + 1].numpy())
        bound = (np.abs(ip).reshape(-1, sc.d_idx) @ np.abs(q[0])) * sc.d_idx * 2.0 ** -24 + 1e-30
        assert np.all(np.abs(s[b] - ref[0]) <= bound)
    # the selection of every sequence, exactly
    for b in range(c.B):
        assert np.array_equal(sel[b], oracle.topk_row(s[b].astype(np.float64), sc.k)), b
    # the decode of two sequences over their selected rows (gathered on the device, decoded by the oracle)
    for b in (1, 6):
        t = torch.as_tensor(sel[b], device=DEV).long()
        rows = c.pool[bt[b, t // 64].long(), t % 64].float().cpu().numpy()
        comp = rows.reshape(sc.k // 64, 64, workloads.D)
        o_ref, l_ref = oracle.decode_absorbed(c.q_abs[b:b + 1].float().cpu().numpy(), comp,
                                              np.arange(sc.k // 64, dtype=np.int32)[None],
                                              np.array([sc.k], np.int32), c.scale)
        extra = _p_rounding_bound(c.q_abs[b, 0].double().cpu().numpy(), rows.astype(np.float64), c.scale)
        _check_sparse_out(o[b:b + 1], o_ref, extra[None, None])
        check_lse(lse[b:b + 1], l_ref)
