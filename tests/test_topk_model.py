"""CPU model of the top-k kernel's selection (topk_gather_kernel), step by step with the kernel's
own constants, checked against the oracle's top-k (the k largest scores, ties to the lower
position, NaN below every number).

The model keeps the kernel's structure, so a slip in the structure fails here without a GPU:
  * 8 CTAs per sequence, each a contiguous slice (a multiple of 4 positions), 32 warps per CTA,
    each a sub-slice (a multiple of 128 positions);
  * order-keeping 32-bit keys (-0 -> +0, NaN -> 0);
  * radix select one byte per pass from the top, the cluster's histograms summed, per-rank counts
    of keys above the chosen bins accumulated from the histograms each CTA reads;
  * after the second pass, per-warp lists of positions whose top byte is at least the first
    pass's chosen byte (at most 128 per warp, else the CTA scans its whole slice), and the
    exchange of the keys that carry the 16-bit prefix (at most 64 per CTA, else all CTAs run the
    third and fourth passes);
  * output offsets from the per-rank counts (equal keys to the lowest ranks first), then per-warp
    compaction in position order.
CPU only."""
import numpy as np
import pytest

import oracle

CLUSTER, WARPS, LIST_CAP, CAND_CAP = 8, 32, 128, 64


def _key(f, keep_signed_zero=False):
    u = int(np.float32(f).view(np.uint32))
    if u == 0x80000000 and not keep_signed_zero:
        u = 0
    if (u & 0x7FFFFFFF) > 0x7F800000:
        return 0
    return (~u & 0xFFFFFFFF) if (u & 0x80000000) else (u | 0x80000000)


def _pick_bin(tot, need):
    """The bin holding the need-th largest key: (bin, keys in the bins above it)."""
    incl = 0
    for v in range(255, -1, -1):
        above = incl
        incl += tot[v]
        if above < need <= incl:
            return v, above
    raise AssertionError("no bin holds the need-th key")


def model_topk(scores, k, stats=None, keep_signed_zero=False):
    """The kernel's selection; keep_signed_zero plants a mistake (-0 ranked below +0 instead of
    tying with it)."""
    L = len(scores)
    keys = [_key(x, keep_signed_zero) for x in scores]
    if k >= L:
        return list(range(L))
    chunk = ((L + CLUSTER - 1) // CLUSTER + 3) & ~3
    slices = []
    for r in range(CLUSTER):
        lo = min(L, r * chunk)
        slices.append((lo, min(L, lo + chunk)))

    def warp_span(lo, hi, w):
        wspan = (((hi - lo) + WARPS - 1) // WARPS + 127) & ~127
        wlo = min(hi, lo + w * wspan)
        return wlo, min(hi, wlo + wspan)

    prefix, mask, need = 0, 0, k
    rank_gt = [0] * CLUSTER
    rank_eq = [0] * CLUSTER
    lists = None
    exchanged = False
    for p in range(4):
        shift = 24 - 8 * p
        hist = [[0] * 256 for _ in range(CLUSTER)]
        for r, (lo, hi) in enumerate(slices):
            for e in range(lo, hi):
                if keys[e] & mask == prefix:
                    hist[r][(keys[e] >> shift) & 0xFF] += 1
        if p == 1:
            v0 = prefix >> 24
            lists = []
            for r, (lo, hi) in enumerate(slices):
                wl = [[e for e in range(*warp_span(lo, hi, w)) if (keys[e] >> 24) >= v0] for w in range(WARPS)]
                lists.append(None if any(len(x) > LIST_CAP for x in wl) else wl)
        tot = [sum(hist[r][b] for r in range(CLUSTER)) for b in range(256)]
        v, above = _pick_bin(tot, need)
        need -= above
        prefix |= v << shift
        mask |= 0xFF << shift
        for r in range(CLUSTER):
            rank_gt[r] += sum(hist[r][b] for b in range(v + 1, 256))
            if p == 3:
                rank_eq[r] = hist[r][v]
        if p == 1:
            # the exchange of the keys carrying the 16-bit prefix
            cands = []
            for r, (lo, hi) in enumerate(slices):
                src = [e for wl in lists[r] for e in wl] if lists[r] is not None else range(lo, hi)
                cands.append([keys[e] for e in src if keys[e] & mask == prefix])
            if all(len(c) <= CAND_CAP for c in cands):
                allk = [(key, r) for r, c in enumerate(cands) for key in c]
                T = None
                for key, _ in allk:
                    gt = sum(o > key for o, _ in allk)
                    ge = sum(o >= key for o, _ in allk)
                    if gt < need <= ge:
                        T, gtT = key, gt
                for key, r in allk:
                    if key > T:
                        rank_gt[r] += 1
                    elif key == T:
                        rank_eq[r] += 1
                need -= gtT
                prefix, mask = T, 0xFFFFFFFF
                exchanged = True
                break
    if stats is not None:
        stats["exchanged"] = stats.get("exchanged", 0) + int(exchanged)
        stats["list_overflow"] = stats.get("list_overflow", 0) + sum(x is None for x in lists)
    out = [None] * k
    for r, (lo, hi) in enumerate(slices):
        out_off = eq_before = 0
        for q in range(r):
            out_off += rank_gt[q] + (0 if eq_before >= need else min(rank_eq[q], need - eq_before))
            eq_before += rank_eq[q]
        use_lists = lists[r] is not None
        counts = []
        for w in range(WARPS):
            wl = lists[r][w] if use_lists else list(range(*warp_span(lo, hi, w)))
            counts.append((wl, sum(keys[e] > prefix for e in wl), sum(keys[e] == prefix for e in wl)))
        n_out, n_eq = out_off, eq_before
        for wl, gt, eq in counts:
            pos, ne = n_out, n_eq
            for e in wl:
                if keys[e] > prefix:
                    out[pos] = e
                    pos += 1
                elif keys[e] == prefix:
                    if ne < need:
                        out[pos] = e
                        pos += 1
                    ne += 1
            n_out += gt + (0 if n_eq >= need else min(eq, need - n_eq))
            n_eq += eq
            assert pos == n_out
    assert None not in out
    return out


def _cases():
    rng = np.random.default_rng(7)
    for trial in range(24):
        L = int(rng.integers(1, 2500))
        mode = trial % 4
        if mode == 0:
            s = rng.standard_normal(L).astype(np.float32)
        elif mode == 1:
            s = rng.integers(-3, 4, L).astype(np.float32)  # tie-heavy: the exchange overflows
        elif mode == 2:
            s = rng.integers(-2, 3, L).astype(np.float32)
            s[rng.random(L) < 0.1] = -np.inf
            s[rng.random(L) < 0.1] = np.nan
            s[(s == 0) & (rng.random(L) < 0.5)] = -0.0
        else:
            s = (rng.standard_normal(L) * 1e-3).astype(np.float32)  # one exponent: lists fill up
        for k in sorted({1, 2, max(1, L // 7), max(1, L // 2), max(1, L - 1), L, L + 3}):
            yield s, k


def test_model_matches_the_oracle():
    stats = {}
    n = 0
    for s, k in _cases():
        got = model_topk(s, k, stats)
        want = list(oracle.topk_row(s.astype(np.float64), k))
        assert got == want, (len(s), k)
        n += 1
    assert n > 100
    assert stats["exchanged"] > 0  # the exchange was taken, and (the tie-heavy rows) given up


@pytest.mark.parametrize("k", [100, 5000])
def test_model_with_overflowing_warp_lists(k):
    """40000 scores of one binade: a warp's 160 positions nearly all share the first byte, so the
    lists overflow and the CTAs scan their whole slices; the result still matches."""
    rng = np.random.default_rng(k)
    s = (1.0 + rng.random(40000)).astype(np.float32)
    stats = {}
    assert model_topk(s, k, stats) == list(oracle.topk_row(s.astype(np.float64), k))
    assert stats["list_overflow"] > 0


def test_model_exchange_fallback_on_ties():
    """Thousands of equal scores: every CTA holds more than 64 keys with the 16-bit prefix, so the
    exchange gives way to the full passes, and the picks are still the lowest positions."""
    s = np.zeros(5000, np.float32)
    s[::3] = 1.0
    stats = {}
    got = model_topk(s, 700, stats)
    assert stats.get("exchanged", 0) == 0
    assert got == list(oracle.topk_row(s.astype(np.float64), 700))
    assert got == list(range(0, 2100, 3))


def test_a_planted_key_mistake_is_caught():
    """Keys that keep -0 below +0 (the kernel maps -0 to +0 so that they tie, as the oracle's
    comparison does) pick different positions among zeros of both signs."""
    rng = np.random.default_rng(3)
    s = np.where(rng.random(3000) < 0.5, -0.0, 0.0).astype(np.float32)
    s[rng.random(3000) < 0.2] = 1.0
    for k in (700, 1500):
        want = list(oracle.topk_row(s.astype(np.float64), k))
        assert model_topk(s, k) == want
        assert model_topk(s, k, keep_signed_zero=True) != want
