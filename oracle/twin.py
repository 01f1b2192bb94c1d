"""Pure-Python brute-force twin of the MLA decode and cache write, for tiny shapes only.

TEST INFRASTRUCTURE ONLY (imported by tests).  Written separately from
``mla_oracle.c`` and structured differently on purpose, so that a slip in one
is unlikely to be repeated in the other:

  * it works on nested Python lists, one (sequence, query token, head) at a
    time, gathering the visible cache rows first;
  * it always takes the *naive* route of the "DeepSeek-V2" explainer, Step 5
    (rebuild each head's key k = W^UK c and value v = W^UV c) plus the
    decoupled RoPE channel of Step 7 (the head's q^R against the token's
    shared k^R), and only then applies the softmax;
  * the softmax weight of token j is computed as 1 / sum_k exp(s_k - s_j),
    and the log-sum-exp with ``math.fsum``.

It has no paged layout of its own beyond resolving the block table to a row
list, and no absorbed form: agreement of the C oracle's absorbed form with
this twin therefore checks the Step 6 associativity independently.

The cache write (Step 5's c = W^DKV h, Step 7's rotated k^R) turns each RoPE
pair as a complex number times a unit phasor, where the C oracle writes out
the cosine/sine rotation; and it finds a token's pool row with ``divmod``.
"""
from __future__ import annotations

import cmath
import math
from typing import List, Sequence


def _matvec(W: Sequence[Sequence[float]], x: Sequence[float]) -> List[float]:
    return [math.fsum(w * v for w, v in zip(row, x)) for row in W]


def _dot(a: Sequence[float], b: Sequence[float]) -> float:
    return math.fsum(x * y for x, y in zip(a, b))


def gather_rows(pool, block_table_row, n_tokens: int, page: int):
    """Logical token j lives in physical page block_table_row[j // page], slot j % page."""
    return [pool[block_table_row[j // page]][j % page] for j in range(n_tokens)]


def attend_naive(q_nope, q_rope, W_uk, W_uv, rows, d_c: int, scale: float):
    """One head, one query: returns (out [d_h], lse) or ([0]*d_h, -inf) for no rows."""
    d_h = len(W_uv)
    if not rows:
        return [0.0] * d_h, -math.inf
    scores = []
    values = []
    for row in rows:
        c, k_r = list(row[:d_c]), list(row[d_c:])
        k = _matvec(W_uk, c)                 # content key of this head
        v = _matvec(W_uv, c)                 # value of this head
        scores.append(scale * (_dot(q_nope, k) + _dot(q_rope, k_r)))
        values.append(v)
    weights = [1.0 / math.fsum(math.exp(sk - sj) for sk in scores) for sj in scores]
    out = [math.fsum(w * v[d] for w, v in zip(weights, values)) for d in range(d_h)]
    top = max(scores)
    lse = top + math.log(math.fsum(math.exp(s - top) for s in scores))
    return out, lse


def attend_latent(q_abs, rows, d_c: int, scale: float):
    """Direct latent-space attention with an already absorbed query (one head, one query).

    Used only where the query is given in absorbed form (no weights exist):
    s_j = scale * q_abs . row_j, o = sum_j p_j row_j[:d_c].
    """
    if not rows:
        return [0.0] * d_c, -math.inf
    scores = [scale * _dot(q_abs, row) for row in rows]
    weights = [1.0 / math.fsum(math.exp(sk - sj) for sk in scores) for sj in scores]
    o = [math.fsum(w * row[i] for w, row in zip(weights, rows)) for i in range(d_c)]
    top = max(scores)
    lse = top + math.log(math.fsum(math.exp(s - top) for s in scores))
    return o, lse


def decode(q_nope, q_rope, W_uk, W_uv, pool, block_table, seq_lens, scale, causal=False):
    """Brute force over nested lists.

    q_nope[b][t][h][d_h], q_rope[b][t][h][d_r], W_uk[h][d_h][d_c], W_uv[h][d_h][d_c],
    pool[page_id][slot][d_c + d_r], block_table[b][p], seq_lens[b].
    Returns (out[b][t][h][d_h], lse[b][t][h]).
    """
    page = len(pool[0])
    d_c = len(W_uk[0][0])
    out, lse = [], []
    for b in range(len(q_nope)):
        Tq = len(q_nope[b])
        ob, lb = [], []
        for t in range(Tq):
            n = seq_lens[b] if not causal else max(0, seq_lens[b] - (Tq - 1 - t))
            rows = gather_rows(pool, block_table[b], n, page)
            ot, lt = [], []
            for h in range(len(q_nope[b][t])):
                o, l = attend_naive(q_nope[b][t][h], q_rope[b][t][h], W_uk[h], W_uv[h], rows, d_c, scale)
                ot.append(o)
                lt.append(l)
            ob.append(ot)
            lb.append(lt)
        out.append(ob)
        lse.append(lb)
    return out, lse


def rope_phasor(x: Sequence[float], pos: float, base: float) -> List[float]:
    """Step 7's rotation written with complex numbers: pair i is the complex number
    x[2i] + 1j * x[2i+1], multiplied by the unit phasor exp(1j * pos * base**(-2i/d))."""
    d = len(x)
    out: List[float] = []
    for i in range(d // 2):
        z = complex(x[2 * i], x[2 * i + 1]) * cmath.exp(1j * pos * base ** (-(2.0 * i) / d))
        out += [z.real, z.imag]
    return out


def cache_rows(h, W_dkv, W_kr, block_table, seq_lens, q_len: int, page: int, num_pages: int, base: float):
    """Brute-force cache write (Step 5 eq. 9 and Step 7), one token at a time over nested lists.

    h[b][t][d_model]; returns {pool row index: row values} for every token that has a valid slot.
    A token's position is its index in the sequence once the q_len new tokens are counted.
    """
    written = {}
    for b, toks in enumerate(h):
        first = seq_lens[b] - q_len
        for t, x in enumerate(toks):
            pos = first + t
            logical_page, offset = divmod(pos, page) if pos >= 0 else (-1, 0)
            if pos < 0 or logical_page >= len(block_table[b]):
                continue
            phys = block_table[b][logical_page]
            if not 0 <= phys < num_pages:
                continue
            written[phys * page + offset] = _matvec(W_dkv, x) + rope_phasor(_matvec(W_kr, x), pos, base)
    return written


def compress_block(rows, z):
    """One merged row of a block, component by component: each token's weight is
    1 / sum_j exp(z_j - z_i) (the softmax over the block's tokens, written as a ratio), and the
    merged value is math.fsum of weight times value."""
    D = len(rows[0])
    out = []
    for k in range(D):
        col = [r[k] for r in rows]
        zc = [zz[k] for zz in z]
        w = [1.0 / math.fsum(math.exp(zj - zi) for zj in zc) for zi in zc]
        out.append(math.fsum(wi * v for wi, v in zip(w, col)))
    return out
