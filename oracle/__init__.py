"""MLA oracle: slow, obviously-correct fp64 CPU reference.

TEST INFRASTRUCTURE ONLY.  Imported by ``tests/``, by ``__graft_entry__.smoke()``
and by the ``cpu_baseline`` / ``--impl reference`` legs of ``bench.py``; the
CUDA library and its Python binding never import, load or call anything here.

The arithmetic lives in ``mla_oracle.c`` (compiled to ``liboracle.so`` by
:func:`build`); this module only marshals numpy arrays.  Inputs are converted
to float32 (bf16 values are exact in float32); every result is float64.

Sources (see the C file for the passage each function follows):
  * "DeepSeek-V2" explainer, Steps 5-8 (latent cache, absorption, decoupled
    RoPE, 576-number cache row; the cache write c = W^DKV h of equation 9 and
    the rotated key k^R of Step 7);
  * DeepSeek-V2 paper breakdown, "How It Works" (latent c_t cached, up-projected
    to K and V, separate RoPE key kept beside it);
  * the DeepSeek page, "KV cache compression" (token-level compression) and
    "KV cache data movement minimization" (the indexer: index scores over every
    cached token, top-k, attention over the selected tokens only).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mla_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None

_f32p = np.ctypeslib.ndpointer(dtype=np.float32, flags="C_CONTIGUOUS")
_f64p = np.ctypeslib.ndpointer(dtype=np.float64, flags="C_CONTIGUOUS")
_i32p = np.ctypeslib.ndpointer(dtype=np.int32, flags="C_CONTIGUOUS")
_i64p = np.ctypeslib.ndpointer(dtype=np.int64, flags="C_CONTIGUOUS")


def build(force: bool = False) -> str:
    """Compile liboracle.so with gcc (fp64, no fast-math, no FMA contraction)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-ffp-contract=off",
               "-fno-fast-math", "-o", _LIB_PATH, _SRC, "-lm"]
        subprocess.check_call(cmd)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        lib.oracle_absorb_q.argtypes = [_f32p, _f32p, _f32p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                        ctypes.c_int, ctypes.c_int, _f64p]
        lib.oracle_up_proj.argtypes = [_f64p, _f32p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                       ctypes.c_int, _f64p]
        lib.oracle_decode_absorbed.argtypes = [ctypes.c_void_p, ctypes.c_void_p, _f32p, _i32p, _i32p,
                                               ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                               ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_double,
                                               ctypes.c_int, ctypes.c_int, _f64p, _f64p]
        lib.oracle_decode_naive.argtypes = [_f32p, _f32p, _f32p, _f32p, _f32p, _i32p, _i32p,
                                            ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                            ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                            ctypes.c_double, ctypes.c_int, ctypes.c_int, _f64p, _f64p]
        lib.oracle_combine.argtypes = [_f64p, _f64p, ctypes.c_int, ctypes.c_long, ctypes.c_int,
                                       _f64p, _f64p]
        lib.oracle_rope.argtypes = [_f64p, ctypes.c_double, ctypes.c_int, ctypes.c_double, _f64p]
        lib.oracle_cache_append.argtypes = [_f32p, _f32p, _f32p, _i32p, _i32p, ctypes.c_int, ctypes.c_int,
                                            ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                            ctypes.c_int, ctypes.c_int, ctypes.c_double, _f64p, _i64p]
        lib.oracle_compress.argtypes = [_f64p, _f64p, ctypes.c_long, ctypes.c_int, ctypes.c_int, _f64p]
        lib.oracle_cache_append_compressed.argtypes = [_f32p, _f32p, _f32p, _f32p, _i32p, _i32p, ctypes.c_int,
                                                       ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                       ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                       ctypes.c_double, _f64p, _i64p]
        lib.oracle_index_scores.argtypes = [_f32p, _f32p, _i32p, _i32p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                            ctypes.c_int, ctypes.c_long, _f64p]
        lib.oracle_topk_row.argtypes = [_f64p, ctypes.c_long, ctypes.c_long,
                                        np.ctypeslib.ndpointer(dtype=np.int64, flags="C_CONTIGUOUS")]
        lib.oracle_topk_row.restype = ctypes.c_long
        _u8p = np.ctypeslib.ndpointer(dtype=np.uint8, flags="C_CONTIGUOUS")
        lib.oracle_e4m3_value.argtypes = [ctypes.c_uint8]
        lib.oracle_e4m3_value.restype = ctypes.c_double
        lib.oracle_index_scores_e4m3.argtypes = [_f32p, _u8p, _f32p, _i32p, _i32p, ctypes.c_int, ctypes.c_int,
                                                 ctypes.c_int, ctypes.c_int, ctypes.c_long, _f64p]
        lib.oracle_index_scores_e4m3.restype = None
        for fn in ("oracle_absorb_q", "oracle_up_proj", "oracle_decode_absorbed", "oracle_decode_naive",
                   "oracle_combine", "oracle_rope", "oracle_cache_append", "oracle_compress",
                   "oracle_cache_append_compressed", "oracle_index_scores"):
            getattr(lib, fn).restype = None
        _lib = lib
    return _lib


def _f32(x) -> np.ndarray:
    if hasattr(x, "detach"):  # torch tensor (bf16 -> f32 is exact)
        x = x.detach().to("cpu").float().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float32))


def _f64(x) -> np.ndarray:
    if hasattr(x, "detach"):
        x = x.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _i32(x) -> np.ndarray:
    if hasattr(x, "detach"):
        x = x.detach().to("cpu").numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.int32))


def default_threads() -> int:
    return len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)


def absorb_q(q_nope, q_rope, w_uk) -> np.ndarray:
    """q_abs[n,h] = [W_UK[h]^T q_nope[n,h] | q_rope[n,h]]  (Step 6 absorption, Step 7 RoPE part).

    q_nope [..., H, d_h], q_rope [..., H, d_r], w_uk [H, d_h, d_c] -> [..., H, d_c + d_r] float64.
    """
    qn, qr, w = _f32(q_nope), _f32(q_rope), _f32(w_uk)
    H, d_h, d_c = w.shape
    lead = qn.shape[:-2]
    N = int(np.prod(lead)) if lead else 1
    d_r = qr.shape[-1]
    out = np.zeros(lead + (H, d_c + d_r), dtype=np.float64)
    if qr.size == 0:
        qr = np.zeros(1, dtype=np.float32)
    _load().oracle_absorb_q(qn, qr, w, N, H, d_h, d_c, d_r, out)
    return out


def up_proj(o_lat, w_uv) -> np.ndarray:
    """out[n,h] = W_UV[h] o_lat[n,h]  (Step 5 value regeneration, applied after attention)."""
    o, w = _f64(o_lat), _f32(w_uv)
    H, d_h, d_c = w.shape
    lead = o.shape[:-2]
    N = int(np.prod(lead)) if lead else 1
    out = np.zeros(lead + (H, d_h), dtype=np.float64)
    _load().oracle_up_proj(o, w, N, H, d_h, d_c, out)
    return out


def decode_absorbed(q_abs, pool, block_table, seq_lens, scale: float, causal: bool = False,
                    d_c: int = 512, nthreads: int | None = None):
    """Absorbed decode over a paged latent cache.

    q_abs [B, Tq, H, D] (float32-exact or float64), pool [P, page, D], block_table [B, max_pages],
    seq_lens [B].  Returns (o_lat [B,Tq,H,d_c] float64, lse [B,Tq,H] float64).
    """
    pl = _f32(pool)
    bt, sl = _i32(block_table), _i32(seq_lens)
    if hasattr(q_abs, "detach"):
        q_abs = q_abs.detach().to("cpu")
        q_abs = q_abs.double().numpy() if str(q_abs.dtype) == "torch.float64" else q_abs.float().numpy()
    if np.asarray(q_abs).dtype != np.float64:
        q32, q64 = _f32(q_abs), None
        q = q32
    else:
        q32, q64 = None, _f64(q_abs)
        q = q64
    B, Tq, H, D = q.shape
    page = pl.shape[1]
    d_r = D - d_c
    max_pages = bt.shape[1]
    o = np.zeros((B, Tq, H, d_c), dtype=np.float64)
    lse = np.zeros((B, Tq, H), dtype=np.float64)
    if nthreads is None:
        nthreads = default_threads()
    _load().oracle_decode_absorbed(
        q32.ctypes.data if q32 is not None else None,
        q64.ctypes.data if q64 is not None else None,
        pl, bt, sl, B, Tq, H, d_c, d_r, page, max_pages, float(scale), int(bool(causal)),
        int(nthreads), o, lse)
    return o, lse


def decode_naive(q_nope, q_rope, w_uk, w_uv, pool, block_table, seq_lens, scale: float,
                 causal: bool = False, nthreads: int | None = None):
    """Naive MHA over per-head keys/values rebuilt from the latent cache.

    q_nope [B,Tq,H,d_h], q_rope [B,Tq,H,d_r], w_uk/w_uv [H,d_h,d_c].
    Returns (out [B,Tq,H,d_h] float64, lse [B,Tq,H] float64).
    """
    qn, qr, wk, wv, pl = _f32(q_nope), _f32(q_rope), _f32(w_uk), _f32(w_uv), _f32(pool)
    bt, sl = _i32(block_table), _i32(seq_lens)
    B, Tq, H, d_h = qn.shape
    d_r = qr.shape[-1]
    d_c = wk.shape[2]
    page = pl.shape[1]
    max_pages = bt.shape[1]
    out = np.zeros((B, Tq, H, d_h), dtype=np.float64)
    lse = np.zeros((B, Tq, H), dtype=np.float64)
    if qr.size == 0:
        qr = np.zeros(1, dtype=np.float32)
    if nthreads is None:
        nthreads = default_threads()
    _load().oracle_decode_naive(qn, qr, wk, wv, pl, bt, sl, B, Tq, H, d_h, d_c, d_r, page,
                                max_pages, float(scale), int(bool(causal)), int(nthreads), out, lse)
    return out, lse


def combine(o_parts, lse_parts):
    """Merge attention results over disjoint token sets.

    o_parts [R, ..., d], lse_parts [R, ...] -> (o [..., d], lse [...]) float64.
    """
    o = _f64(o_parts)
    l = _f64(lse_parts)
    R = o.shape[0]
    d = o.shape[-1]
    M = int(np.prod(o.shape[1:-1])) if o.ndim > 2 else 1
    out = np.zeros(o.shape[1:], dtype=np.float64)
    lse = np.zeros(l.shape[1:], dtype=np.float64)
    _load().oracle_combine(o, l, R, M, d, out, lse)
    return out, lse


def rope(x, pos: float, base: float = 10000.0) -> np.ndarray:
    """Rotate the pairs (2i, 2i+1) of x [d] by pos * base^(-2i/d)  (Step 7, decoupled RoPE key)."""
    v = _f64(x).reshape(-1)
    out = np.zeros_like(v)
    _load().oracle_rope(v, float(pos), int(v.size), float(base), out)
    return out


def cache_append(h, w_dkv, w_kr, block_table, seq_lens, q_len: int, num_pages: int, page: int = 64,
                 rope_base: float = 10000.0):
    """Cache rows of new tokens and the pool rows they go to (Step 5 eq. 9 and Step 7).

    h [B*Tq, d_model] (or [B, Tq, d_model]), w_dkv [d_c, d_model], w_kr [d_r, d_model],
    block_table [B, max_pages], seq_lens [B] (already counting the Tq new tokens).
    Returns (rows [B*Tq, d_c + d_r] float64, slot [B*Tq] int64; -1 for a token with no valid slot).
    """
    x = _f32(h)
    wd, wr = _f32(w_dkv), _f32(w_kr)
    bt, sl = _i32(block_table), _i32(seq_lens)
    B, max_pages = bt.shape
    d_c, d_model = wd.shape
    d_r = wr.shape[0]
    x = x.reshape(B * q_len, d_model)
    rows = np.zeros((B * q_len, d_c + d_r), dtype=np.float64)
    slot = np.zeros(B * q_len, dtype=np.int64)
    if wr.size == 0:
        wr = np.zeros(1, dtype=np.float32)
    _load().oracle_cache_append(x, wd, wr, bt, sl, B, int(q_len), d_model, d_c, d_r, int(page), max_pages,
                                int(num_pages), float(rope_base), rows, slot)
    return rows, slot


def compress(rows, z, m: int) -> np.ndarray:
    """Merge blocks of m consecutive rows: out[g, k] = sum_i softmax_i(z[g*m+i, k]) rows[g*m+i, k]
    (the token-level compression of the DeepSeek page's "KV cache compression" section)."""
    r, zz = _f64(rows), _f64(z)
    n, D = r.shape
    assert zz.shape == r.shape and n % m == 0
    out = np.zeros((n // m, D), dtype=np.float64)
    _load().oracle_compress(r, zz, n // m, int(m), D, out)
    return out


def cache_append_compressed(h, w_dkv, w_kr, w_z, block_table, seq_lens, n_blocks: int, m: int, num_pages: int,
                            page: int = 64, rope_base: float = 10000.0):
    """Compressed cache write: n_blocks new compressed rows per sequence, each the merge of m new
    tokens' rows ([W^DKV h | RoPE_pos(W^KR h)], weights softmax over the m tokens of W^Z h, per
    component).  seq_lens counts compressed rows including the new ones.  h [B * n_blocks * m,
    d_model].  Returns (rows [B * n_blocks, D] float64, slot [B * n_blocks] int64)."""
    x = _f32(h)
    wd, wr, wz = _f32(w_dkv), _f32(w_kr), _f32(w_z)
    bt, sl = _i32(block_table), _i32(seq_lens)
    B, max_pages = bt.shape
    d_c, d_model = wd.shape
    d_r = wr.shape[0]
    x = x.reshape(B * n_blocks * m, d_model)
    rows = np.zeros((B * n_blocks, d_c + d_r), dtype=np.float64)
    slot = np.zeros(B * n_blocks, dtype=np.int64)
    _load().oracle_cache_append_compressed(x, wd, wr, wz, bt, sl, B, int(n_blocks), int(m), d_model, d_c, d_r,
                                           int(page), max_pages, int(num_pages), float(rope_base), rows, slot)
    return rows, slot


def index_scores(q_idx, idx_pool, block_table, seq_lens, max_len: int | None = None) -> np.ndarray:
    """s[b, t] = q_idx[b] . k_idx(b, t) for t < seq_lens[b] (NaN elsewhere): the indexer's
    scores over every cached token (the DeepSeek page's "indexer" method).  q_idx [B, d_idx],
    idx_pool [P, page, d_idx]."""
    q, ip = _f32(q_idx), _f32(idx_pool)
    bt, sl = _i32(block_table), _i32(seq_lens)
    B, d_idx = q.shape
    page = ip.shape[1]
    if max_len is None:
        max_len = int(sl.max()) if sl.size else 0
    out = np.full((B, max(1, max_len)), np.nan, dtype=np.float64)
    _load().oracle_index_scores(q, ip, bt, sl, B, d_idx, page, bt.shape[1], max(1, max_len), out)
    return out[:, :max_len]


def topk_row(scores, k: int) -> np.ndarray:
    """Indices of the k largest scores (ties: the lower index), ascending; all if k >= n."""
    s = _f64(scores).reshape(-1)
    out = np.zeros(max(1, min(k, s.size)), dtype=np.int64)
    n = _load().oracle_topk_row(s, s.size, int(k), out)
    return out[:n]


def decode_sparse(q_abs, q_idx, pool, idx_pool, block_table, seq_lens, k: int, scale: float, d_c: int = 512):
    """Top-k sparse decode (one query token per sequence): index scores over every cached token,
    the k best (ties: lower index), then the absorbed decode over those tokens only.
    Returns (o_lat [B, 1, H, d_c], lse [B, 1, H], selected: list of index arrays)."""
    q = _f64(q_abs)
    B = q.shape[0]
    pl = _f32(pool)
    bt, sl = _i32(block_table), _i32(seq_lens)
    page, D = pl.shape[1], pl.shape[2]
    sc = index_scores(q_idx, idx_pool, bt, sl)
    sel, rows = [], []
    for b in range(B):
        idx = topk_row(sc[b, :int(sl[b])], k) if sl[b] > 0 else np.zeros(0, dtype=np.int64)
        sel.append(idx)
        rows.append(np.stack([pl[bt[b, t // page], t % page] for t in idx]) if idx.size else np.zeros((0, D), np.float32))
    kmax = max(1, max(r.shape[0] for r in rows))
    n_pages = (kmax + page - 1) // page
    comp = np.zeros((B * n_pages, page, D), dtype=np.float32)
    cbt = np.arange(B * n_pages, dtype=np.int32).reshape(B, n_pages)
    lens = np.array([r.shape[0] for r in rows], dtype=np.int32)
    for b in range(B):
        comp.reshape(B, n_pages * page, D)[b, :rows[b].shape[0]] = rows[b]
    o, lse = decode_absorbed(q, comp, cbt, lens, scale, causal=False, d_c=d_c)
    return o, lse, sel


def e4m3_value(code: int) -> float:
    """The value of one FP8 E4M3 code (1 sign, 4 exponent bits with bias 7, 3 mantissa bits,
    subnormals at exponent 0, S.1111.111 NaN, no infinity)."""
    return float(_load().oracle_e4m3_value(int(code) & 0xFF))


def index_scores_e4m3(q_idx, idx_codes, idx_scale, block_table, seq_lens, max_len: int | None = None) -> np.ndarray:
    """s[b, t] = scale(b, t) * q_idx[b] . value(codes(b, t)) for t < seq_lens[b] (NaN elsewhere).
    idx_codes [P, page, d_idx] uint8 (E4M3 codes), idx_scale [P, page] float32."""
    q = _f32(q_idx)
    codes = np.ascontiguousarray(np.asarray(idx_codes.cpu() if hasattr(idx_codes, "cpu") else idx_codes,
                                            dtype=np.uint8))
    sc = _f32(idx_scale)
    bt, sl = _i32(block_table), _i32(seq_lens)
    B, d_idx = q.shape
    page = codes.shape[1]
    if max_len is None:
        max_len = int(sl.max()) if sl.size else 0
    out = np.full((B, max(1, max_len)), np.nan, dtype=np.float64)
    _load().oracle_index_scores_e4m3(q, codes, sc, bt, sl, B, d_idx, page, bt.shape[1], max(1, max_len), out)
    return out[:, :max_len]
