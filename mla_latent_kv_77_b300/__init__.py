"""Python binding of the B300 MLA decode library (``libmla.so``, C ABI in include/mla.h).

Argument marshalling only: every numeric step runs in the library's CUDA kernels.
PyTorch is used for device memory and streams.  If ``libmla.so`` has not been
built the calls raise :class:`MLAError` -- there is no fallback of any kind.

Method: weight-absorbed Multi-head Latent Attention decode ("DeepSeek-V2"
explainer, Part B Steps 5-8): the cache holds one 576-number row per token
([512-d latent c | 64-d rotated RoPE key k^R]); the query is absorbed through
W_UK into latent space, all 128 heads attend over the shared rows, and W_UV is
applied to the latent output afterwards.
"""
from __future__ import annotations

import ctypes
import enum
import math
import os
from typing import Optional, Tuple

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmla.so")

H = 128
D_C = 512
D_R = 64
D_H = 128
D = D_C + D_R
PAGE = 64
SCALE = 1.0 / math.sqrt(D_H + D_R)
ROPE_BASE = 10000.0  # RoPE frequency base of the cache write (pair i turns at ROPE_BASE^(-2i/64) per position)

# device status bits (MLA_DEV_* in mla.h)
DEV_BAD_BLOCK_TABLE = 0x1
DEV_BAD_SEQ_LEN = 0x2
DEV_WAIT_TIMEOUT = 0x4
DEV_PLAN_OVERFLOW = 0x8
DEV_SELECT_OVERFLOW = 0x10


class Status(enum.IntEnum):
    OK = 0
    INVALID_ARG = 1
    SHAPE = 2
    ALIGNMENT = 3
    WORKSPACE = 4
    UNSUPPORTED = 5
    CUDA = 6
    DEVICE_FAULT = 7


class MLAError(RuntimeError):
    def __init__(self, status, where: str = ""):
        self.status = Status(status) if status in Status._value2member_map_ else status
        super().__init__(f"{where}: {self.status!r}")


_lib = None

# (name, restype, argtypes) of every symbol declared in include/mla.h and include/mla_testing.h
_VP, _I, _F, _SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
EXPORTS = {
    "mla_absorb_q": (_I, [_VP, _VP, _VP, _VP, _I, _I, _VP]),
    "mla_decode_workspace_size": (_SZ, [_I, _I, _I]),
    "mla_decode": (_I, [_VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, _F, _I, _I, _VP, _VP, _VP, _SZ, _VP]),
    "mla_decode_static_scratch": (_I, [_VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, _F, _I, _I, _VP, _VP, _VP]),
    "mla_combine": (_I, [_VP, _VP, _I, _I, _VP, _VP, _VP]),
    "mla_up_proj": (_I, [_VP, _VP, _VP, _I, _I, _VP]),
    "mla_cache_append": (_I, [_VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, _F, _VP, _VP]),
    "mla_cache_append_compressed": (_I, [_VP, _VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, _I, _F, _VP, _VP]),
    "mla_index_scores": (_I, [_VP, _VP, _VP, _VP, _I, _I, _I, _I, _VP, _VP]),
    "mla_index_scores_e4m3": (_I, [_VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _VP, _VP]),
    "mla_topk_gather": (_I, [_VP, _VP, _VP, _VP, _I, _I, _I, _I, _VP, _VP, _VP, _VP, _VP]),
    "mla_decode_sparse_workspace_size": (_SZ, [_I, _I, _I]),
    "mla_decode_sparse": (_I, [_VP, _VP, _VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, _I, _F, _VP, _VP, _VP, _VP,
                               _SZ, _VP]),
    "mla_get_device_status": (_I, [_VP, ctypes.POINTER(ctypes.c_uint32)]),
    "mla_cache_bytes": (ctypes.c_uint64, [ctypes.c_int64, _I, _I, _I, _I]),
    "mla_status_string": (ctypes.c_char_p, [_I]),
    "mla_version": (_I, []),
    "mla_test_bounded_wait": (_I, [_I, _VP]),
    "mla_test_launch_count": (ctypes.c_uint64, []),
}


def lib():
    """Load libmla.so (raises MLAError if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise MLAError(Status.UNSUPPORTED, f"{LIB_PATH} missing: build it with __graft_entry__.build()")
        l = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in EXPORTS.items():
            fn = getattr(l, name)
            fn.restype = res
            fn.argtypes = args
        _lib = l
    return _lib


def _check(st: int, where: str):
    if st != 0:
        raise MLAError(st, where)


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _need(t, dtype, name):
    import torch
    if not isinstance(t, torch.Tensor) or t.dtype != dtype or not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name}: expected a contiguous CUDA tensor of {dtype}")


def status_string(code: int) -> str:
    return lib().mla_status_string(int(code)).decode()


def version() -> int:
    return int(lib().mla_version())


def cache_bytes(tokens: int, layers: int, d_c: int = D_C, d_r: int = D_R, bytes_per_elem: int = 2) -> int:
    return int(lib().mla_cache_bytes(tokens, layers, d_c, d_r, bytes_per_elem))


def decode_workspace_size(batch: int, q_len: int, num_splits: int = 0) -> int:
    return int(lib().mla_decode_workspace_size(batch, q_len, num_splits))


def absorb_q(q_nope, q_rope, w_uk, out=None, stream=None):
    """q_abs[n,h] = [W_UK[h]^T q_nope[n,h] | q_rope[n,h]] in bf16.  q_nope [..., 128, 128]."""
    import torch
    for t, n in ((q_nope, "q_nope"), (q_rope, "q_rope"), (w_uk, "w_uk")):
        _need(t, torch.bfloat16, n)
    lead = q_nope.shape[:-2]
    n_tok = int(math.prod(lead)) if lead else 1
    if out is None:
        out = torch.empty(*lead, q_nope.shape[-2], D, dtype=torch.bfloat16, device=q_nope.device)
    _need(out, torch.bfloat16, "out")
    _check(lib().mla_absorb_q(_ptr(q_nope), _ptr(q_rope), _ptr(w_uk), _ptr(out), n_tok, q_nope.shape[-2],
                              _stream(stream)), "mla_absorb_q")
    return out


def up_proj(o_lat, w_uv, out=None, stream=None):
    """out[n,h] = W_UV[h] o_lat[n,h] in bf16.  o_lat [..., 128, 512]."""
    import torch
    _need(o_lat, torch.bfloat16, "o_lat")
    _need(w_uv, torch.bfloat16, "w_uv")
    lead = o_lat.shape[:-2]
    n_tok = int(math.prod(lead)) if lead else 1
    if out is None:
        out = torch.empty(*lead, o_lat.shape[-2], D_H, dtype=torch.bfloat16, device=o_lat.device)
    _need(out, torch.bfloat16, "out")
    _check(lib().mla_up_proj(_ptr(o_lat), _ptr(w_uv), _ptr(out), n_tok, o_lat.shape[-2], _stream(stream)),
           "mla_up_proj")
    return out


def cache_append(h, w_dkv, w_kr, block_table, seq_lens, kv_pool, q_len: int = 1, rope_base: float = ROPE_BASE,
                 stream=None):
    """Write the cache rows [W^DKV h | RoPE_pos(W^KR h)] of new tokens into the paged pool, in place.

    h [B * q_len, d_model] (or [B, q_len, d_model]) bf16, w_dkv [512, d_model] bf16, w_kr [64, d_model]
    bf16, block_table [B, max_pages] int32, seq_lens [B] int32 counting the new tokens (token t of
    sequence b sits at position seq_lens[b] - q_len + t), kv_pool [P, 64, 576] bf16.  Returns kv_pool.
    """
    import torch
    for t, n in ((h, "h"), (w_dkv, "w_dkv"), (w_kr, "w_kr"), (kv_pool, "kv_pool")):
        _need(t, torch.bfloat16, n)
    _need(block_table, torch.int32, "block_table")
    _need(seq_lens, torch.int32, "seq_lens")
    B = block_table.shape[0]
    d_model = h.shape[-1]
    if h.numel() != B * q_len * d_model:
        raise ValueError(f"h: expected {B} x {q_len} tokens of width {d_model}")
    st = lib().mla_cache_append(_ptr(h), _ptr(w_dkv), _ptr(w_kr), _ptr(block_table), _ptr(seq_lens), B,
                                int(q_len), d_model, kv_pool.shape[0], block_table.shape[1], float(rope_base),
                                _ptr(kv_pool), _stream(stream))
    _check(st, "mla_cache_append")
    return kv_pool


def cache_append_compressed(h, w_dkv, w_kr, w_z, block_table, seq_lens, kv_pool, n_blocks: int = 1, m: int = 4,
                            rope_base: float = ROPE_BASE, stream=None):
    """Compressed cache write: n_blocks new rows per sequence, each the component-wise softmax
    merge (weights from W^Z h) of m new tokens' rows [W^DKV h | RoPE_pos(W^KR h)].

    h [B * n_blocks * m, d_model] bf16, w_z [576, d_model] bf16; seq_lens counts compressed rows
    (the new ones included).  Returns kv_pool."""
    import torch
    for t, n in ((h, "h"), (w_dkv, "w_dkv"), (w_kr, "w_kr"), (w_z, "w_z"), (kv_pool, "kv_pool")):
        _need(t, torch.bfloat16, n)
    _need(block_table, torch.int32, "block_table")
    _need(seq_lens, torch.int32, "seq_lens")
    B = block_table.shape[0]
    d_model = h.shape[-1]
    if h.numel() != B * n_blocks * m * d_model:
        raise ValueError(f"h: expected {B} x {n_blocks} x {m} tokens of width {d_model}")
    st = lib().mla_cache_append_compressed(_ptr(h), _ptr(w_dkv), _ptr(w_kr), _ptr(w_z), _ptr(block_table),
                                           _ptr(seq_lens), B, int(n_blocks), int(m), d_model, kv_pool.shape[0],
                                           block_table.shape[1], float(rope_base), _ptr(kv_pool), _stream(stream))
    _check(st, "mla_cache_append_compressed")
    return kv_pool


def decode(q_abs, kv_pool, block_table, seq_lens, scale: float = SCALE, causal: bool = False,
           num_splits: int = 0, o_lat=None, lse=None, workspace=None, stream=None) -> Tuple:
    """Absorbed MLA decode over a paged latent cache.

    q_abs [B, Tq, 128, 576] bf16, kv_pool [P, 64, 576] bf16, block_table [B, max_pages] int32,
    seq_lens [B] int32 (all on the GPU).  Returns (o_lat [B, Tq, 128, 512] bf16, lse [B, Tq, 128] f32).
    """
    import torch
    _need(q_abs, torch.bfloat16, "q_abs")
    _need(kv_pool, torch.bfloat16, "kv_pool")
    _need(block_table, torch.int32, "block_table")
    _need(seq_lens, torch.int32, "seq_lens")
    B, Tq, nh, _ = q_abs.shape
    dev = q_abs.device
    if o_lat is None:
        o_lat = torch.empty(B, Tq, nh, D_C, dtype=torch.bfloat16, device=dev)
    if lse is None:
        lse = torch.empty(B, Tq, nh, dtype=torch.float32, device=dev)
    _need(o_lat, torch.bfloat16, "o_lat")
    _need(lse, torch.float32, "lse")
    if workspace is None:
        workspace = torch.empty(max(1, decode_workspace_size(B, Tq, num_splits)), dtype=torch.uint8, device=dev)
    st = lib().mla_decode(_ptr(q_abs), _ptr(kv_pool), _ptr(block_table), _ptr(seq_lens), B, Tq, nh,
                          kv_pool.shape[0], block_table.shape[1], float(scale), int(bool(causal)),
                          int(num_splits), _ptr(o_lat), _ptr(lse), _ptr(workspace), workspace.numel(),
                          _stream(stream))
    _check(st, "mla_decode")
    return o_lat, lse


def decode_static_scratch(q_abs, kv_pool, block_table, seq_lens, scale: float = SCALE, causal: bool = False,
                          num_splits: int = 0, o_lat=None, lse=None, stream=None) -> Tuple:
    """Like decode(), without a workspace: the library's own fixed device scratch is used
    (for callers that cannot allocate; calls on one device must not overlap)."""
    import torch
    _need(q_abs, torch.bfloat16, "q_abs")
    _need(kv_pool, torch.bfloat16, "kv_pool")
    _need(block_table, torch.int32, "block_table")
    _need(seq_lens, torch.int32, "seq_lens")
    B, Tq, nh, _ = q_abs.shape
    if o_lat is None:
        o_lat = torch.empty(B, Tq, nh, D_C, dtype=torch.bfloat16, device=q_abs.device)
    if lse is None:
        lse = torch.empty(B, Tq, nh, dtype=torch.float32, device=q_abs.device)
    st = lib().mla_decode_static_scratch(_ptr(q_abs), _ptr(kv_pool), _ptr(block_table), _ptr(seq_lens), B, Tq,
                                         nh, kv_pool.shape[0], block_table.shape[1], float(scale),
                                         int(bool(causal)), int(num_splits), _ptr(o_lat), _ptr(lse),
                                         _stream(stream))
    _check(st, "mla_decode_static_scratch")
    return o_lat, lse


def combine(o_parts, lse_parts, o_out=None, lse_out=None, stream=None):
    """Merge partial results over disjoint token sets: o_parts [R, rows, 512] f32, lse_parts [R, rows] f32."""
    import torch
    _need(o_parts, torch.float32, "o_parts")
    _need(lse_parts, torch.float32, "lse_parts")
    R, rows = lse_parts.shape
    if o_out is None:
        o_out = torch.empty(rows, D_C, dtype=torch.bfloat16, device=o_parts.device)
    if lse_out is None:
        lse_out = torch.empty(rows, dtype=torch.float32, device=o_parts.device)
    _check(lib().mla_combine(_ptr(o_parts), _ptr(lse_parts), R, rows, _ptr(o_out), _ptr(lse_out),
                             _stream(stream)), "mla_combine")
    return o_out, lse_out


def index_scores(q_idx, idx_pool, block_table, seq_lens, scores=None, stream=None):
    """Index scores of every cached token: scores[b, t] = q_idx[b] . idx_pool[block_table[b, t // 64], t % 64]
    for t < seq_lens[b] (later entries are not written).  q_idx [B, d_idx] bf16, idx_pool [P, 64, d_idx]
    bf16.  Returns scores [B, max_pages * 64] f32."""
    import torch
    _need(q_idx, torch.bfloat16, "q_idx")
    _need(idx_pool, torch.bfloat16, "idx_pool")
    _need(block_table, torch.int32, "block_table")
    _need(seq_lens, torch.int32, "seq_lens")
    B, d_idx = q_idx.shape
    max_pages = block_table.shape[1]
    if scores is None:
        scores = torch.empty(B, max_pages * PAGE, dtype=torch.float32, device=q_idx.device)
    _need(scores, torch.float32, "scores")
    _check(lib().mla_index_scores(_ptr(q_idx), _ptr(idx_pool), _ptr(block_table), _ptr(seq_lens), B, d_idx,
                                  idx_pool.shape[0], max_pages, _ptr(scores), _stream(stream)), "mla_index_scores")
    return scores


def index_scores_e4m3(q_idx, idx_codes, idx_scale, block_table, seq_lens, scores=None, stream=None):
    """Index scores over an E4M3 index cache: scores[b, t] = scale(b, t) * q_idx[b] . value(codes(b, t)).
    idx_codes [P, 64, d_idx] uint8 (or float8_e4m3fn), idx_scale [P, 64] f32.  Returns [B, max_pages * 64] f32."""
    import torch
    _need(q_idx, torch.bfloat16, "q_idx")
    if idx_codes.dtype != torch.uint8:
        idx_codes = idx_codes.view(torch.uint8)
    _need(idx_codes, torch.uint8, "idx_codes")
    _need(idx_scale, torch.float32, "idx_scale")
    _need(block_table, torch.int32, "block_table")
    _need(seq_lens, torch.int32, "seq_lens")
    B, d_idx = q_idx.shape
    max_pages = block_table.shape[1]
    if scores is None:
        scores = torch.empty(B, max_pages * PAGE, dtype=torch.float32, device=q_idx.device)
    _need(scores, torch.float32, "scores")
    _check(lib().mla_index_scores_e4m3(_ptr(q_idx), _ptr(idx_codes), _ptr(idx_scale), _ptr(block_table),
                                       _ptr(seq_lens), B, d_idx, idx_codes.shape[0], max_pages, _ptr(scores),
                                       _stream(stream)), "mla_index_scores_e4m3")
    return scores


def topk_gather(scores, seq_lens, kv_pool, block_table, k: int, stream=None):
    """The k best-scored tokens of each sequence (ties: lower position; NaN last) and their cache rows.

    Returns (sel_index [B, k] int32, sel_pool [B * npk, 64, 576] bf16, sel_block_table [B, npk] int32,
    sel_lens [B] int32), npk = ceil(k / 64)."""
    import torch
    _need(scores, torch.float32, "scores")
    _need(kv_pool, torch.bfloat16, "kv_pool")
    _need(block_table, torch.int32, "block_table")
    _need(seq_lens, torch.int32, "seq_lens")
    B, max_pages = block_table.shape
    npk = (int(k) + PAGE - 1) // PAGE
    dev = scores.device
    sel_index = torch.empty(B, max(1, int(k)), dtype=torch.int32, device=dev)
    sel_pool = torch.empty(max(1, B * npk), PAGE, D, dtype=torch.bfloat16, device=dev)
    sel_bt = torch.empty(B, max(1, npk), dtype=torch.int32, device=dev)
    sel_lens = torch.empty(B, dtype=torch.int32, device=dev)
    _check(lib().mla_topk_gather(_ptr(scores), _ptr(seq_lens), _ptr(kv_pool), _ptr(block_table), B,
                                 kv_pool.shape[0], max_pages, int(k), _ptr(sel_index), _ptr(sel_pool), _ptr(sel_bt),
                                 _ptr(sel_lens), _stream(stream)), "mla_topk_gather")
    return sel_index, sel_pool, sel_bt, sel_lens


def decode_sparse_workspace_size(batch: int, max_pages: int, k: int) -> int:
    return int(lib().mla_decode_sparse_workspace_size(batch, max_pages, k))


def decode_sparse(q_abs, q_idx, kv_pool, idx_pool, block_table, seq_lens, k: int, scale: float = SCALE,
                  o_lat=None, lse=None, sel_index=None, workspace=None, stream=None, idx_scale=None) -> Tuple:
    """The indexer decode of one new token per sequence: index scores, top k, the decode over the k
    selected tokens.  q_abs [B, 1, 128, 576] bf16, q_idx [B, d_idx] bf16, idx_pool [P, 64, d_idx] bf16
    (or, with idx_scale [P, 64] f32, E4M3 codes as uint8 / float8_e4m3fn).
    Returns (o_lat [B, 1, 128, 512] bf16, lse [B, 1, 128] f32, sel_index [B, k] int32)."""
    import torch
    _need(q_abs, torch.bfloat16, "q_abs")
    _need(q_idx, torch.bfloat16, "q_idx")
    _need(kv_pool, torch.bfloat16, "kv_pool")
    if idx_scale is None:
        _need(idx_pool, torch.bfloat16, "idx_pool")
    else:
        if idx_pool.dtype != torch.uint8:
            idx_pool = idx_pool.view(torch.uint8)
        _need(idx_pool, torch.uint8, "idx_pool")
        _need(idx_scale, torch.float32, "idx_scale")
    _need(block_table, torch.int32, "block_table")
    _need(seq_lens, torch.int32, "seq_lens")
    B, Tq, nh, _ = q_abs.shape
    if Tq != 1:
        raise ValueError("decode_sparse: one new token per sequence (q_abs [B, 1, 128, 576])")
    dev = q_abs.device
    if o_lat is None:
        o_lat = torch.empty(B, 1, nh, D_C, dtype=torch.bfloat16, device=dev)
    if lse is None:
        lse = torch.empty(B, 1, nh, dtype=torch.float32, device=dev)
    if sel_index is None:
        sel_index = torch.empty(B, max(1, int(k)), dtype=torch.int32, device=dev)
    _need(o_lat, torch.bfloat16, "o_lat")
    _need(lse, torch.float32, "lse")
    _need(sel_index, torch.int32, "sel_index")
    max_pages = block_table.shape[1]
    if workspace is None:
        workspace = torch.empty(max(1, decode_sparse_workspace_size(B, max_pages, int(k))), dtype=torch.uint8,
                                device=dev)
    st = lib().mla_decode_sparse(_ptr(q_abs), _ptr(q_idx), _ptr(kv_pool), _ptr(idx_pool),
                                 _ptr(idx_scale) if idx_scale is not None else None, _ptr(block_table),
                                 _ptr(seq_lens), B, nh, q_idx.shape[1], kv_pool.shape[0], max_pages, int(k),
                                 float(scale), _ptr(o_lat), _ptr(lse), _ptr(sel_index), _ptr(workspace),
                                 workspace.numel(), _stream(stream))
    _check(st, "mla_decode_sparse")
    return o_lat, lse, sel_index


def get_device_status(stream=None) -> Tuple[int, int]:
    """Synchronise the stream; read and clear the device status word.  Returns (status, word)."""
    w = ctypes.c_uint32(0)
    st = lib().mla_get_device_status(_stream(stream), ctypes.byref(w))
    return int(st), int(w.value)


def launch_count() -> int:
    """Kernels the library has enqueued in this process so far."""
    return int(lib().mla_test_launch_count())


def test_bounded_wait(limit_ms: int = 50, stream=None) -> None:
    """Enqueue the bounded-wait probe (a wait nothing completes; it must give up)."""
    _check(lib().mla_test_bounded_wait(int(limit_ms), _stream(stream)), "mla_test_bounded_wait")
