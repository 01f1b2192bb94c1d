"""The C-ABI library loads, exports every function include/*.h declares, and rejects
bad arguments on the host (no GPU needed: these calls return before any CUDA call)."""
import ctypes
import json
import os
import re

import pytest

import mla_latent_kv_77_b300 as mla
from mla_latent_kv_77_b300 import build as mla_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    mla_build.build()
    return mla.lib()


def _declared_functions():
    names = []
    for h in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if not h.endswith(".h"):
            continue
        src = open(os.path.join(ROOT, "include", h)).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        names += re.findall(r"^[A-Za-z_][\w\s\*]*?\b(mla_\w+)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_every_declared_symbol_is_exported(lib):
    declared = _declared_functions()
    assert "mla_decode" in declared and "mla_absorb_q" in declared and "mla_up_proj" in declared
    for name in declared:
        assert hasattr(lib, name), name
    assert set(declared) == set(mla.EXPORTS), (set(declared) ^ set(mla.EXPORTS))


def test_version_and_status_strings(lib):
    assert mla.version() >= 100
    for s in mla.Status:
        assert mla.status_string(int(s)) == "MLA_" + ("OK" if s == 0 else "ERR_" + s.name)


def test_cache_bytes_matches_printed_arithmetic(lib):
    """Step 8: 576 numbers per token per layer; 128K tokens x 60 layers x 2 bytes ~ 9.1 GB."""
    g = json.load(open(os.path.join(ROOT, "tests", "golden", "cache_arithmetic.json")))
    pr = g["printed"]
    per_token = mla.cache_bytes(1, 60, 512, 64, 1)
    assert per_token == pr["mla_numbers_per_token"]["value"]
    assert mla.cache_bytes(1, 1, 512, 64, 1) == pr["mla_numbers_per_token_layer"]["value"]
    gb = mla.cache_bytes(131072, 60, 512, 64, 2) / 1e9
    assert abs(gb - pr["mla_gb_report"]["value"]) <= pr["mla_gb_report"]["rounding"]
    assert mla.cache_bytes(-1, 60, 512, 64, 2) == 0


def test_workspace_size(lib):
    a = mla.decode_workspace_size(64, 1, 0)
    assert a > 0
    assert mla.decode_workspace_size(64, 1, 4) > 0
    assert mla.decode_workspace_size(0, 1, 0) == 0
    assert mla.decode_workspace_size(1, 65, 0) == 0        # q_len above the limit
    assert mla.decode_workspace_size(65536, 2, 0) == 0     # too many rows
    assert mla.decode_workspace_size(128, 1, 0) > mla.decode_workspace_size(64, 1, 0)


def _decode_args(**over):
    ws_bytes = mla.decode_workspace_size(2, 1, 0)
    a = dict(q=16, kv=32, bt=48, sl=64, B=2, Tq=1, H=128, P=4, maxp=2, scale=0.07, causal=0, splits=0,
             o=80, lse=96, ws=128, ws_bytes=ws_bytes, stream=None)
    a.update(over)
    return a


def _call_decode(lib, a):
    vp = lambda x: ctypes.c_void_p(x) if x is not None else None
    return lib.mla_decode(vp(a["q"]), vp(a["kv"]), vp(a["bt"]), vp(a["sl"]), a["B"], a["Tq"], a["H"], a["P"],
                          a["maxp"], a["scale"], a["causal"], a["splits"], vp(a["o"]), vp(a["lse"]), vp(a["ws"]),
                          a["ws_bytes"], None)


@pytest.mark.parametrize("over,code", [
    (dict(q=None), mla.Status.INVALID_ARG),
    (dict(kv=None), mla.Status.INVALID_ARG),
    (dict(bt=None), mla.Status.INVALID_ARG),
    (dict(sl=None), mla.Status.INVALID_ARG),
    (dict(o=None), mla.Status.INVALID_ARG),
    (dict(lse=None), mla.Status.INVALID_ARG),
    (dict(B=0), mla.Status.INVALID_ARG),
    (dict(Tq=0), mla.Status.INVALID_ARG),
    (dict(P=0), mla.Status.INVALID_ARG),
    (dict(splits=-1), mla.Status.INVALID_ARG),
    (dict(scale=0.0), mla.Status.INVALID_ARG),
    (dict(scale=float("nan")), mla.Status.INVALID_ARG),
    (dict(H=64), mla.Status.UNSUPPORTED),
    (dict(Tq=65), mla.Status.SHAPE),
    (dict(q=24), mla.Status.ALIGNMENT),
    (dict(kv=8), mla.Status.ALIGNMENT),
    (dict(ws=None), mla.Status.WORKSPACE),
    (dict(ws_bytes=100), mla.Status.WORKSPACE),
])
def test_decode_rejects_bad_arguments_on_host(lib, over, code):
    assert _call_decode(lib, _decode_args(**over)) == code


def test_absorb_and_up_proj_reject_bad_arguments_on_host(lib):
    vp = ctypes.c_void_p
    assert lib.mla_absorb_q(None, vp(16), vp(32), vp(48), 4, 128, None) == mla.Status.INVALID_ARG
    assert lib.mla_absorb_q(vp(16), vp(16), vp(32), vp(48), 0, 128, None) == mla.Status.INVALID_ARG
    assert lib.mla_absorb_q(vp(16), vp(16), vp(32), vp(48), 4, 96, None) == mla.Status.UNSUPPORTED
    assert lib.mla_absorb_q(vp(18), vp(16), vp(32), vp(48), 4, 128, None) == mla.Status.ALIGNMENT
    assert lib.mla_up_proj(vp(16), None, vp(48), 4, 128, None) == mla.Status.INVALID_ARG
    assert lib.mla_up_proj(vp(16), vp(32), vp(48), 4, 100, None) == mla.Status.UNSUPPORTED
    assert lib.mla_up_proj(vp(16), vp(32), vp(50), 4, 128, None) == mla.Status.ALIGNMENT
    assert lib.mla_combine(None, vp(16), 2, 4, vp(32), vp(48), None) == mla.Status.INVALID_ARG
    assert lib.mla_combine(vp(16), vp(16), 0, 4, vp(32), vp(48), None) == mla.Status.INVALID_ARG
    assert lib.mla_test_bounded_wait(0, None) == mla.Status.INVALID_ARG


def _append_args(**over):
    a = dict(h=16, wd=32, wr=48, bt=64, sl=80, B=2, Tq=1, d=5120, P=4, maxp=2, base=10000.0, pool=96)
    a.update(over)
    return a


def _call_append(lib, a):
    vp = lambda x: ctypes.c_void_p(x) if x is not None else None
    return lib.mla_cache_append(vp(a["h"]), vp(a["wd"]), vp(a["wr"]), vp(a["bt"]), vp(a["sl"]), a["B"], a["Tq"],
                                a["d"], a["P"], a["maxp"], a["base"], vp(a["pool"]), None)


@pytest.mark.parametrize("over,code", [
    (dict(h=None), mla.Status.INVALID_ARG),
    (dict(wd=None), mla.Status.INVALID_ARG),
    (dict(wr=None), mla.Status.INVALID_ARG),
    (dict(bt=None), mla.Status.INVALID_ARG),
    (dict(sl=None), mla.Status.INVALID_ARG),
    (dict(pool=None), mla.Status.INVALID_ARG),
    (dict(B=0), mla.Status.INVALID_ARG),
    (dict(Tq=0), mla.Status.INVALID_ARG),
    (dict(P=0), mla.Status.INVALID_ARG),
    (dict(maxp=0), mla.Status.INVALID_ARG),
    (dict(base=1.0), mla.Status.INVALID_ARG),
    (dict(base=float("inf")), mla.Status.INVALID_ARG),
    (dict(d=5000), mla.Status.SHAPE),
    (dict(d=0), mla.Status.SHAPE),
    (dict(B=1 << 11, Tq=1 << 10), mla.Status.SHAPE),
    (dict(h=24), mla.Status.ALIGNMENT),
    (dict(pool=8), mla.Status.ALIGNMENT),
    (dict(bt=66), mla.Status.ALIGNMENT),
])
def test_cache_append_rejects_bad_arguments_on_host(lib, over, code):
    assert _call_append(lib, _append_args(**over)) == code


def test_cache_append_compressed_rejects_bad_arguments_on_host(lib):
    vp = ctypes.c_void_p

    def call(m=4, nb=1, d=5120, wz=64, pool=96):
        return lib.mla_cache_append_compressed(vp(16), vp(32), vp(48), vp(wz) if wz else None, vp(80), vp(112), 2, nb,
                                               m, d, 4, 2, 10000.0, vp(pool), None)
    assert call(wz=None) == mla.Status.INVALID_ARG
    assert call(m=3) == mla.Status.INVALID_ARG
    assert call(m=256) == mla.Status.INVALID_ARG
    assert call(m=0) == mla.Status.INVALID_ARG
    assert call(nb=0) == mla.Status.INVALID_ARG
    assert call(d=100) == mla.Status.SHAPE
    assert call(wz=72) == mla.Status.ALIGNMENT
    assert call(pool=104) == mla.Status.ALIGNMENT


def test_indexer_calls_reject_bad_arguments_on_host(lib):
    vp = ctypes.c_void_p

    def scores(d_idx=128, B=2, q=16, pool=32, sc=64):
        return lib.mla_index_scores(vp(q) if q else None, vp(pool), vp(48), vp(80), B, d_idx, 4, 2,
                                    vp(sc) if sc else None, None)
    assert scores(q=None) == mla.Status.INVALID_ARG
    assert scores(sc=None) == mla.Status.INVALID_ARG
    assert scores(B=0) == mla.Status.INVALID_ARG
    for d in (0, 16, 96, 512):
        assert scores(d_idx=d) == mla.Status.SHAPE
    assert scores(q=24) == mla.Status.ALIGNMENT
    assert scores(pool=40) == mla.Status.ALIGNMENT
    assert scores(sc=66) == mla.Status.ALIGNMENT

    def scores8(d_idx=128, codes=32, scale=64):
        return lib.mla_index_scores_e4m3(vp(16), vp(codes), vp(scale) if scale else None, vp(48), vp(80), 2, d_idx,
                                         4, 2, vp(96), None)
    assert scores8(scale=None) == mla.Status.INVALID_ARG
    assert scores8(d_idx=48) == mla.Status.SHAPE
    assert scores8(codes=40) == mla.Status.ALIGNMENT
    assert scores8(scale=66) == mla.Status.ALIGNMENT

    def topk(k=512, B=2, sc=16, pool=32, sp=48, si=64):
        return lib.mla_topk_gather(vp(sc), vp(80), vp(pool), vp(96), B, 4, 2, k, vp(si) if si else None, vp(sp),
                                   vp(112), vp(128), None)
    assert topk(si=None) == mla.Status.INVALID_ARG
    assert topk(k=0) == mla.Status.INVALID_ARG
    assert topk(B=0) == mla.Status.INVALID_ARG
    assert topk(k=(1 << 18) + 1) == mla.Status.SHAPE
    assert topk(sc=20) == mla.Status.ALIGNMENT
    assert topk(sp=56) == mla.Status.ALIGNMENT
    assert topk(pool=40) == mla.Status.ALIGNMENT

    assert lib.mla_decode_sparse_workspace_size(0, 4, 512) == 0
    assert lib.mla_decode_sparse_workspace_size(2, 4, 0) == 0
    assert lib.mla_decode_sparse_workspace_size(2, 4, (1 << 18) + 1) == 0
    need = lib.mla_decode_sparse_workspace_size(8, 2048, 512)
    # at least the scores, the selection, the compact pool and the decode's own workspace
    assert need >= 8 * 2048 * 64 * 4 + 8 * 512 * 4 + 8 * 8 * 64 * 576 * 2 + lib.mla_decode_workspace_size(8, 1, 0)

    def sparse(k=512, nh=128, d_idx=128, ws=256, nbytes=None, scale=0.07, qa=16):
        nb = need if nbytes is None else nbytes
        return lib.mla_decode_sparse(vp(qa), vp(32), vp(48), vp(64), None, vp(80), vp(96), 8, nh, d_idx, 4096, 2048,
                                     k, scale, vp(112), vp(128), None, vp(ws) if ws else None, nb, None)
    assert sparse(ws=None) == mla.Status.WORKSPACE
    assert sparse(nbytes=need - 1) == mla.Status.WORKSPACE
    assert sparse(nh=64) == mla.Status.UNSUPPORTED
    assert sparse(d_idx=100) == mla.Status.SHAPE
    assert sparse(k=0) == mla.Status.INVALID_ARG
    assert sparse(scale=0.0) == mla.Status.INVALID_ARG
    assert sparse(ws=264) == mla.Status.ALIGNMENT
    assert sparse(qa=20) == mla.Status.ALIGNMENT


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(mla, "_lib", None)
    monkeypatch.setattr(mla, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(mla.MLAError):
        mla.lib()
