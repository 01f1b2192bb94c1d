"""Per-warp event timeline of the decode kernel (a profiling tool; the library itself is built
without it).

  python -m mla_latent_kv_77_b300.trace [--workload NAME] [--out FILE.npz]
  python -m mla_latent_kv_77_b300.trace --append NAME [--out FILE.npz]
  python -m mla_latent_kv_77_b300.trace --topk NAME [--out FILE.npz]

builds ``libmla_trace.so`` from the same sources with ``-DMLA_TRACE`` (every role of the decode
and cache-write kernels then stamps its waits and issues with the SM cycle counter, see ``Tracer``
in ``csrc/ptx.cuh``), runs one ``mla_decode`` (or ``mla_cache_append``) call of the workload with a
trace buffer, saves the raw records and prints, per role, the median time of each wait and piece of
work per page (for the cache write: each step's time since the CTA's setup, and the spread of the
CTAs' start and end times).

Record layout: [CTA][warp][slot] 64-bit words, tag in bits 48-63, SM cycles (or, for tags >=
0x8000, the global nanosecond timer) in bits 0-47; CTAs in linear block order.  In the decode,
even CTAs score, odd CTAs accumulate.
"""
from __future__ import annotations

import argparse
import ctypes
import os
import subprocess
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
TRACE_LIB = os.path.join(HERE, "libmla_trace.so")
SLOTS, WARPS = 2048, 16

# (role, warp, CTA parity, start tag, end tag): the intervals the summary reports
INTERVALS = [
    ("score issuer: wait for its page's data", 9, 0, 0x22, 0x23),
    ("score issuer: wait for its S buffer", 9, 0, 0x23, 0x25),
    ("score issuer: issue the page's 36 MMAs", 9, 0, 0x25, 0x26),
    ("softmax: wait for S", 0, 0, 0x32, 0x33),
    ("softmax: load S, release the buffer", 0, 0, 0x33, 0x34),
    ("softmax: maximum, exponentials, sums", 0, 0, 0x34, 0x35),
    ("softmax: wait for a free ring slot", 0, 0, 0x35, 0x36),
    ("softmax: write the message", 0, 0, 0x36, 0x37),
    ("score producer: wait for a free stage", 8, 0, 0x10, 0x11),
    ("shipper: wait for a staged message", 12, 0, 0x40, 0x41),
    ("accumulate: wait for the page's P", 9, 1, 0x70, 0x71),
    ("accumulate: wait for the page's values", 9, 1, 0x71, 0x74),
    ("accumulate: issue the page's PV MMAs", 9, 1, 0x74, 0x75),
    ("value producer: wait for a free stage", 8, 1, 0x50, 0x51),
    ("P loader: wait for a published message", 10, 1, 0x60, 0x61),
    ("P loader: wait for a free P buffer", 10, 1, 0x61, 0x62),
]


def build() -> str:
    from mla_latent_kv_77_b300 import build as b
    cmd = [b.nvcc(), "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-lineinfo", "-std=c++17",
           "--expt-relaxed-constexpr", "-Xcompiler", "-fPIC", "-shared", "-DMLA_TRACE", "-o", TRACE_LIB] + b.SOURCES
    subprocess.check_call(cmd, cwd=b.CSRC)
    return TRACE_LIB


def record(workload: str, out: str) -> str:
    import torch
    import mla_latent_kv_77_b300 as mla
    from mla_latent_kv_77_b300 import workloads
    if mla._lib is not None:
        raise RuntimeError("the untraced library is already loaded in this process")
    mla.LIB_PATH = TRACE_LIB
    lib = mla.lib()
    lib.mla_trace_set.restype = ctypes.c_int
    lib.mla_trace_set.argtypes = [ctypes.c_void_p]
    dev = torch.device("cuda")
    case = workloads.make_workload(workload, seed=0, device=dev)
    q = case.q_abs if case.q_abs is not None else mla.absorb_q(case.q_nope, case.q_rope, case.w_uk)
    bt, sl = case.block_table.to(dev), case.seq_lens.to(dev)
    ws = torch.empty(mla.decode_workspace_size(case.B, case.Tq, 0), dtype=torch.uint8, device=dev)
    buf = torch.zeros(148 * WARPS * SLOTS, dtype=torch.int64, device=dev)
    for _ in range(3):
        mla.decode(q, case.pool, bt, sl, case.scale, causal=case.causal, workspace=ws)
    torch.cuda.synchronize()
    if lib.mla_trace_set(ctypes.c_void_p(buf.data_ptr())) != 0:
        raise RuntimeError("mla_trace_set failed")
    mla.decode(q, case.pool, bt, sl, case.scale, causal=case.causal, workspace=ws)
    torch.cuda.synchronize()
    lib.mla_trace_set(ctypes.c_void_p(0))
    st, word = mla.get_device_status()
    if st != 0:
        raise RuntimeError(f"device status {word:#x}")
    np.savez_compressed(out, trace=buf.cpu().numpy(), workload=workload)
    return out


def record_append(workload: str, out: str) -> str:
    import torch
    import mla_latent_kv_77_b300 as mla
    from mla_latent_kv_77_b300 import workloads
    if mla._lib is not None:
        raise RuntimeError("the untraced library is already loaded in this process")
    mla.LIB_PATH = TRACE_LIB
    lib = mla.lib()
    lib.mla_trace_set.restype = ctypes.c_int
    lib.mla_trace_set.argtypes = [ctypes.c_void_p]
    dev = torch.device("cuda")
    ac = workloads.make_append_workload(workload, seed=0, device=dev)
    c = ac.case
    bt, sl = c.block_table.to(dev), c.seq_lens.to(dev)
    buf = torch.zeros(148 * WARPS * SLOTS, dtype=torch.int64, device=dev)
    for _ in range(3):
        mla.cache_append(ac.h, ac.w_dkv, ac.w_kr, bt, sl, c.pool, q_len=c.Tq)
    # fresh weights, as in a model's layer loop, so the traced call reads them from HBM
    w_dkv, w_kr, h = ac.w_dkv.clone(), ac.w_kr.clone(), ac.h.clone()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    flush.fill_(1)
    torch.cuda.synchronize()
    if lib.mla_trace_set(ctypes.c_void_p(buf.data_ptr())) != 0:
        raise RuntimeError("mla_trace_set failed")
    mla.cache_append(h, w_dkv, w_kr, bt, sl, c.pool, q_len=c.Tq)
    torch.cuda.synchronize()
    lib.mla_trace_set(ctypes.c_void_p(0))
    st, word = mla.get_device_status()
    if st != 0:
        raise RuntimeError(f"device status {word:#x}")
    np.savez_compressed(out, trace=buf.cpu().numpy(), workload=workload, kind="append")
    return out


# cache-write steps: (name, warp, tag); times since the warp's setup stamp (0x102)
APPEND_STEPS = [
    ("producer: every load issued", 0, 0x111),
    ("producer: every load landed", 0, 0x112),
    ("MMA: first stage landed", 1, 0x120),
    ("MMA: last MMA issued", 1, 0x121),
    ("epilogue: accumulator complete", 2, 0x130),
    ("epilogue: partial staged", 2, 0x131),
    ("epilogue: cluster partials visible", 2, 0x140),
    ("epilogue: rows written", 2, 0x141),
]


def summarize_append(path: str, mhz: float = 2032.0) -> str:
    d = np.load(path)
    tr = d["trace"].reshape(148, WARPS, SLOTS)
    ctas = [b for b in range(148) if (tr[b, 2] != 0).any()]
    lines = [f"{path}: {len(ctas)} CTAs; medians (max) over them, us since the CTA's setup at {mhz:.0f} MHz"]
    for name, warp, tag in APPEND_STEPS:
        xs = []
        for b in ctas:
            tags, t = _events(tr, b, warp)
            t0 = t[tags == 0x102]
            t1 = t[tags == tag]
            if t0.size and t1.size:
                xs.append((t1[0] - t0[0]) / mhz)
        if xs:
            lines.append(f"  {name:40s} {np.median(xs):7.3f} ({np.max(xs):.3f})")
    starts, ends = [], []
    for b in ctas:
        tags, t = _events(tr, b, 2)
        if (tags == 0x8101).any() and (tags == 0x8142).any():
            starts.append(t[tags == 0x8101][0])
            ends.append(t[tags == 0x8142][0])
    if starts:
        t0 = min(starts)
        s_ = (np.array(starts) - t0) / 1000.0
        e_ = (np.array(ends) - t0) / 1000.0
        lines.append(f"  CTA start (global timer, us after the first): median {np.median(s_):.3f} max {s_.max():.3f}")
        lines.append(f"  CTA end: median {np.median(e_):.3f} max {e_.max():.3f}")
    return "\n".join(lines)


def record_topk(workload: str, out: str) -> str:
    import torch
    import mla_latent_kv_77_b300 as mla
    from mla_latent_kv_77_b300 import workloads
    if mla._lib is not None:
        raise RuntimeError("the untraced library is already loaded in this process")
    mla.LIB_PATH = TRACE_LIB
    lib = mla.lib()
    lib.mla_trace_set.restype = ctypes.c_int
    lib.mla_trace_set.argtypes = [ctypes.c_void_p]
    dev = torch.device("cuda")
    sc = workloads.make_sparse_workload(workload, seed=0, device=dev)
    c = sc.case
    bt, sl = c.block_table.to(dev), c.seq_lens.to(dev)
    scores = mla.index_scores(sc.q_idx, sc.idx_pool, bt, sl)
    n_cta = max(148, c.B * TOPK_CLUSTER)
    buf = torch.zeros(n_cta * WARPS * SLOTS, dtype=torch.int64, device=dev)
    for _ in range(3):
        mla.topk_gather(scores, sl, c.pool, bt, sc.k)
    torch.cuda.synchronize()
    if lib.mla_trace_set(ctypes.c_void_p(buf.data_ptr())) != 0:
        raise RuntimeError("mla_trace_set failed")
    mla.topk_gather(scores, sl, c.pool, bt, sc.k)
    torch.cuda.synchronize()
    lib.mla_trace_set(ctypes.c_void_p(0))
    st, word = mla.get_device_status()
    if st != 0:
        raise RuntimeError(f"device status {word:#x}")
    np.savez_compressed(out, trace=buf.cpu().numpy(), workload=workload, kind="topk", n_cta=n_cta,
                        busy=c.B * TOPK_CLUSTER)
    return out


TOPK_CLUSTER = 8
# top-k steps (warp 0, global timer): (name, tag)
TOPK_STEPS = [("keys staged", 0x8201)] + [
    (f"pass {i}: {what}", tag + i) for i in range(4) for what, tag in (
        ("histogram counted", 0x8210), ("cluster barrier passed", 0x8240), ("cluster sum read", 0x8250),
        ("bin chosen", 0x8260), ("rank counts added", 0x8220))] + [
    ("candidates exchanged, threshold found", 0x8270)] + [
    ("output offsets known", 0x8231), ("positions written", 0x8232), ("rows' pool offsets", 0x8233),
    ("rows copied", 0x8234)]


def summarize_topk(path: str) -> str:
    d = np.load(path)
    n_cta, busy = int(d["n_cta"]), int(d["busy"])
    tr = d["trace"].reshape(n_cta, WARPS, SLOTS)
    starts = []
    for b in range(busy):
        tags, t = _events(tr, b, 0)
        if (tags == 0x8200).any():
            starts.append(t[tags == 0x8200][0])
    t_first = min(starts)
    lines = [f"{path}: {busy} CTAs; us after the first CTA's start (global timer): median (max) over CTAs"]
    lines.append(f"  {'start':34s} {np.median((np.array(starts) - t_first) / 1e3):7.3f} "
                 f"({(max(starts) - t_first) / 1e3:.3f})")
    for name, tag in TOPK_STEPS:
        xs = []
        for b in range(busy):
            tags, t = _events(tr, b, 0)
            if (tags == tag).any():
                xs.append((t[tags == tag][0] - t_first) / 1e3)
        if xs:
            lines.append(f"  {name:34s} {np.median(xs):7.3f} ({np.max(xs):.3f})")
    return "\n".join(lines)


def _events(tr, cta, warp):
    x = tr[cta, warp]
    x = x[x != 0]
    return ((x >> 48) & 0xFFFF).astype(np.int64), (x & 0xFFFFFFFFFFFF).astype(np.int64)


def _durations(tags, t, a, b):
    out = []
    for i in np.where(tags == a)[0]:
        j = i + 1
        while j < len(tags) and tags[j] not in (a, b):
            j += 1
        if j < len(tags) and tags[j] == b:
            out.append(t[j] - t[i])
    return np.array(out, dtype=np.float64)


def summarize(path: str, mhz: float = 2032.0) -> str:
    d = np.load(path)
    tr = d["trace"].reshape(148, WARPS, SLOTS)
    busy = [c for c in range(0, 148, 2) if (_events(tr, c, 9)[0] == 0x26).any()]
    lines = [f"{path}: {len(busy)} busy CTA pairs; medians over them, per page, in us at {mhz:.0f} MHz"]
    for name, warp, parity, a, b in INTERVALS:
        med = []
        for c in busy:
            tags, t = _events(tr, c + parity, warp)
            x = _durations(tags, t, a, b)
            if x.size:
                med.append(np.median(x))
        if med:
            lines.append(f"  {name:46s} {np.median(med) / mhz:7.3f}")
    gaps = []
    for c in busy:
        tags, t = _events(tr, c, 9)
        s = t[tags == 0x26]
        if s.size > 2:
            gaps.append(np.median(np.diff(s)))
    if gaps:
        lines.append(f"  {'score issuer 0: time between its pages':46s} {np.median(gaps) / mhz:7.3f}")
    return "\n".join(lines)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default="b64_l4096")
    ap.add_argument("--out", default=None)
    ap.add_argument("--append", default=None, help="trace the cache write on this workload instead")
    ap.add_argument("--topk", default=None, help="trace the top-k selection on this indexer workload instead")
    ap.add_argument("--summarize", default=None, help="only summarise an existing record")
    args = ap.parse_args()
    if args.summarize:
        kind = str(np.load(args.summarize).get("kind", "decode"))
        print({"append": summarize_append, "topk": summarize_topk}.get(kind, summarize)(args.summarize))
        return 0
    build()
    if args.topk:
        out = args.out or f"trace_{args.topk}.npz"
        record_topk(args.topk, out)
        print(summarize_topk(out))
        return 0
    if args.append:
        out = args.out or f"trace_{args.append}.npz"
        record_append(args.append, out)
        print(summarize_append(out))
        return 0
    out = args.out or f"trace_{args.workload}.npz"
    record(args.workload, out)
    print(summarize(out))
    return 0


if __name__ == "__main__":
    sys.exit(main())
