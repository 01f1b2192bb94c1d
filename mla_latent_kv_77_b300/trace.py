"""Per-warp event timeline of the decode kernel (a profiling tool; the library itself is built
without it).

  python -m mla_latent_kv_77_b300.trace [--workload NAME] [--out FILE.npz]

builds ``libmla_trace.so`` from the same sources with ``-DMLA_TRACE`` (every role of the decode
kernel then stamps its waits and issues with the SM cycle counter, see ``Tracer`` in
``csrc/ptx.cuh``), runs one ``mla_decode`` call of the workload with a trace buffer, saves the raw
records and prints, per role, the median time of each wait and piece of work per page.

Record layout: [CTA][warp][slot] 64-bit words, tag in bits 48-63, SM cycles (or, for tags >=
0x8000, the global nanosecond timer) in bits 0-47.  Even CTAs score, odd CTAs accumulate.
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
    ap.add_argument("--summarize", default=None, help="only summarise an existing record")
    args = ap.parse_args()
    if args.summarize:
        print(summarize(args.summarize))
        return 0
    build()
    out = args.out or f"trace_{args.workload}.npz"
    record(args.workload, out)
    print(summarize(out))
    return 0


if __name__ == "__main__":
    sys.exit(main())
