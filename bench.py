"""Benchmark: MLA decode tokens/s and fraction of roofline on B300.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

One step = one `mla_decode` call (split plan + decode kernel + LSE combine) over one
batch of synthetic queries against a resident paged latent cache.  Default workload:
batch 64, 4096-token contexts, 128 heads, 576-wide bf16 rows in 64-token pages.
`value` is device-timed whole-job throughput (query tokens / s) with inputs resident in
HBM; `e2e` is the same metric through the C ABI with host buffers (queries copied in,
latent output and LSE copied out every step).  `--impl reference` times the fp64 CPU
oracle (the only reference implementation there is) on a bounded sample of the same
workload.  Multi-GPU (torchrun): every rank decodes its own batch (weak scaling), no
collective on the data path; the barrier and max-over-ranks only bracket the timing.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MLA decode tokens/s and % roofline (HBM GB/s, TC util), B=64 H=128 L=4K"
UNIT = "tokens/s"
# the same metric, named for each workload the bench can run (the default one is the first)
METRICS = {
    "b64_l4096": METRIC,
    "b1_l512": "MLA decode tokens/s and % roofline (HBM GB/s, TC util), B=1 H=128 L=512",
    "b128_ragged32k": "MLA decode tokens/s and % roofline (HBM GB/s, TC util), B=128 H=128 L~U[1,32K]",
    "b8_l128k_peaked": "MLA decode tokens/s and % roofline (HBM GB/s, TC util), B=8 H=128 L=128K peaked",
    "b32_tq4_causal_fused": "MLA decode tokens/s and % roofline (HBM GB/s, TC util), B=32 Tq=4 H=128 L=8K causal",
}
ROW_BYTES = 576 * 2
FLOP_PER_TOKEN_QUERY = 2 * 128 * (576 + 512)
E2E_SLOTS = 4  # device buffer sets the end-to-end loop rotates through
L2_BYTES = 126 * 1024 * 1024


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return dict(hbm_gbs=d["hbm_gbs"], bf16_tflops=d["bf16_tflops"],
                    bf16_tflops_sustained=d.get("bf16_tflops_sustained"), source="measured")
    return dict(hbm_gbs=6400.0, bf16_tflops=1800.0, bf16_tflops_sustained=1400.0, source="fallback")


def kernel_source_hash() -> str:
    """Hash of what the decode launch is built from: the decode kernels, the PTX wrappers they
    use, and the decode's launch code in mla.cu (decode_enqueue and mla_decode; the rest of
    mla.cu serves other calls)."""
    csrc = os.path.join(ROOT, "mla_latent_kv_77_b300", "csrc")
    h = hashlib.sha256()
    for f in ("decode_kernels.cuh", "ptx.cuh"):
        h.update(open(os.path.join(csrc, f), "rb").read())
    host = open(os.path.join(csrc, "mla.cu"), "rb").read()
    for start, end in ((b"mla_status_t decode_enqueue(", b"// (end of the decode launch code)"),
                       (b"mla_status_t mla_decode(", b"mla_status_t mla_decode_static_scratch(")):
        a, b = host.find(start), host.find(end)
        h.update(host[a:b] if 0 <= a < b else host)
    return h.hexdigest()[:16]


def profiled_traffic(workload: str):
    """DRAM bytes per decode launch from the committed ncu summary, if it was taken on the
    current kernel sources (else None)."""
    p = os.path.join(ROOT, "profiles", "decode_traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p))
    e = d.get(workload)
    if not e or e.get("source_hash") != kernel_source_hash():
        return None
    return e.get("dram_bytes_per_launch")


class _Nvml:
    """The few NVML calls the sampler needs, through ctypes on the driver's libnvidia-ml
    (read-only queries)."""

    CLOCK_SM = 1

    def __init__(self, index: int):
        import ctypes
        self.c = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit failed")
        self.dev = ctypes.c_void_p()
        if self.lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(index), ctypes.byref(self.dev)) != 0:
            raise RuntimeError("no NVML device")
        self.reasons_fn = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.lib.nvmlDeviceGetCurrentClocksThrottleReasons

    def _clock(self, fn) -> float:
        v = self.c.c_uint()
        if fn(self.dev, self.c.c_int(self.CLOCK_SM), self.c.byref(v)) != 0:
            raise RuntimeError("NVML clock query failed")
        return float(v.value)

    def sm_clock(self) -> float:
        return self._clock(self.lib.nvmlDeviceGetClockInfo)

    def sm_max_clock(self) -> float:
        return self._clock(self.lib.nvmlDeviceGetMaxClockInfo)

    def reasons(self) -> int:
        v = self.c.c_ulonglong()
        if self.reasons_fn(self.dev, self.c.byref(v)) != 0:
            raise RuntimeError("NVML reasons query failed")
        return int(v.value)

    def close(self):
        self.lib.nvmlShutdown()


class ClockSampler:
    """SM clock and throttle reasons sampled during the timed region (read only).

    NVML is polled from a background thread about every 0.2 ms, so even a timed region of a
    couple of milliseconds holds about ten samples; only those between mark_begin() and mark_end() are
    reported.  Without NVML it falls back to nvidia-smi at 100 ms (whose samples then mostly
    fall outside a short timed region; `source` says which was used)."""

    # NVML clock-event reason bits
    REASONS = (("sw_power_cap", 0x4), ("hw_slowdown", 0x8), ("sw_thermal_slowdown", 0x20),
               ("hw_thermal_slowdown", 0x40))
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, period_s: float = 0.0002):
        self.gpu, self.period = gpu_index, period_s
        self.nv = self.proc = None
        self.samples, self.t_begin, self.t_end = [], None, None
        self.path = os.path.join("/tmp", f"mla_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            import threading
            self.nv = _Nvml(self.gpu)
            self.smax = self.nv.sm_max_clock()
            self.stop = threading.Event()
            self.thread = threading.Thread(target=self._poll, daemon=True)
            self.thread.start()
            time.sleep(0.02)
            return self
        except Exception:
            self.nv = None
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def _poll(self):
        while not self.stop.is_set():
            try:
                t = time.perf_counter()
                self.samples.append((t, self.nv.sm_clock(), self.nv.reasons()))
            except Exception:
                return
            time.sleep(self.period)

    def mark_begin(self):
        self.t_begin = time.perf_counter()

    def mark_end(self):
        self.t_end = time.perf_counter()

    def __exit__(self, *a):
        if self.nv is not None:
            self.stop.set()
            self.thread.join(timeout=5)
            try:
                self.nv.close()
            except Exception:
                pass
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.nv is not None:
            lo = self.t_begin if self.t_begin is not None else -math.inf
            hi = self.t_end if self.t_end is not None else math.inf
            win = [x for x in self.samples if lo <= x[0] <= hi]
            reasons = set()
            for _, _, rs in win:
                for name, bit in self.REASONS:
                    if rs & bit:
                        reasons.add(name)
            sm = [x[1] for x in win]
            return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": self.smax,
                    "reasons": sorted(reasons), "samples": len(sm), "source": "nvml, about 0.2 ms, timed region only"}
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["clock sampling unavailable"]}
        sm, smax, reasons = [], None, set()
        names = ["active", "hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names[1:], parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        try:
            os.remove(self.path)
        except OSError:
            pass
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm), "source": "nvidia-smi, 100 ms"}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(x: float, world: int, device=None) -> float:
    """The slowest rank's value, on every rank (x itself with one rank): the job's time is
    that of its slowest replica."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(units_per_step: int, steps: int, world: int, slowest_ms: float) -> float:
    """Whole-job throughput: the units all ranks processed over the slowest rank's time."""
    return units_per_step * steps * world / (slowest_ms / 1000.0)


def cpu_oracle_rate(case, budget_s: float = 12.0, max_seqs: int = None):
    """Time the fp64 oracle (absorbed form, all host cores) on a bounded sample of whole
    sequences of the workload; returns (tokens/s, cores, sample description)."""
    import oracle
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    from helpers import sub_problem
    cores = oracle.default_threads()
    B = case.B
    # calibrate on one sequence, then size the sample to the budget
    q, pool, bt, lens = sub_problem(case, [0])
    t0 = time.perf_counter()
    oracle.decode_absorbed(q, pool, bt, lens, case.scale, causal=case.causal, nthreads=cores)
    t1 = time.perf_counter() - t0
    n = max(1, min(B if max_seqs is None else max_seqs, int(budget_s / max(t1, 1e-3))))
    seqs = list(range(1, 1 + n)) if n + 1 <= B else list(range(n))
    seqs = [s % B for s in seqs]
    q, pool, bt, lens = sub_problem(case, seqs)
    t0 = time.perf_counter()
    oracle.decode_absorbed(q, pool, bt, lens, case.scale, causal=case.causal, nthreads=cores)
    dt = time.perf_counter() - t0
    toks = n * case.Tq
    return toks / dt, cores, f"{n} of {B} sequences x {case.Tq} query tokens x 128 heads ({dt:.1f} s)"


def graph_us(calls, reps: int) -> float:
    """Device time per call of `calls` (each takes the stream to enqueue on), captured once into a
    CUDA graph and replayed `reps` times back to back between one event pair: the host's per-call
    cost (argument checks, tensor-map encoding, Python) stays out of the timed region, as in a
    serving loop that replays a captured decode step."""
    import torch
    gs = torch.cuda.Stream()
    gs.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=gs):
        for c in calls:
            c(gs)
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    cur = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(cur)
    for _ in range(reps):
        g.replay()
    e1.record(cur)
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) * 1000.0 / (reps * len(calls))
    del g
    return us


def _l2_copies(bytes_per_copy: int) -> int:
    """Copies of a call's inputs that cover twice the 126 MB L2, so no call finds its inputs cached."""
    return max(2, -(-2 * 126 * 2 ** 20 // bytes_per_copy))


def fused_leg(mla, workloads, dev, stream, steps: int, warmup: int, pk) -> dict:
    """The fused absorb -> decode -> up-projection chain on the batch-32, 4-query causal
    workload (8192 + 4 cached tokens per sequence).  Each call and the whole chain are captured
    into CUDA graphs and replayed (graph_us).  Inputs larger than L2: the GEMMs cycle through
    copies of their 16.8 MB weights covering twice the L2, and the decode streams 302 MB of cache.
    Fractions are of the HBM roofline over algorithmic bytes (weights, inputs and outputs for the
    GEMMs; the cache rows for the decode)."""
    import torch
    case = workloads.make_workload("b32_tq4_causal_fused", seed=0, device=dev)
    B, Tq = case.B, case.Tq
    n = B * Tq
    qn, qr = case.q_nope.reshape(n, 128, 128), case.q_rope.reshape(n, 128, 64)
    q_abs = torch.empty(n, 128, 576, dtype=torch.bfloat16, device=dev)
    o_lat = torch.empty(B, Tq, 128, 512, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(B, Tq, 128, dtype=torch.float32, device=dev)
    out = torch.empty(n, 128, 128, dtype=torch.bfloat16, device=dev)
    bt, sl = case.block_table.to(dev), case.seq_lens.to(dev)
    ws = torch.empty(mla.decode_workspace_size(B, Tq, 0), dtype=torch.uint8, device=dev)
    w_bytes = 128 * 128 * 512 * 2
    copies = _l2_copies(w_bytes)
    w_uk = [case.w_uk.clone() for _ in range(copies)]
    w_uv = [case.w_uv.clone() for _ in range(copies)]

    def absorb(i):
        return lambda st: mla.absorb_q(qn, qr, w_uk[i % copies], out=q_abs, stream=st)

    def decode(st):
        mla.decode(q_abs.view(B, Tq, 128, 576), case.pool, bt, sl, case.scale, causal=True, o_lat=o_lat, lse=lse,
                   workspace=ws, stream=st)

    def up(i):
        return lambda st: mla.up_proj(o_lat.view(n, 128, 512), w_uv[i % copies], out=out, stream=st)
    for i in range(warmup):
        absorb(i)(stream)
        decode(stream)
        up(i)(stream)
    torch.cuda.synchronize()
    us = {
        "mla_absorb_q": graph_us([absorb(i) for i in range(copies)], max(1, steps // copies)),
        "mla_decode": graph_us([decode] * 10, max(1, steps // 10)),
        "mla_up_proj": graph_us([up(i) for i in range(copies)], max(1, steps // copies)),
    }
    chain = []
    for i in range(8):
        chain += [absorb(i), decode, up(i)]
    chain_us = graph_us(chain, max(1, steps // 8)) * 3
    bytes_ = {
        "mla_absorb_q": w_bytes + n * 128 * (128 + 64) * 2 + n * 128 * 576 * 2,
        "mla_decode": int(case.seq_lens.to(torch.int64).sum()) * ROW_BYTES,
        "mla_up_proj": w_bytes + n * 128 * 512 * 2 + n * 128 * 128 * 2,
    }
    res = {"workload": "b32_tq4_causal_fused", "tokens": n, "unit": "us per call", "steps": steps,
           "timing": "CUDA-graph replays; GEMM weights rotate over %d copies (2 x L2)" % copies}
    for k in us:
        gbs = bytes_[k] / (us[k] * 1e-6) / 1e9
        res[k] = {"us": us[k], "bytes": bytes_[k], "achieved_gbs": gbs, "frac_hbm": gbs / pk["hbm_gbs"]}
    flops = 2 * 128 * sum(max(0, 8196 - (Tq - 1 - t)) for t in range(Tq)) * B * (576 + 512)
    res["mla_decode"]["tensor_frac"] = flops / (res["mla_decode"]["us"] * 1e-6) / 1e12 / pk["bf16_tflops"]
    res["chain_us"] = chain_us
    st, word = mla.get_device_status()
    assert st == 0, f"device status {word:#x}"
    del case, w_uk, w_uv
    torch.cuda.empty_cache()
    return res


def append_leg(mla, workloads, dev, stream, steps: int, warmup: int, pk) -> dict:
    """The cache write (mla_cache_append: c = W^DKV h, rotated k^R, scattered into the pool) on its
    three workloads: one decode step's 64 new tokens, the causal step's 128, and a 4096-token
    prompt, all at d_model 5120; and the compressed write (mla_cache_append_compressed) with
    blocks of 4 (64 tokens) and of 128.  Captured into a CUDA graph and replayed (graph_us); inputs larger
    than L2: the calls cycle through copies of (h, W^DKV, W^KR) covering twice the 126 MB L2.
    Roofline: the HBM bytes a call must move (both weights, h, the written rows) and the tensor
    FLOPs (2 x tokens x 576 x d_model); the prompt is the tensor-bound one."""
    import torch
    res = {"unit": "us per call", "steps": steps, "d_model": workloads.D_MODEL,
           "timing": "CUDA-graph replays; inputs rotate over copies covering 2 x 126 MB of L2"}
    for name in workloads.APPEND_WORKLOADS:
        ac = workloads.make_append_workload(name, seed=0, device=dev)
        c = ac.case
        n, d = ac.n_tokens, ac.d_model
        copies = _l2_copies(ac.weight_bytes() + n * d * 2)
        hs = [ac.h.clone() for _ in range(copies)]
        wds = [ac.w_dkv.clone() for _ in range(copies)]
        wrs = [ac.w_kr.clone() for _ in range(copies)]
        bt, sl, pool = c.block_table.to(dev), c.seq_lens.to(dev), c.pool

        def call(k):
            return lambda st: mla.cache_append(hs[k], wds[k], wrs[k], bt, sl, pool, q_len=c.Tq, stream=st)
        for i in range(max(warmup, copies)):
            call(i % copies)(stream)
        torch.cuda.synchronize()
        n0 = mla.launch_count()
        call(0)(stream)
        launches = mla.launch_count() - n0
        us = graph_us([call(k) for k in range(copies)], max(1, steps // copies))
        bytes_ = ac.weight_bytes() + n * d * 2 + n * ROW_BYTES
        flops = 2.0 * n * 576 * d
        gbs = bytes_ / (us * 1e-6) / 1e9
        tf = flops / (us * 1e-6) / 1e12
        t_roof = max(bytes_ / (pk["hbm_gbs"] * 1e9), flops / (pk["bf16_tflops"] * 1e12))
        res[name] = {"tokens": n, "us": us, "bytes": bytes_, "achieved_gbs": gbs, "frac_hbm": gbs / pk["hbm_gbs"],
                     "tflops": tf, "frac_tensor": tf / pk["bf16_tflops"], "t_roof_us": t_roof * 1e6,
                     "roofline_frac": t_roof / (us * 1e-6), "launches_per_call": launches, "copies": copies}
        del hs, wds, wrs, ac, c, pool
        torch.cuda.empty_cache()
    for name in workloads.COMPRESS_WORKLOADS:
        cc = workloads.make_compress_workload(name, seed=0, device=dev)
        c = cc.case
        n, d = cc.n_tokens, cc.d_model
        copies = _l2_copies(cc.weight_bytes() + n * d * 2)
        hs = [cc.h.clone() for _ in range(copies)]
        wds = [cc.w_dkv.clone() for _ in range(copies)]
        wrs = [cc.w_kr.clone() for _ in range(copies)]
        wzs = [cc.w_z.clone() for _ in range(copies)]
        bt, sl, pool = c.block_table.to(dev), c.seq_lens.to(dev), c.pool

        def ccall(k):
            return lambda st: mla.cache_append_compressed(hs[k], wds[k], wrs[k], wzs[k], bt, sl, pool,
                                                          n_blocks=cc.n_blocks, m=cc.m, stream=st)
        for i in range(max(warmup, copies)):
            ccall(i % copies)(stream)
        torch.cuda.synchronize()
        us = graph_us([ccall(k) for k in range(copies)], max(1, steps // copies))
        bytes_ = cc.weight_bytes() + n * d * 2 + (n // cc.m) * ROW_BYTES
        flops = 2.0 * n * 2 * 576 * d
        gbs = bytes_ / (us * 1e-6) / 1e9
        t_roof = max(bytes_ / (pk["hbm_gbs"] * 1e9), flops / (pk["bf16_tflops"] * 1e12))
        res[name] = {"tokens": n, "m": cc.m, "us": us, "bytes": bytes_, "achieved_gbs": gbs,
                     "frac_hbm": gbs / pk["hbm_gbs"], "t_roof_us": t_roof * 1e6,
                     "roofline_frac": t_roof / (us * 1e-6), "copies": copies}
        del hs, wds, wrs, wzs, cc, c, pool
        torch.cuda.empty_cache()
    st, word = mla.get_device_status()
    assert st == 0, f"device status {word:#x}"
    return res


def other_workloads_leg(mla, workloads, dev, steps: int, warmup: int, pk, gpu_index: int = 0) -> dict:
    """The decode on the other large workloads, timed as the headline is (K calls back to back
    between one event pair, two alternating caches so no call finds its cache in L2): the
    batch-8 131072-token peaked rows, the 128 ragged sequences on a randomly paged pool, and
    the batch-32 four-query causal decode.  Per workload: us per call, tokens/s, and the
    fraction of the roofline (HBM bytes or bf16 FLOPs, whichever binds)."""
    import torch
    res = {"unit": "us per call", "steps": steps,
           "timing": "K calls back to back between one event pair; two alternating caches"}
    stream = torch.cuda.current_stream()
    for name in ("b32_tq4_causal_fused", "b8_l128k_peaked", "b128_ragged32k"):
        case = workloads.make_workload(name, seed=0, device=dev)
        pools = [case.pool, case.pool.clone()]
        q_abs = case.q_abs if case.q_abs is not None else mla.absorb_q(case.q_nope, case.q_rope, case.w_uk)
        q_abs = q_abs.view(case.B, case.Tq, 128, 576)
        bt, sl = case.block_table.to(dev), case.seq_lens.to(dev)
        o = torch.empty(case.B, case.Tq, 128, 512, dtype=torch.bfloat16, device=dev)
        l = torch.empty(case.B, case.Tq, 128, dtype=torch.float32, device=dev)
        ws = torch.empty(mla.decode_workspace_size(case.B, case.Tq, 0), dtype=torch.uint8, device=dev)

        def call(i):
            mla.decode(q_abs, pools[i & 1], bt, sl, case.scale, causal=case.causal, o_lat=o, lse=l, workspace=ws,
                       stream=stream)
        for i in range(warmup):
            call(i)
        torch.cuda.synchronize()
        with ClockSampler(gpu_index) as clk:
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            clk.mark_begin()
            e0.record(stream)
            for i in range(steps):
                call(i)
            e1.record(stream)
            torch.cuda.synchronize()
            clk.mark_end()
        us = e0.elapsed_time(e1) * 1000.0 / steps
        lens = case.seq_lens.to(torch.int64)
        cache = int(lens.sum()) * ROW_BYTES
        if case.causal:
            vis = sum(max(0, int(L) - (case.Tq - 1 - t)) for L in case.seq_lens for t in range(case.Tq))
        else:
            vis = int(lens.sum()) * case.Tq
        flops = vis * FLOP_PER_TOKEN_QUERY
        t_mem, t_tc = cache / (pk["hbm_gbs"] * 1e9), flops / (pk["bf16_tflops"] * 1e12)
        res[name] = {"us": us, "tokens_per_s": case.B * case.Tq / (us * 1e-6), "cache_bytes": cache,
                     "bound": "hbm" if t_mem >= t_tc else "tensor",
                     "roofline_frac": max(t_mem, t_tc) / (us * 1e-6), "clocks": clk.summary()}
        st, word = mla.get_device_status()
        assert st == 0, f"device status {word:#x}"
        del case, pools, q_abs, o, l, ws
        torch.cuda.empty_cache()
    return res


def sparse_leg(mla, workloads, dev, steps: int, warmup: int, pk, gpu_index: int = 0) -> dict:
    """The indexer decode (mla_decode_sparse: index scores over every cached token, top k, the
    decode over the k selected rows) on the batch-8, 131072-token workload with k = 512 and a
    128-wide index vector per token.  The whole call (five kernels) is captured into CUDA graphs,
    one per cache of two alternating caches of index vectors and latent rows, each larger than
    L2, and replayed (graph_us): issued from Python one call at a time, the host's per-call cost
    (five launches and their argument checks) comes close to the device time, so the calls
    issued back to back between one event pair are also reported, as `us_issued`.  Each of its
    two own kernels alone is replayed the same way (the index scores alternating between the two
    index caches).  The whole call is also timed over the E4M3 form of the index cache (codes and
    one scale per token: d_idx + 4 bytes per token instead of 2 d_idx), as `e4m3_index`.  Roofline of the call:
    the index vectors it must read plus the selected rows; of the score kernel: the index vectors."""
    import torch
    name = "sparse_b8_l128k_k512"
    sc = workloads.make_sparse_workload(name, seed=0, device=dev)
    c = sc.case
    stream = torch.cuda.current_stream()
    pools = [c.pool, c.pool.clone()]
    idxs = [sc.idx_pool, sc.idx_pool.clone()]
    bt, sl = c.block_table.to(dev), c.seq_lens.to(dev)
    o = torch.empty(c.B, 1, 128, 512, dtype=torch.bfloat16, device=dev)
    l = torch.empty(c.B, 1, 128, dtype=torch.float32, device=dev)
    si = torch.empty(c.B, sc.k, dtype=torch.int32, device=dev)
    ws = torch.empty(mla.decode_sparse_workspace_size(c.B, c.max_pages, sc.k), dtype=torch.uint8, device=dev)

    def call(i, st=None):
        mla.decode_sparse(c.q_abs, sc.q_idx, pools[i & 1], idxs[i & 1], bt, sl, sc.k, c.scale, o_lat=o, lse=l,
                          sel_index=si, workspace=ws, stream=st or stream)
    for i in range(warmup):
        call(i)
    torch.cuda.synchronize()
    n0 = mla.launch_count()
    with ClockSampler(gpu_index) as clk:
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        clk.mark_begin()
        e0.record(stream)
        for i in range(steps):
            call(i)
        e1.record(stream)
        torch.cuda.synchronize()
        clk.mark_end()
    launches = (mla.launch_count() - n0) // steps
    us_issued = e0.elapsed_time(e1) * 1000.0 / steps
    us = graph_us([lambda st, k=k: call(k, st) for k in range(2)], max(1, steps // 2))
    scores = torch.empty(c.B, c.max_pages * 64, dtype=torch.float32, device=dev)
    score_us = graph_us([lambda st, k=k: mla.index_scores(sc.q_idx, idxs[k], bt, sl, scores=scores, stream=st)
                         for k in range(2)], max(1, steps // 2))
    mla.index_scores(sc.q_idx, idxs[0], bt, sl, scores=scores)
    sel = mla.topk_gather(scores, sl, pools[0], bt, sc.k)
    topk_us = graph_us([lambda st: mla.lib().mla_topk_gather(
        mla._ptr(scores), mla._ptr(sl), mla._ptr(pools[0]), mla._ptr(bt), c.B, c.num_pages, c.max_pages, sc.k,
        mla._ptr(sel[0]), mla._ptr(sel[1]), mla._ptr(sel[2]), mla._ptr(sel[3]), mla._stream(st))], steps)
    # the same call over the E4M3 form of the index cache (codes and one scale per token)
    sc8 = workloads.make_sparse_workload(name, seed=0, device=dev, e4m3=True)
    codes = [sc8.idx_codes, sc8.idx_codes.clone()]
    scl = [sc8.idx_scale, sc8.idx_scale.clone()]
    us8 = graph_us([lambda st, k=k: mla.decode_sparse(c.q_abs, sc8.q_idx, pools[k], codes[k], bt, sl, sc.k, c.scale,
                                                      o_lat=o, lse=l, sel_index=si, workspace=ws, stream=st,
                                                      idx_scale=scl[k]) for k in range(2)], max(1, steps // 2))
    score8_us = graph_us([lambda st, k=k: mla.index_scores_e4m3(sc8.q_idx, codes[k], scl[k], bt, sl, scores=scores,
                                                                stream=st) for k in range(2)], max(1, steps // 2))
    st_, word = mla.get_device_status()
    assert st_ == 0, f"device status {word:#x}"
    idx8_bytes = sc8.index_bytes(e4m3=True)
    idx_bytes, sel_bytes = sc.index_bytes(), sc.selected_bytes()
    call_bytes = idx_bytes + sel_bytes
    res = {"workload": name, "batch": c.B, "context": int(c.seq_lens.max()), "k": sc.k, "d_idx": sc.d_idx,
           "us": us, "us_issued": us_issued, "tokens_per_s": c.B / (us * 1e-6), "launches_per_call": launches,
           "call_bytes": call_bytes, "call_roofline_frac": call_bytes / (pk["hbm_gbs"] * 1e9) / (us * 1e-6),
           "index_scores": {"us": score_us, "bytes": idx_bytes, "achieved_gbs": idx_bytes / (score_us * 1e-6) / 1e9,
                            "frac": idx_bytes / (score_us * 1e-6) / 1e9 / pk["hbm_gbs"]},
           "topk_gather_us": topk_us,
           "e4m3_index": {"us": us8, "tokens_per_s": c.B / (us8 * 1e-6),
                          "call_roofline_frac": (idx8_bytes + sel_bytes) / (pk["hbm_gbs"] * 1e9) / (us8 * 1e-6),
                          "index_scores": {"us": score8_us, "bytes": idx8_bytes,
                                           "achieved_gbs": idx8_bytes / (score8_us * 1e-6) / 1e9,
                                           "frac": idx8_bytes / (score8_us * 1e-6) / 1e9 / pk["hbm_gbs"]}},
           "timing": "CUDA-graph replays alternating two caches (the whole call and each kernel alone); "
                     "us_issued: K calls issued back to back from Python between one event pair",
           "clocks": clk.summary()}
    del sc, c, pools, idxs, ws, scores, sel, sc8, codes, scl
    torch.cuda.empty_cache()
    return res


def run_reference(args):
    """The reference arm: the fp64 CPU oracle, as it stands, on the host cores.  Each step
    decodes a bounded sample (`--ref-seqs` whole sequences, all heads and query tokens) of
    the same workload; rank 0 alone runs it under torchrun."""
    world, rank, local = dist_setup()
    if rank != 0:
        return 0
    import oracle
    from mla_latent_kv_77_b300 import workloads
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    from helpers import sub_problem
    spec = dict(workloads.WORKLOADS[args.workload])
    if "ragged" in spec:
        Bf, lo, hi = spec.pop("ragged")
        spec["seq_lens"] = workloads.ragged_lengths(Bf, lo, hi, 0)
    full_B = len(spec["seq_lens"])
    n = min(args.ref_seqs, full_B)
    spec["seq_lens"] = spec["seq_lens"][:n]          # the sample: the first n sequences
    case = workloads.make_case(args.workload, seed=0, device="cpu", **spec)
    if case.q_abs is None:
        case.q_abs = oracle.absorb_q(case.q_nope, case.q_rope, case.w_uk)
    q, pool, bt, lens = sub_problem(case, list(range(n)))
    cores = oracle.default_threads()
    times = []
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        oracle.decode_absorbed(q, pool, bt, lens, case.scale, causal=case.causal, nthreads=cores)
        if i >= args.warmup:
            times.append(time.perf_counter() - t0)
    toks = n * case.Tq
    value = toks * len(times) / sum(times)
    sample = f"{n} of {full_B} sequences x {case.Tq} query tokens x 128 heads per step"
    line = {"metric": METRICS[args.workload], "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1000.0 * sum(times) / len(times), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": {"workload": args.workload, "batch": full_B, "q_len": case.Tq, "heads": 128,
                       "context": int(max(spec["seq_lens"])), "page": 64},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="b64_l4096")
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-fused", action="store_true", help="skip the fused absorb/decode/up-projection timing")
    ap.add_argument("--no-append", action="store_true", help="skip the cache-write timing")
    ap.add_argument("--no-others", action="store_true", help="skip the other large workloads' decode timing")
    ap.add_argument("--no-sparse", action="store_true", help="skip the indexer (top-k sparse) decode timing")
    ap.add_argument("--ref-seqs", type=int, default=2)
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)

    import torch
    world, rank, local = dist_setup()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    import mla_latent_kv_77_b300 as mla
    from mla_latent_kv_77_b300 import build as mla_build, workloads
    mla_build.build()

    # every rank decodes its own batch of the workload (seed offset by rank)
    case = workloads.make_workload(args.workload, seed=rank, device=dev)
    pools = [case.pool, case.pool.clone()]          # alternate two caches: each step misses L2
    if case.q_abs is None:  # fused workload: absorbed queries come from mla_absorb_q first
        q_abs = mla.absorb_q(case.q_nope, case.q_rope, case.w_uk)
    else:
        q_abs = case.q_abs
    bt = case.block_table.to(dev)
    sl = case.seq_lens.to(dev)
    B, Tq = case.B, case.Tq
    o_lat = torch.empty(B, Tq, 128, 512, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(B, Tq, 128, dtype=torch.float32, device=dev)
    ws = torch.empty(mla.decode_workspace_size(B, Tq, 0), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def step(i):
        mla.decode(q_abs, pools[i & 1], bt, sl, case.scale, causal=case.causal, o_lat=o_lat, lse=lse,
                   workspace=ws, stream=stream)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    st, word = mla.get_device_status()
    assert st == 0, f"device status {word:#x}"

    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        t_start = torch.cuda.Event(enable_timing=True)
        t_end = torch.cuda.Event(enable_timing=True)
        n0 = mla.launch_count()
        clk.mark_begin()
        t_start.record(stream)
        for i in range(args.steps):
            step(i)
        t_end.record(stream)
        torch.cuda.synchronize()
        clk.mark_end()
        launches = mla.launch_count() - n0
    if world > 1:
        torch.distributed.barrier()
    total_ms = max_over_ranks(t_start.elapsed_time(t_end), world, dev)
    st, word = mla.get_device_status()
    assert st == 0, f"device status {word:#x}"

    tokens_per_step = B * Tq
    value = job_rate(tokens_per_step, args.steps, world, total_ms)
    ms_per_step = total_ms / args.steps
    cache_bytes = int(case.seq_lens.to(torch.int64).sum()) * ROW_BYTES
    vis = case.seq_lens.to(torch.int64)
    if case.causal:
        vis_total = sum(max(0, int(L) - (Tq - 1 - t)) for L in case.seq_lens for t in range(Tq))
    else:
        vis_total = int(vis.sum()) * Tq
    flops = vis_total * FLOP_PER_TOKEN_QUERY
    # the K calls run back to back between one event pair: an event pair around every call
    # would itself add device time between the calls
    avg_launch_s = total_ms / args.steps / 1000.0
    pk = peaks()
    achieved_gbs = cache_bytes / avg_launch_s / 1e9
    achieved_tflops = flops / avg_launch_s / 1e12
    t_roof = max(cache_bytes / (pk["hbm_gbs"] * 1e9), flops / (pk["bf16_tflops"] * 1e12))
    mem_bound = cache_bytes / (pk["hbm_gbs"] * 1e9) >= flops / (pk["bf16_tflops"] * 1e12)

    # end to end through the C ABI with host buffers, as a serving loop runs it: every step
    # uploads its queries from pinned host memory and downloads its latent output and lse.  The
    # copies run on two copy streams with E2E_SLOTS device buffer sets, so step i's upload
    # overlaps earlier steps' decodes and downloads, and step i's download overlaps later steps'
    # uploads and decodes; every copy stays inside the timed region.  Alone, the box's link moves
    # the 9.4 MB up or 8.4 MB down in about 0.17 and 0.15 ms; both at once take about 0.25 ms.
    q_host = q_abs.cpu().pin_memory()
    slots = E2E_SLOTS
    o_host = [torch.empty(o_lat.shape, dtype=o_lat.dtype).pin_memory() for _ in range(slots)]
    l_host = [torch.empty(lse.shape, dtype=lse.dtype).pin_memory() for _ in range(slots)]
    q_dev = [torch.empty_like(q_abs) for _ in range(slots)]
    o_dev = [torch.empty_like(o_lat) for _ in range(slots)]
    l_dev = [torch.empty_like(lse) for _ in range(slots)]
    h2d = q_host.numel() * q_host.element_size()
    d2h = o_host[0].numel() * o_host[0].element_size() + l_host[0].numel() * l_host[0].element_size()
    up, down = torch.cuda.Stream(), torch.cuda.Stream()
    ev_up = [torch.cuda.Event() for _ in range(slots)]    # slot's queries uploaded
    ev_dec = [torch.cuda.Event() for _ in range(slots)]   # slot's decode done (its queries are free)
    ev_down = [torch.cuda.Event() for _ in range(slots)]  # slot's results downloaded (its outputs are free)

    def e2e_step(i, start):
        k = i % slots
        up.wait_event(ev_dec[k] if i >= slots else start)
        with torch.cuda.stream(up):
            q_dev[k].copy_(q_host, non_blocking=True)
        ev_up[k].record(up)
        stream.wait_event(ev_up[k])
        if i >= slots:
            stream.wait_event(ev_down[k])
        mla.decode(q_dev[k], pools[i & 1], bt, sl, case.scale, causal=case.causal, o_lat=o_dev[k], lse=l_dev[k],
                   workspace=ws, stream=stream)
        ev_dec[k].record(stream)
        down.wait_event(ev_dec[k])
        with torch.cuda.stream(down):
            o_host[k].copy_(o_dev[k], non_blocking=True)
            l_host[k].copy_(l_dev[k], non_blocking=True)
        ev_down[k].record(down)

    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    for rep in range(2):  # the first pass warms up
        n = args.warmup if rep == 0 else args.steps
        torch.cuda.synchronize()
        e0.record(stream)
        for i in range(n):
            e2e_step(i, e0)
        for k in range(min(slots, n)):
            stream.wait_event(ev_down[k])
        e1.record(stream)
        torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world, dev)
    e2e_value = job_rate(tokens_per_step, args.steps, world, e2e_ms)

    fused = None
    if rank == 0 and args.workload == "b64_l4096" and not args.no_fused:
        fused = fused_leg(mla, workloads, dev, stream, steps=max(args.steps, 10), warmup=args.warmup, pk=peaks())
    others = None
    if rank == 0 and world == 1 and args.workload == "b64_l4096" and not args.no_others:
        others = other_workloads_leg(mla, workloads, dev, steps=max(args.steps, 10), warmup=args.warmup, pk=peaks(),
                                     gpu_index=local)
    sparse = None
    if rank == 0 and world == 1 and args.workload == "b64_l4096" and not args.no_sparse:
        sparse = sparse_leg(mla, workloads, dev, steps=max(args.steps, 10), warmup=args.warmup, pk=peaks(),
                            gpu_index=local)
    append = None
    if rank == 0 and args.workload == "b64_l4096" and not args.no_append:
        append = append_leg(mla, workloads, dev, stream, steps=max(args.steps, 20), warmup=args.warmup, pk=peaks())

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        if case.q_abs is None:
            case.q_abs = q_abs
        rate, cores, sample = cpu_oracle_rate(case, budget_s=12.0)
        cpu = {"value": rate, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample}

    if rank == 0:
        traffic = profiled_traffic(args.workload)
        line = {
            "metric": METRICS[args.workload], "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": args.workload, "batch": B, "q_len": Tq, "heads": 128, "d_c": 512, "d_r": 64,
                       "context": int(case.seq_lens.max()), "total_cached_tokens": int(vis.sum()), "page": 64,
                       "causal": bool(case.causal), "parallelism": f"replicas x{world}",
                       "l2": "inputs larger than L2: two alternating caches of %.0f MB each" % (cache_bytes / 1e6)},
            "roofline": {"bound": "hbm" if mem_bound else "tensor",
                         "achieved": achieved_gbs if mem_bound else achieved_tflops,
                         "peak": pk["hbm_gbs"] if mem_bound else pk["bf16_tflops"],
                         "unit": "GB/s" if mem_bound else "TFLOP/s",
                         "frac": (achieved_gbs / pk["hbm_gbs"]) if mem_bound else (achieved_tflops / pk["bf16_tflops"]),
                         "traffic": traffic,
                         "peak_source": pk["source"],
                         "t_roof_us": t_roof * 1e6, "t_launch_us": avg_launch_s * 1e6,
                         "roofline_frac": t_roof / avg_launch_s,
                         "tensor_tflops": achieved_tflops, "tensor_frac": achieved_tflops / pk["bf16_tflops"],
                         "timed_unit": "one mla_decode call (plan + decode + combine kernels); K calls "
                                       "back to back between one CUDA event pair"},
            "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
            "gpu_launches": launches,
            "clocks": clk.summary(),
            "cpu_baseline": cpu,
            "fused": fused,
            "append": append,
            "other_workloads": others,
            "sparse": sparse,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
