"""Shared helpers of the GPU parity tests: tolerance checks and oracle sub-problems."""
import numpy as np
import torch

import oracle

# Tolerances on bf16 outputs vs the fp64 oracle: max abs 2e-2, relative L2 5e-3; lse abs 1e-3.
# Where |oracle| is large (peaked rows) one bf16 ulp of the reference exceeds 2e-2, so the
# elementwise bound is max(2e-2, ulp_bf16(|ref|)) -- the format cannot do better.
ATOL = 2e-2
RTOL_L2 = 5e-3
LSE_ATOL = 1e-3


def bf16_ulp(x: np.ndarray) -> np.ndarray:
    ax = np.maximum(np.abs(x), np.finfo(np.float32).tiny)
    e = np.floor(np.log2(ax))
    return np.exp2(e - 7)


def check_out(gpu, ref, what="o_lat", atol=ATOL, rtol_l2=RTOL_L2):
    g = gpu.detach().float().cpu().numpy().astype(np.float64) if hasattr(gpu, "detach") else np.asarray(gpu)
    ref = np.asarray(ref, dtype=np.float64)
    assert g.shape == ref.shape, (g.shape, ref.shape)
    assert np.all(np.isfinite(g)), f"{what}: non-finite values"
    err = np.abs(g - ref)
    bound = np.maximum(atol, bf16_ulp(ref))
    worst = float((err / bound).max()) if err.size else 0.0
    nrm = np.linalg.norm(ref)
    rel = float(np.linalg.norm(g - ref) / nrm) if nrm > 0 else float(np.linalg.norm(g))
    assert worst <= 1.0, f"{what}: max |err|/bound = {worst:.3f} (max abs err {err.max():.3e})"
    assert rel <= rtol_l2, f"{what}: relative L2 {rel:.3e} > {rtol_l2}"
    return float(err.max()), rel


def check_lse(gpu, ref, atol=LSE_ATOL):
    g = gpu.detach().float().cpu().numpy().astype(np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    inf = np.isneginf(ref)
    assert np.array_equal(np.isneginf(g), inf), "lse: -inf pattern differs"
    d = np.abs(g[~inf] - ref[~inf])
    m = float(d.max()) if d.size else 0.0
    assert m <= atol, f"lse: max abs err {m:.3e}"
    return m


def sub_problem(case, seqs, q_abs=None):
    """Compact copy (CPU) of the pages of sequences `seqs`, with a remapped block table,
    so the oracle can check sampled outputs of a large workload."""
    bt = case.block_table[seqs]
    lens = case.seq_lens[seqs]
    new_bt = torch.full_like(bt, -1)
    ids, cur = [], 0
    for i in range(len(seqs)):
        n = (int(lens[i]) + 63) // 64
        ids.append(bt[i, :n].to(torch.int64))
        new_bt[i, :n] = torch.arange(cur, cur + n, dtype=torch.int32)
        cur += n
    ids = torch.cat(ids) if cur > 0 else torch.zeros(1, dtype=torch.int64)
    pool = case.pool.index_select(0, ids.to(case.pool.device)).cpu()
    q = (case.q_abs if q_abs is None else q_abs)[seqs].cpu()
    return q, pool, new_bt, lens


def oracle_decode(case, seqs=None, heads=None, q_abs=None):
    """Oracle o_lat, lse for sequences `seqs` (default all) and heads `heads` (default all)."""
    if seqs is None:
        seqs = list(range(case.B))
    q, pool, bt, lens = sub_problem(case, seqs, q_abs)
    if heads is not None:
        q = q[:, :, heads]
    return oracle.decode_absorbed(q, pool, bt, lens, case.scale, causal=case.causal)
