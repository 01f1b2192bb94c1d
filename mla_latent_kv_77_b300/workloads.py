"""Seeded synthetic inputs for MLA decode: the only code shared by the CUDA path's
tests/benchmark and the oracle's tests.  It draws tensors and builds block
tables; it contains none of the attention arithmetic.

Recipe (all draws from fresh ``torch.Generator`` objects, one per tensor, seeded
``1000 * seed + k`` for the k-th tensor of the list below, so every tensor is
reproducible on its own; the ragged lengths come first, from a generator seeded
``seed`` itself):

  --   sequence lengths (ragged workload only): ``randint(lo, hi + 1)``
  k=1  cache rows   ~ N(0, 1) * 0.5, rounded to bf16 (round-to-nearest-even)
  k=2  q_abs        ~ N(0, 1) * 0.5, bf16
  k=3  q_nope       ~ N(0, 1) * 0.5, bf16
  k=4  q_rope       ~ N(0, 1) * 0.5, bf16
  k=5  W_UK         ~ N(0, 1) / sqrt(512), bf16   (standard deviation 1/sqrt(512))
  k=6  W_UV         ~ N(0, 1) / sqrt(512), bf16
  k=7  block-table permutation of the page pool (shuffled layouts)
  k=8  choice of the peaked rows (1% of each sequence's rows scaled by 8 before
       the bf16 rounding)
  --   optional garbage (NaN or 1e30) written into pool pages and tail slots that
       no sequence may read
  k=9  h (cache write: the new tokens' hidden vectors) ~ N(0, 1), bf16
  k=10 W^DKV        ~ N(0, 1) / sqrt(d_model), bf16   (so c ~ N(0, 1))
  k=11 W^KR         ~ N(0, 1) / sqrt(d_model), bf16
  k=12 W^Z (compressed cache write) ~ N(0, 1) / sqrt(d_model), bf16
  k=13 index cache (indexer decode) ~ N(0, 1) / sqrt(d_idx), bf16, one d_idx-wide vector per
       pool row; with ``ties`` set, instead integers uniform in [-2, 2] (many exactly equal
       scores, to exercise the tie rule)
  k=14 q_idx        ~ N(0, 1), bf16 (with ``ties``: integers uniform in [-2, 2])
  --   the E4M3 form of the index cache (no draw): each token's scale is its largest
       |coordinate| / 448 (float32), its codes the coordinates divided by the scale, converted
       by torch's float8_e4m3fn (round to nearest even)

Shapes follow the DeepSeek-V2 attention: 128 heads, 512-d latent, 64-d decoupled
RoPE key, 128-d head, 576-number cache row, 64-token pages.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Dict, List, Optional

import torch

H = 128
D_C = 512
D_R = 64
D_H = 128
D = D_C + D_R
PAGE = 64
SCALE = 1.0 / math.sqrt(D_H + D_R)
D_MODEL = 5120  # DeepSeek-V2 hidden size: the cache write projects 5,120 numbers down to 512


@dataclass
class Case:
    name: str
    B: int
    Tq: int
    causal: bool
    seq_lens: torch.Tensor          # [B] int32 (CPU)
    block_table: torch.Tensor       # [B, max_pages] int32 (CPU), -1 padded
    pool: torch.Tensor              # [num_pages, PAGE, D] bf16
    q_abs: Optional[torch.Tensor] = None   # [B, Tq, H, D] bf16
    q_nope: Optional[torch.Tensor] = None  # [B, Tq, H, D_H] bf16
    q_rope: Optional[torch.Tensor] = None  # [B, Tq, H, D_R] bf16
    w_uk: Optional[torch.Tensor] = None    # [H, D_H, D_C] bf16
    w_uv: Optional[torch.Tensor] = None    # [H, D_H, D_C] bf16
    scale: float = SCALE
    meta: Dict = field(default_factory=dict)

    @property
    def num_pages(self) -> int:
        return int(self.pool.shape[0])

    @property
    def max_pages(self) -> int:
        return int(self.block_table.shape[1])

    def cache_bytes(self) -> int:
        """Bytes of latent cache one decode step must read (each visible row once)."""
        return int(self.seq_lens.to(torch.int64).sum()) * D * 2


def _gen(seed: int, k: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed * 1000 + k)
    return g


def _randn_bf16(shape, std: float, seed: int, k: int, device) -> torch.Tensor:
    x = torch.randn(shape, generator=_gen(seed, k, device), device=device, dtype=torch.float32)
    return (x * std).to(torch.bfloat16)


def make_case(name: str, seq_lens: List[int], Tq: int = 1, causal: bool = False,
              shuffle: bool = False, spare_pages: int = 0, garbage: Optional[str] = None,
              peaked_frac: float = 0.0, q_mode: str = "abs", seed: int = 0,
              device="cpu") -> Case:
    """Build one synthetic decode problem.

    seq_lens     cached tokens per sequence (includes the Tq new tokens when causal).
    shuffle      place pages by a seeded random permutation of the pool (else in order).
    spare_pages  extra pool pages no sequence owns.
    garbage      None, "nan" or "big": fill the unowned pages and the unused tail slots
                 of every sequence's last page with NaN or 1e30, to prove they are never read.
    peaked_frac  fraction of each sequence's rows multiplied by 8 (whole 576-wide row).
    q_mode       "abs": draw q_abs; "nope": draw q_nope, q_rope, W_UK, W_UV; "both"; "none".
    """
    device = torch.device(device)
    B = len(seq_lens)
    lens = torch.tensor(seq_lens, dtype=torch.int32)
    pages_per = [(int(L) + PAGE - 1) // PAGE for L in seq_lens]
    owned = sum(pages_per)
    num_pages = max(1, owned + spare_pages)
    max_pages = max(1, max(pages_per) if pages_per else 1)

    if shuffle:
        perm = torch.randperm(num_pages, generator=_gen(seed, 7, "cpu")).to(torch.int32)
    else:
        perm = torch.arange(num_pages, dtype=torch.int32)
    block_table = torch.full((B, max_pages), -1, dtype=torch.int32)
    cursor = 0
    for b in range(B):
        n = pages_per[b]
        block_table[b, :n] = perm[cursor:cursor + n]
        cursor += n

    base = torch.randn((num_pages, PAGE, D), generator=_gen(seed, 1, device), device=device,
                       dtype=torch.float32) * 0.5
    if peaked_frac > 0.0:
        # scale whole rows by 8 before the bf16 rounding
        g = _gen(seed, 8, "cpu")
        mask = torch.zeros((num_pages, PAGE), dtype=torch.bool)
        for b in range(B):
            L = int(seq_lens[b])
            k = int(math.floor(peaked_frac * L))
            if k == 0:
                continue
            rows = torch.randperm(L, generator=g)[:k]
            pg = block_table[b, (rows // PAGE)].to(torch.int64)
            mask[pg, (rows % PAGE)] = True
        base[mask.to(device)] *= 8.0
    pool = base.to(torch.bfloat16)
    del base

    if garbage is not None:
        val = float("nan") if garbage == "nan" else 1e30
        used = torch.zeros((num_pages, PAGE), dtype=torch.bool)
        for b in range(B):
            L = int(seq_lens[b])
            n = pages_per[b]
            if n == 0:
                continue
            pg = block_table[b, :n].to(torch.int64)
            used[pg[:-1], :] = True
            used[pg[-1], : L - (n - 1) * PAGE] = True
        pool[(~used).to(device)] = val

    case = Case(name=name, B=B, Tq=Tq, causal=causal, seq_lens=lens, block_table=block_table,
                pool=pool)
    if q_mode in ("abs", "both"):
        case.q_abs = _randn_bf16((B, Tq, H, D), 0.5, seed, 2, device)
    if q_mode in ("nope", "both"):
        case.q_nope = _randn_bf16((B, Tq, H, D_H), 0.5, seed, 3, device)
        case.q_rope = _randn_bf16((B, Tq, H, D_R), 0.5, seed, 4, device)
        case.w_uk = _randn_bf16((H, D_H, D_C), 1.0 / math.sqrt(D_C), seed, 5, device)
        case.w_uv = _randn_bf16((H, D_H, D_C), 1.0 / math.sqrt(D_C), seed, 6, device)
    case.meta = dict(seed=seed, shuffle=shuffle, spare_pages=spare_pages, garbage=garbage,
                     peaked_frac=peaked_frac)
    return case


def ragged_lengths(B: int, lo: int, hi: int, seed: int = 0) -> List[int]:
    """Lengths uniform in [lo, hi], drawn first from a generator seeded `seed`."""
    g = torch.Generator()
    g.manual_seed(seed)
    return [int(x) for x in torch.randint(lo, hi + 1, (B,), generator=g)]


# ---------------------------------------------------------------------------
# The five workloads (full size).  Names describe the workload, not an index.
# ---------------------------------------------------------------------------
WORKLOADS = {
    # batch 1, 512-token contiguous cache (identity block table), naive-vs-absorbed check
    "b1_l512": dict(seq_lens=[512], q_mode="both"),
    # batch 64 x 4096 tokens, pages in order
    "b64_l4096": dict(seq_lens=[4096] * 64),
    # batch 128, lengths uniform in [1, 32768], shuffled block table over one pool
    "b128_ragged32k": dict(ragged=(128, 1, 32768), shuffle=True),
    # batch 8 x 131072 tokens, 1% of rows scaled x8 (peaked softmax rows)
    "b8_l128k_peaked": dict(seq_lens=[131072] * 8, peaked_frac=0.01),
    # batch 32, 4 causal query tokens over 8192 prior + 4 new tokens; fused absorb/up-proj
    "b32_tq4_causal_fused": dict(seq_lens=[8192 + 4] * 32, Tq=4, causal=True, q_mode="both"),
}


def make_workload(name: str, seed: int = 0, device="cpu") -> Case:
    spec = dict(WORKLOADS[name])
    if "ragged" in spec:
        B, lo, hi = spec.pop("ragged")
        spec["seq_lens"] = ragged_lengths(B, lo, hi, seed)
    return make_case(name, seed=seed, device=device, **spec)


@dataclass
class AppendCase:
    """A cache write: Tq new tokens per sequence, already counted in the case's seq_lens."""
    case: Case                      # the pool (prior content), block table, lengths
    h: torch.Tensor                 # [B * Tq, d_model] bf16
    w_dkv: torch.Tensor             # [D_C, d_model] bf16
    w_kr: torch.Tensor              # [D_R, d_model] bf16

    @property
    def n_tokens(self) -> int:
        return int(self.h.shape[0])

    @property
    def d_model(self) -> int:
        return int(self.h.shape[1])

    def weight_bytes(self) -> int:
        return (D_C + D_R) * self.d_model * 2


def make_append_case(name: str, seq_lens: List[int], Tq: int = 1, d_model: int = D_MODEL,
                     shuffle: bool = False, spare_pages: int = 0, garbage: Optional[str] = None,
                     seed: int = 0, device="cpu") -> AppendCase:
    """A pool as make_case builds it, plus the new tokens' hidden vectors and the two weights."""
    case = make_case(name, seq_lens, Tq=Tq, causal=True, shuffle=shuffle, spare_pages=spare_pages,
                     garbage=garbage, q_mode="none", seed=seed, device=device)
    h, w_dkv, w_kr = append_inputs(len(seq_lens) * Tq, d_model, seed, device)
    return AppendCase(case=case, h=h, w_dkv=w_dkv, w_kr=w_kr)


def append_inputs(n_tokens: int, d_model: int = D_MODEL, seed: int = 0, device="cpu"):
    """The cache write's inputs (tensors k = 9, 10, 11 of the recipe): h [n_tokens, d_model],
    W^DKV [D_C, d_model], W^KR [D_R, d_model], all bf16."""
    h = _randn_bf16((n_tokens, d_model), 1.0, seed, 9, device)
    w_dkv = _randn_bf16((D_C, d_model), 1.0 / math.sqrt(d_model), seed, 10, device)
    w_kr = _randn_bf16((D_R, d_model), 1.0 / math.sqrt(d_model), seed, 11, device)
    return h, w_dkv, w_kr


# Cache-write workloads: one decode step's new tokens at the decode workloads' batches, and a prefill.
APPEND_WORKLOADS = {
    # batch 64, one new token each after 4095 cached (the batch-64, 4096-token decode step)
    "append_b64_l4096": dict(seq_lens=[4096] * 64, Tq=1),
    # batch 32, four new tokens each after 8192 cached (the fused causal workload's step)
    "append_b32_tq4": dict(seq_lens=[8192 + 4] * 32, Tq=4),
    # one 4096-token prompt written at once (the prefill form)
    "prefill_l4096": dict(seq_lens=[4096], Tq=4096),
}


def make_append_workload(name: str, seed: int = 0, device="cpu") -> AppendCase:
    return make_append_case(name, seed=seed, device=device, **APPEND_WORKLOADS[name])


@dataclass
class CompressCase:
    """A compressed cache write: n_blocks new rows per sequence, each merging m new tokens."""
    case: Case                      # the pool, block table, compressed lengths
    h: torch.Tensor                 # [B * n_blocks * m, d_model] bf16
    w_dkv: torch.Tensor
    w_kr: torch.Tensor
    w_z: torch.Tensor               # [D, d_model] bf16
    n_blocks: int
    m: int

    @property
    def n_tokens(self) -> int:
        return int(self.h.shape[0])

    @property
    def d_model(self) -> int:
        return int(self.h.shape[1])

    def weight_bytes(self) -> int:
        return 2 * D * self.d_model * 2


def make_compress_case(name: str, seq_lens: List[int], n_blocks: int, m: int, d_model: int = D_MODEL,
                       shuffle: bool = False, seed: int = 0, device="cpu") -> CompressCase:
    """seq_lens: compressed lengths, the n_blocks new rows included."""
    case = make_case(name, seq_lens, Tq=n_blocks, causal=True, shuffle=shuffle, q_mode="none", seed=seed,
                     device=device)
    h, w_dkv, w_kr = append_inputs(len(seq_lens) * n_blocks * m, d_model, seed, device)
    w_z = _randn_bf16((D, d_model), 1.0 / math.sqrt(d_model), seed, 12, device)
    return CompressCase(case=case, h=h, w_dkv=w_dkv, w_kr=w_kr, w_z=w_z, n_blocks=n_blocks, m=m)


# Compressed cache-write workloads: CSA's blocks of 4 and HCA's blocks of 128 (m from the page).
COMPRESS_WORKLOADS = {
    # 16 sequences, one new block of 4 tokens each (64 tokens), after 1023 compressed rows
    "compress_b16_m4": dict(seq_lens=[1024] * 16, n_blocks=1, m=4),
    # one sequence, one new block of 128 tokens, after 31 compressed rows
    "compress_b1_m128": dict(seq_lens=[32], n_blocks=1, m=128),
}


def make_compress_workload(name: str, seed: int = 0, device="cpu") -> CompressCase:
    return make_compress_case(name, seed=seed, device=device, **COMPRESS_WORKLOADS[name])


D_IDX = 128  # index vector width of the indexer workloads (the pages give none)


@dataclass
class SparseCase:
    """An indexer decode: a decode case plus the paged index cache and the index queries."""
    case: Case                      # pool, block table, lengths, q_abs
    idx_pool: torch.Tensor          # [num_pages, PAGE, d_idx] bf16
    q_idx: torch.Tensor             # [B, d_idx] bf16
    k: int
    idx_codes: Optional[torch.Tensor] = None  # [num_pages, PAGE, d_idx] uint8 (E4M3 codes)
    idx_scale: Optional[torch.Tensor] = None  # [num_pages, PAGE] float32

    @property
    def d_idx(self) -> int:
        return int(self.idx_pool.shape[2])

    def index_bytes(self, e4m3: bool = False) -> int:
        """Bytes of index cache one step reads (each visible token's vector once; in E4M3, its
        codes and its scale)."""
        per = self.d_idx + 4 if e4m3 else self.d_idx * 2
        return int(self.case.seq_lens.to(torch.int64).sum()) * per

    def selected_bytes(self) -> int:
        """Bytes of latent cache rows the selection gathers: min(k, L_b) rows per sequence."""
        return int(self.case.seq_lens.clamp(max=self.k).to(torch.int64).sum()) * D * 2


def make_sparse_case(name: str, seq_lens: List[int], k: int, d_idx: int = D_IDX, ties: bool = False,
                     shuffle: bool = False, spare_pages: int = 0, garbage: Optional[str] = None,
                     peaked_frac: float = 0.0, e4m3: bool = False, seed: int = 0, device="cpu") -> SparseCase:
    case = make_case(name, seq_lens, Tq=1, causal=False, shuffle=shuffle, spare_pages=spare_pages,
                     garbage=garbage, peaked_frac=peaked_frac, q_mode="abs", seed=seed, device=device)
    shape = (case.num_pages, PAGE, d_idx)
    if ties:
        idx = torch.randint(-2, 3, shape, generator=_gen(seed, 13, device), device=device).to(torch.bfloat16)
        q_idx = torch.randint(-2, 3, (case.B, d_idx), generator=_gen(seed, 14, device), device=device)
        q_idx = q_idx.to(torch.bfloat16)
    else:
        idx = _randn_bf16(shape, 1.0 / math.sqrt(d_idx), seed, 13, device)
        q_idx = _randn_bf16((case.B, d_idx), 1.0, seed, 14, device)
    sc = SparseCase(case=case, idx_pool=idx, q_idx=q_idx, k=int(k))
    if e4m3:
        v = idx.float()
        scale = (v.abs().amax(dim=2) / 448.0).clamp_min(2.0 ** -100)
        sc.idx_codes = (v / scale[..., None]).to(torch.float8_e4m3fn).view(torch.uint8).contiguous()
        sc.idx_scale = scale.contiguous()
    return sc


# Indexer decode workloads: the 128K-token batch with the page's top-k of 512.
SPARSE_WORKLOADS = {
    # batch 8 x 131072 tokens (1% of rows peaked, as the dense 128K workload), top 512 by a
    # 128-wide index vector per token
    "sparse_b8_l128k_k512": dict(seq_lens=[131072] * 8, k=512, peaked_frac=0.01),
}


def make_sparse_workload(name: str, seed: int = 0, device="cpu", e4m3: bool = False) -> SparseCase:
    return make_sparse_case(name, seed=seed, device=device, e4m3=e4m3, **SPARSE_WORKLOADS[name])
