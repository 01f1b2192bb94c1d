"""Cache-size arithmetic of the "DeepSeek-V2" explainer (Steps 2, 4 and 8).

TEST INFRASTRUCTURE ONLY.  The pages print the results of this arithmetic
(3.93 MB per token, ~515 GB for 131,072 tokens, 576 and 34,560 numbers,
56.9x, ~9.1 GB, 98.2%, 2.25 groups, 93.3%); the tests compare these
functions, and the C library's ``mla_cache_bytes``, against those printed
numbers (tests/golden/cache_arithmetic.json).
"""
from __future__ import annotations


def mha_numbers_per_token(heads: int = 128, d_head: int = 128, layers: int = 60) -> int:
    """Step 2: one key and one value per head per layer."""
    return 2 * heads * d_head * layers


def mla_numbers_per_token(d_c: int = 512, d_r: int = 64, layers: int = 60) -> int:
    """Step 8: latent note (d_c) plus the shared rotated key strip (d_r), per layer."""
    return (d_c + d_r) * layers


def cache_bytes(numbers_per_token: int, tokens: int, bytes_per_number: float = 2.0) -> float:
    """Steps 2 and 8: BF16 is two bytes per number."""
    return numbers_per_token * tokens * bytes_per_number


def gqa_equivalent_groups(d_c: int = 512, d_r: int = 64, d_head: int = 128) -> float:
    """Step 8: the MLA row costs as much as GQA with g groups: 2 * g * d_head = d_c + d_r."""
    return (d_c + d_r) / (2 * d_head)


def gqa_reduction(heads: int = 128, groups: int = 8) -> float:
    """Step 4: sharing one K/V pair per group cuts the cache by heads / groups."""
    return heads / groups


def reduction_fraction(new: float, old: float) -> float:
    """Step 8 audit: fraction of the old cache that is saved."""
    return 1.0 - new / old
