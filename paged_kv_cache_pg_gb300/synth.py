"""Seeded synthetic inputs for the paged KV-cache path.

This module holds no arithmetic of the method: it draws bf16 bit patterns
and page tables, and nothing else.  The CUDA path and the CPU oracle both
read what it draws, and each places the rows into its own caches.

bf16 values are the top 16 bits of float32 draws from N(0, 1) (truncation:
no rounding step is involved).  Page tables are random permutations of an
arena's page ids, dealt to the streams without overlap, or a reversed table
(the pages' check mode: each stream read through a reversed table of
n-position pages).
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import List, Sequence

import numpy as np


def normal_bf16(seed: int, shape: Sequence[int]) -> np.ndarray:
    """bf16 bit patterns (uint16) of N(0, 1) float32 draws, seeded."""
    rng = np.random.default_rng(seed)
    x = rng.standard_normal(tuple(shape), dtype=np.float32)
    return (x.view(np.uint32) >> 16).astype(np.uint16)


def scale_pow2(bits: np.ndarray, e) -> np.ndarray:
    """bf16 bit patterns times 2**e, exactly: a power of two moves the
    exponent only.  `e` is an int or an integer array broadcastable to `bits`.
    Raises if a nonzero result would leave the normal bf16 range."""
    x = (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    y = (x * np.exp2(np.asarray(e, np.float64))).astype(np.float32)
    a = np.abs(y)
    if not np.all((a == 0) | ((a >= 2.0 ** -126) & (a < 2.0 ** 127))):
        raise ValueError("scaled value outside the normal bf16 range")
    u = y.view(np.uint32)
    if np.any(u & 0xFFFF):
        raise ValueError("scaling was not exact")
    return (u >> 16).astype(np.uint16)


def pages_for(length: int, ptok: int) -> int:
    """Pages a stream of `length` positions occupies."""
    return -(-length // ptok)


def shuffled_tables(seed: int, n_pages: int, counts: Sequence[int]) -> List[np.ndarray]:
    """Deal a random permutation of the arena's pages to streams, no overlap."""
    if sum(counts) > n_pages:
        raise ValueError("streams need more pages than the arena holds")
    perm = np.random.default_rng(seed).permutation(n_pages).astype(np.int32)
    out, at = [], 0
    for c in counts:
        out.append(np.ascontiguousarray(perm[at:at + c]))
        at += c
    return out


def reversed_table(n: int, first: int = 0) -> np.ndarray:
    """Pages first+n-1 .. first: the last logical page sits lowest."""
    return np.arange(first + n - 1, first - 1, -1, dtype=np.int32)


@dataclass
class Stream:
    """Logical (contiguous, token-major) rows of one stream, all layers."""
    length: int
    k: np.ndarray       # [layers][T][Hkv][D]
    v: np.ndarray       # [layers][T][Hkv][D]
    ik: np.ndarray      # [layers][T][Di]   (empty when Di == 0)


def make_stream(seed: int, n_layers: int, length: int, n_kv_heads: int, head_dim: int,
                idx_dim: int) -> Stream:
    k = normal_bf16(seed * 1000 + 1, (n_layers, length, n_kv_heads, head_dim))
    v = normal_bf16(seed * 1000 + 2, (n_layers, length, n_kv_heads, head_dim))
    ik = normal_bf16(seed * 1000 + 3, (n_layers, length, idx_dim))
    return Stream(length, k, v, ik)


def queries(seed: int, n_tokens: int, n_q_heads: int, dim: int) -> np.ndarray:
    """Packed query rows [tokens][Hq][dim]."""
    return normal_bf16(seed * 1000 + 7, (n_tokens, n_q_heads, dim))


@dataclass
class Workload:
    """A synthetic workload shaped like one of the pages' cases."""
    name: str
    n_layers: int
    n_q_heads: int
    n_kv_heads: int
    lengths: List[int]              # positions cached per stream, before new tokens
    n_new: List[int]                # new tokens (queries) per stream
    page_sizes: List[int]
    head_dim: int = 256
    idx_dim: int = 128
    top_k: int = 0
    extra: dict = field(default_factory=dict)


# 1 layer, 1 stream, 4/1 heads, 64 cached positions, pages of 16, reversed table.
TINY = Workload("tiny paged decode", 1, 4, 1, [64], [0], [16])
# 4 streams shuffled through one arena, 1 new token each (stored, then attended).
MULTI = Workload("multi-stream paged decode", 13, 16, 2, [1000, 3000, 6000, 9000],
                 [1, 1, 1, 1], [16, 48, 128, 256, 512])
# 2 streams at 9000, pages of 128, top-64 of the pooled blocks.
SPARSE = Workload("block-sparse paged decode", 1, 16, 2, [9000, 9000], [0, 0], [128],
                  top_k=64)
# 512-query chunk appended to 31,000 cached positions, pages of 256.
PREFILL = Workload("chunked prefill", 1, 16, 2, [31000], [512], [256])
# 792 x 256 arena; 3 streams with 4-token draft windows, 1 stream in a 2048 chunk.
MIX = Workload("serving-shaped mix", 1, 16, 2, [9000, 24000, 40956, 16384], [4, 4, 4, 2048],
               [256], extra={"arena_pages": 792})
