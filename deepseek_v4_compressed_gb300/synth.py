"""Seeded synthetic inputs for the decode path (shared by tests, smoke check and bench).

This module only draws numbers: normal and uniform float32 arrays, page tables
(random permutations of physical pages), sorted index sets and the workload
shapes.  It holds none of the method's arithmetic (no compression, no
quantisation, no dtype rounding); callers turn the float32 arrays into bf16 /
fp8 / cache bytes themselves.

Workloads (the decode shapes of the compressed-sparse-attention path):
  tiny_c4a       1 sequence, context 512, 8 query heads, 4 indexer heads,
                 top-k 32 over 128 compressed slots (the whole token stream
                 goes through the compressor), seed 0.
  c4a_32k        32 sequences, context 32768, 64 heads, indexer 64 x 128,
                 8192 compressed slots, top-k 512, seed 1.
  c128a_128k     64 sequences, context 131072, 64 heads, 1024 compressed
                 slots, top-k 512 given as sorted metadata, seed 2.
  mixed_60l      60-layer stack (swaonly / c4a / c128a), batch 16, context
                 65536, 64 heads, top-k 512, IndexCache freq 2, seed 3.
  long_c4a_1m    4 sequences, context 1,048,576, 128 heads, indexer 64 x 128,
                 262,144 compressed slots, top-k 2048, seed 4.
"""
from dataclasses import dataclass

import numpy as np

NOPE_DIM = 512
ROPE_DIM = 64
HEAD_DIM = NOPE_DIM + ROPE_DIM   # 576: latent + rope, one KV head
IDX_DIM = 128
WINDOW = 128
PAGE = 64


@dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    context: int
    n_heads: int
    idx_heads: int
    topk: int
    ratio: int          # 4 (c4a) or 128 (c128a); the mixed stack uses per-layer ratios
    seed: int
    layers: int = 1

    @property
    def n_compressed(self) -> int:
        return self.context // self.ratio


WORKLOADS = {
    "tiny_c4a": Workload("tiny_c4a", 1, 512, 8, 4, 32, 4, 0),
    "c4a_32k": Workload("c4a_32k", 32, 32768, 64, 64, 512, 4, 1),
    "c128a_128k": Workload("c128a_128k", 64, 131072, 64, 0, 512, 128, 2),
    "mixed_60l": Workload("mixed_60l", 16, 65536, 64, 64, 512, 4, 3, layers=60),
    "long_c4a_1m": Workload("long_c4a_1m", 4, 1048576, 128, 64, 2048, 4, 4),
}


def rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def normal(g: np.random.Generator, shape, std: float = 1.0) -> np.ndarray:
    return (g.standard_normal(shape, dtype=np.float32) * np.float32(std)).astype(np.float32)


def uniform(g: np.random.Generator, shape, lo: float = 0.0, hi: float = 1.0) -> np.ndarray:
    return g.uniform(lo, hi, size=shape).astype(np.float32)


def page_tables(g: np.random.Generator, n_seqs: int, pages_per_seq: int,
                extra_pages: int = 0) -> np.ndarray:
    """Each sequence gets distinct physical pages, a random permutation of the pool."""
    total = n_seqs * pages_per_seq + extra_pages
    perm = g.permutation(total).astype(np.int32)
    return perm[: n_seqs * pages_per_seq].reshape(n_seqs, pages_per_seq)


def sorted_sample(g: np.random.Generator, n: int, k: int) -> np.ndarray:
    """k distinct integers from [0, n), uniformly, sorted ascending."""
    k = min(k, n)
    return np.sort(g.choice(n, size=k, replace=False)).astype(np.int32)


def mixed_stack_ratios(n_layers: int = 60) -> np.ndarray:
    """Per-layer compress ratios of the 60-layer stack: layers 0 and 1 swaonly (1),
    c4a (4) at the 21 even layers 2..42, c128a (128) elsewhere."""
    r = np.full(n_layers, 128, np.int32)
    r[0:2] = 1
    r[2:43:2] = 4
    return r
