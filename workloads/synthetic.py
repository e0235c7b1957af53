"""Seeded generators for the five MSA workloads.

The sizes follow the workloads the M3.1-Flash post describes for long-context agentic
decode ("vLLM liefert Day-0-Unterstützung für MiniMax-M3.1-Flash", §MSA-Grundlagen:
128-token blocks, top-16 blocks, 4 KV heads x 128 dims, one shared index-key head),
the speculative-decode verification shape of the M3 post ("MiniMax M3 x vLLM：百万
token 多模态推理的 Day-0 部署", §Decode Kernel 中的投机解码) and its chunked prefill
(§Prefill 执行).

Every value is drawn from a counter-based Philox stream keyed by
(workload seed, tensor kind, sequence, block), so that any block of any sequence can be
regenerated alone, in any order, on any machine, without drawing the rest.

Values: q, K, V and index keys are N(0, 1) float32; every index key of block n of
sequence b additionally gets the same offset vector o[b, n] ~ N(0, 2^2) (standard
deviation 2), so that block scores separate.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, Tuple

import numpy as np

BLOCK = 128          # tokens per KV block (the cache page size)
HEAD_DIM = 128       # D
INDEX_DIM = 128      # Di
NUM_KV_GROUPS = 4    # G
TOP_K = 16

# tensor kinds (part of the Philox key)
KIND_K, KIND_V, KIND_IDX, KIND_OFFSET, KIND_Q, KIND_QI, KIND_LENS, KIND_TABLE = range(8)


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    seed: int
    batch: int
    q_len: int                 # T, query tokens per sequence (already in the cache)
    heads_per_group: int       # Hg
    ctx: Tuple[int, int]       # context length range in tokens (inclusive), multiples of 128 when ragged
    ragged: bool               # context lengths drawn uniformly in ctx, rounded to 128
    shuffled_table: bool       # one shared page pool, random permutation split into rows
    offset_std: float = 2.0
    description: str = ""

    @property
    def num_heads(self) -> int:
        return NUM_KV_GROUPS * self.heads_per_group


WORKLOADS: Dict[str, Workload] = {
    "tiny": Workload("tiny", 1001, 1, 1, 4, (4096, 4096), False, False,
                     description="B1 T1 ctx 4,096 (32 blocks), 4 KV groups x 4 q heads"),
    "b8_32k": Workload("b8_32k", 1002, 8, 1, 8, (32768, 32768), False, False,
                       description="B8 T1 ctx 32,768 (256 blocks), 32 q heads, contiguous table"),
    "ragged64_128k": Workload("ragged64_128k", 1003, 64, 1, 8, (16384, 131072), True, True,
                              description="B64 T1 ctx uniform in [16K,128K] (x128), shuffled shared pool, 32 q heads"),
    "spec4_512k": Workload("spec4_512k", 1004, 4, 8, 8, (524288, 524288), False, False,
                           description="B4 T8 (1+7 draft tokens) ctx 524,288, per-token selection, 32 q heads"),
    "prefill_4k_on_64k": Workload("prefill_4k_on_64k", 1005, 1, 4096, 8, (69632, 69632), False, False,
                                  description="1 seq, 4,096 new tokens on a 65,536-token cache (69,632 = 544 blocks), 32 q heads"),
}


def _philox(seed: int, kind: int, b: int, n: int) -> np.random.Generator:
    key = np.array([(seed << 8) | kind, (b << 32) | n], dtype=np.uint64)
    return np.random.Generator(np.random.Philox(key=key))


def _normal(rng: np.random.Generator, shape) -> np.ndarray:
    return rng.standard_normal(size=shape, dtype=np.float32)


def seq_lens(w: Workload) -> np.ndarray:
    """Context length L_b of each sequence (tokens in the cache, including the T new ones)."""
    if not w.ragged:
        return np.full(w.batch, w.ctx[0], dtype=np.int32)
    rng = _philox(w.seed, KIND_LENS, 0, 0)
    lo, hi = w.ctx[0] // BLOCK, w.ctx[1] // BLOCK
    return (rng.integers(lo, hi + 1, size=w.batch) * BLOCK).astype(np.int32)


def layout(w: Workload, lens: np.ndarray | None = None):
    """Page pool size, block table [B, max_blocks] (int32, -1 past the end) and lens."""
    if lens is None:
        lens = seq_lens(w)
    nblocks = (lens.astype(np.int64) + BLOCK - 1) // BLOCK
    max_blocks = int(nblocks.max())
    num_pages = int(nblocks.sum())
    table = np.full((w.batch, max_blocks), -1, dtype=np.int32)
    if w.shuffled_table:
        perm = _philox(w.seed, KIND_TABLE, 0, 0).permutation(num_pages).astype(np.int32)
    else:
        perm = np.arange(num_pages, dtype=np.int32)
    start = 0
    for b in range(w.batch):
        table[b, : nblocks[b]] = perm[start: start + nblocks[b]]
        start += int(nblocks[b])
    return num_pages, table, lens


def gen_index_block_fp32(w: Workload, b: int, n: int) -> np.ndarray:
    """fp32 index keys of block n of sequence b, [128, Di], with the block's offset vector."""
    idx = _normal(_philox(w.seed, KIND_IDX, b, n), (BLOCK, INDEX_DIM))
    off = _normal(_philox(w.seed, KIND_OFFSET, b, n), (INDEX_DIM,)) * np.float32(w.offset_std)
    idx += off[None, :]
    return idx


def gen_kv_block_fp32(w: Workload, b: int, n: int):
    """fp32 K and V of block n of sequence b, each [128, G, D]."""
    k = _normal(_philox(w.seed, KIND_K, b, n), (BLOCK, NUM_KV_GROUPS, HEAD_DIM))
    v = _normal(_philox(w.seed, KIND_V, b, n), (BLOCK, NUM_KV_GROUPS, HEAD_DIM))
    return k, v


def gen_block_fp32(w: Workload, b: int, n: int):
    """fp32 values of block n of sequence b.

    Returns (k [128, G, D], v [128, G, D], idx [128, Di]); the index keys already carry the
    block's offset vector.  Tokens past the sequence end are generated too (they are never
    visible to any query).  Each tensor has its own stream, so the parts can be drawn alone
    (gen_index_block_fp32, gen_kv_block_fp32) with the same values.
    """
    k, v = gen_kv_block_fp32(w, b, n)
    return k, v, gen_index_block_fp32(w, b, n)


def gen_queries(w: Workload, b: int) -> np.ndarray:
    """fp32 attention queries of sequence b, [T, H, D]."""
    return _normal(_philox(w.seed, KIND_Q, b, 0), (w.q_len, w.num_heads, HEAD_DIM))


def gen_index_queries(w: Workload, b: int) -> np.ndarray:
    """fp32 index queries of sequence b, one per KV group, [T, G, Di]."""
    return _normal(_philox(w.seed, KIND_QI, b, 0), (w.q_len, NUM_KV_GROUPS, INDEX_DIM))


def custom(name: str, seed: int, batch: int, q_len: int, heads_per_group: int, lens, shuffled=False,
           offset_std: float = 2.0) -> Tuple[Workload, np.ndarray]:
    """A small ad-hoc workload with explicit lengths (tests: ragged tails, tiny contexts)."""
    lens = np.asarray(lens, dtype=np.int32)
    w = Workload(name, seed, batch, q_len, heads_per_group, (int(lens.min()), int(lens.max())), False,
                 shuffled, offset_std)
    return w, lens


def total_tokens(lens: np.ndarray) -> int:
    return int(np.asarray(lens, dtype=np.int64).sum())


def ceil_div(a: int, b: int) -> int:
    return -(-a // b)


__all__ = ["WORKLOADS", "Workload", "seq_lens", "layout", "gen_block_fp32", "gen_index_block_fp32",
           "gen_kv_block_fp32", "gen_queries",
           "gen_index_queries", "custom", "BLOCK", "HEAD_DIM", "INDEX_DIM", "NUM_KV_GROUPS", "TOP_K",
           "total_tokens", "ceil_div"]
