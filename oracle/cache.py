"""Oracle-side construction of the quantised paged cache and the FP8 queries.

TEST INFRASTRUCTURE ONLY (see oracle/formats.py).  The oracle quantises the seeded fp32
workload with its own quantiser; it never reads bytes produced by the CUDA path.

Cache layout (one page = one 128-token block; byte order fixed by the design notes):
  idx_data  uint8 [P, 128, 64]     idx_scale uint8 [P, 128, 8]
  k_data    uint8 [P, G, 128, 64]  k_scale   uint8 [P, G, 128, 8]   (v_* alike)
"""
from __future__ import annotations

from typing import Iterable, Optional

import numpy as np

from workloads import synthetic as syn

from .formats import e4m3_encode, nvfp4_quantize


def empty_cache(num_pages: int, groups: int = syn.NUM_KV_GROUPS, dim: int = syn.HEAD_DIM,
                index_dim: int = syn.INDEX_DIM):
    z = np.zeros
    return (z((num_pages, groups, syn.BLOCK, dim // 2), np.uint8), z((num_pages, groups, syn.BLOCK, dim // 16), np.uint8),
            z((num_pages, groups, syn.BLOCK, dim // 2), np.uint8), z((num_pages, groups, syn.BLOCK, dim // 16), np.uint8),
            z((num_pages, syn.BLOCK, index_dim // 2), np.uint8), z((num_pages, syn.BLOCK, index_dim // 16), np.uint8))


def fill_kv_block(cache, page: int, k, v):
    k_data, k_scale, v_data, v_scale = cache[:4]
    d, s = nvfp4_quantize(k.transpose(1, 0, 2))        # [G, 128, D]
    k_data[page], k_scale[page] = d, s
    d, s = nvfp4_quantize(v.transpose(1, 0, 2))
    v_data[page], v_scale[page] = d, s


def fill_index_block(cache, page: int, idx):
    d, s = nvfp4_quantize(idx)
    cache[4][page], cache[5][page] = d, s


def fill_block(cache, page: int, k, v, idx):
    fill_kv_block(cache, page, k, v)
    fill_index_block(cache, page, idx)


def _run(jobs, fn, threads):
    if threads and len(jobs) > 64:
        from concurrent.futures import ThreadPoolExecutor
        with ThreadPoolExecutor(threads) as ex:
            list(ex.map(fn, jobs))
    else:
        for job in jobs:
            fn(job)


def _index_codes(args):
    """Worker of the process pool: NVFP4 codes of the index keys of a list of blocks."""
    w, blocks = args
    return [nvfp4_quantize(syn.gen_index_block_fp32(w, b, n)) for b, n in blocks]


def _fill_index_blocks_pool(cache, w, table, jobs, procs):
    """Index keys of many blocks through a pool of `procs` processes (the quantiser's small
    numpy steps hold the interpreter lock, so threads do not scale).  The pool starts with
    'spawn': no process is forked from one that may hold a CUDA context."""
    import multiprocessing as mp
    from concurrent.futures import ProcessPoolExecutor
    step = 256
    chunks = [jobs[i:i + step] for i in range(0, len(jobs), step)]
    with ProcessPoolExecutor(procs, mp_context=mp.get_context("spawn")) as ex:
        for chunk, codes in zip(chunks, ex.map(_index_codes, [(w, c) for c in chunks])):
            for (b, n), (d, s) in zip(chunk, codes):
                page = int(table[b, n])
                cache[4][page], cache[5][page] = d, s


def build_cache(w: syn.Workload, lens: Optional[np.ndarray] = None, sequences: Optional[Iterable[int]] = None,
                threads: int = 0, index_only: bool = False):
    """Quantise the workload's cache.  Only the pages of `sequences` (default: all) are
    filled; the others stay zero.  With index_only, K and V stay zero too (add_kv_blocks
    fills the blocks a check needs).  Returns (cache tuple, block_table, lens, num_pages)."""
    num_pages, table, lens = syn.layout(w, lens)
    cache = empty_cache(num_pages)
    seqs = range(w.batch) if sequences is None else list(sequences)
    jobs = [(b, n) for b in seqs for n in range(-(-int(lens[b]) // syn.BLOCK))]

    def one(job):
        b, n = job
        if index_only:
            fill_index_block(cache, int(table[b, n]), syn.gen_index_block_fp32(w, b, n))
        else:
            fill_block(cache, int(table[b, n]), *syn.gen_block_fp32(w, b, n))

    if index_only and threads and len(jobs) >= 4096:
        _fill_index_blocks_pool(cache, w, table, jobs, threads)
    else:
        _run(jobs, one, threads)
    return cache, table, lens, num_pages


def add_kv_blocks(cache, w: syn.Workload, table, blocks: Iterable, threads: int = 0):
    """Quantise K and V of the logical blocks (b, n) into their pages of a cache built with
    index_only (the attention of a check reads only its selected blocks)."""
    jobs = sorted({(int(b), int(n)) for b, n in blocks})

    def one(job):
        b, n = job
        fill_kv_block(cache, int(table[b, n]), *syn.gen_kv_block_fp32(w, b, n))

    _run(jobs, one, threads)


def encode_queries(w: syn.Workload, sequences: Optional[Iterable[int]] = None):
    """FP8 E4M3 codes of the attention queries [B, T, H, D] and index queries [B, T, G, Di]."""
    q = np.zeros((w.batch, w.q_len, w.num_heads, syn.HEAD_DIM), np.uint8)
    qi = np.zeros((w.batch, w.q_len, syn.NUM_KV_GROUPS, syn.INDEX_DIM), np.uint8)
    for b in (range(w.batch) if sequences is None else sequences):
        q[b] = e4m3_encode(syn.gen_queries(w, b))
        qi[b] = e4m3_encode(syn.gen_index_queries(w, b))
    return q, qi
