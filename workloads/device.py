"""Puts a synthetic workload on the GPU through the library's public entry points.

The fp32 values come from workloads.synthetic (seeded, regenerable per block); this module
only stages them in pinned host memory, copies them to the device and calls the library's
own msa_nvfp4_insert / msa_fp8_quantize kernels to build the NVFP4 cache and the FP8
queries.  It holds no arithmetic of the method.  (The oracle never imports this module.)
"""
from __future__ import annotations

import dataclasses
import os
from concurrent.futures import ThreadPoolExecutor
from typing import Optional

import numpy as np
import torch

import block_sparse_attention_indexer_gb300 as msa

from . import synthetic as syn


@dataclasses.dataclass
class DeviceWorkload:
    w: syn.Workload
    cfg: msa.Config
    cache: msa.PagedCache
    batch: msa.Batch
    q: torch.Tensor          # uint8 E4M3 [B, T, H, D]
    qi: torch.Tensor         # uint8 E4M3 [B, T, G, Di]
    lens: np.ndarray
    table: np.ndarray
    num_pages: int


def _threads() -> int:
    return max(1, min(32, os.cpu_count() or 1))


def upload(w: syn.Workload, lens: Optional[np.ndarray] = None, device="cuda", blocks_per_chunk: int = 512,
           threads: Optional[int] = None) -> DeviceWorkload:
    num_pages, table, lens = syn.layout(w, lens)
    G, D, Di, BL = syn.NUM_KV_GROUPS, syn.HEAD_DIM, syn.INDEX_DIM, syn.BLOCK
    cfg = msa.Config(num_kv_groups=G, heads_per_group=w.heads_per_group)
    cache = msa.PagedCache(num_pages, G, D, Di, BL, device=device)
    jobs = [(b, n, int(table[b, n])) for b in range(w.batch) for n in range(-(-int(lens[b]) // BL))]
    nthreads = threads or _threads()
    stream = torch.cuda.current_stream()
    staging = []
    for _ in range(2):
        staging.append(dict(
            k=torch.empty(blocks_per_chunk * BL, G, D, dtype=torch.float32, pin_memory=True),
            v=torch.empty(blocks_per_chunk * BL, G, D, dtype=torch.float32, pin_memory=True),
            i=torch.empty(blocks_per_chunk * BL, 1, Di, dtype=torch.float32, pin_memory=True),
            s=torch.empty(blocks_per_chunk * BL, dtype=torch.int64, pin_memory=True),
            ev=None))
    dev = dict(k=torch.empty(blocks_per_chunk * BL, G, D, dtype=torch.float32, device=device),
               v=torch.empty(blocks_per_chunk * BL, G, D, dtype=torch.float32, device=device),
               i=torch.empty(blocks_per_chunk * BL, 1, Di, dtype=torch.float32, device=device),
               s=torch.empty(blocks_per_chunk * BL, dtype=torch.int64, device=device))
    with ThreadPoolExecutor(nthreads) as ex:
        for ci, start in enumerate(range(0, len(jobs), blocks_per_chunk)):
            chunk = jobs[start: start + blocks_per_chunk]
            st = staging[ci % 2]
            if st["ev"] is not None:
                st["ev"].synchronize()
            kh, vh, ih, sh = st["k"].numpy(), st["v"].numpy(), st["i"].numpy(), st["s"].numpy()

            def fill(j):
                b, n, page = chunk[j]
                k, v, idx = syn.gen_block_fp32(w, b, n)
                kh[j * BL:(j + 1) * BL] = k
                vh[j * BL:(j + 1) * BL] = v
                ih[j * BL:(j + 1) * BL, 0] = idx
                sh[j * BL:(j + 1) * BL] = page * BL + np.arange(BL)

            list(ex.map(fill, range(len(chunk))))
            m = len(chunk) * BL
            for key in ("k", "v", "i", "s"):
                dev[key][:m].copy_(st[key][:m], non_blocking=True)
            msa.msa_nvfp4_insert(dev["k"][:m], dev["s"][:m], cache.k_data, cache.k_scale, BL, stream)
            msa.msa_nvfp4_insert(dev["v"][:m], dev["s"][:m], cache.v_data, cache.v_scale, BL, stream)
            msa.msa_nvfp4_insert(dev["i"][:m], dev["s"][:m], cache.idx_data.view(num_pages, 1, BL, Di // 2),
                                 cache.idx_scale.view(num_pages, 1, BL, Di // 16), BL, stream)
            ev = torch.cuda.Event()
            ev.record(stream)
            st["ev"] = ev
    q32 = torch.from_numpy(np.stack([syn.gen_queries(w, b) for b in range(w.batch)])).to(device)
    qi32 = torch.from_numpy(np.stack([syn.gen_index_queries(w, b) for b in range(w.batch)])).to(device)
    q = torch.empty(q32.shape, dtype=torch.uint8, device=device)
    qi = torch.empty(qi32.shape, dtype=torch.uint8, device=device)
    msa.msa_fp8_quantize(q32, q)
    msa.msa_fp8_quantize(qi32, qi)
    batch = msa.Batch(torch.from_numpy(table).to(device), torch.from_numpy(lens.astype(np.int32)).to(device),
                      w.q_len)
    torch.cuda.synchronize()
    return DeviceWorkload(w, cfg, cache, batch, q, qi, lens, table, num_pages)
