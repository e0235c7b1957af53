"""World-size-2 CPU ranks (gloo): the decode-context-parallel candidate exchange of the
indexer, and the bench's replica / max-over-ranks aggregation.

Decode context parallelism splits the indexer's context scan across GPUs: each scores all
index heads over its share of the pages and sends its local top-16 per head to the head's
owner, which merges them; the selection stays exact ("vLLM liefert Day-0-Unterstützung für
MiniMax-M3.1-Flash", §NVFP4-Indexer-DCP).  Here the ranks are CPU processes and the
exchange is a gloo all_gather of (score, block) candidate lists."""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _dcp_rank(rank, world, port, q):
    import torch.distributed as dist
    from oracle import msa as M
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    rng = np.random.default_rng(123)
    ok = True
    for _ in range(40):
        nb = int(rng.integers(2, 600))
        row = np.round(rng.standard_normal(nb) * 2, 1)        # ties across shards
        pos = int(rng.integers(0, nb * 128))
        cuts = np.linspace(0, nb, world + 1).astype(int)
        local = M.dcp_local_candidates(row, pos, int(cuts[rank]), int(cuts[rank + 1]))
        lists = [None] * world
        dist.all_gather_object(lists, local)
        merged = M.dcp_merge(lists, pos)
        ok &= bool(np.array_equal(merged, M.select_row(row, pos)))
    dist.destroy_process_group()
    q.put((rank, ok))


def _bench_rank(rank, world, port, q):
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w = bench.replica_workload("ragged64_128k", rank)
    vals = bench.reduce_max([1.0 + rank, 5.0 - rank], world)
    dist.destroy_process_group()
    q.put((rank, w.seed, vals))


def _spawn(fn, world=2):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=fn, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    return sorted(out)


def test_dcp_merge_across_two_cpu_ranks():
    res = _spawn(_dcp_rank)
    assert all(ok for _, ok in res)


def test_bench_replicas_and_max_reduction():
    res = _spawn(_bench_rank)
    (r0, s0, v0), (r1, s1, v1) = res
    assert s0 != s1                         # each rank decodes its own replica
    assert v0 == v1 == [2.0, 5.0]           # the job time is the slowest rank's
