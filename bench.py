"""Benchmark of fused MSA decode (indexer -> top-16 select -> sparse attention) on GB300.

python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

One step = one msa_decode call over the whole batch of the workload (every row of the hot
path: block scores of the full context, selection, attention, split merge), inputs
resident in HBM.  Prints ONE JSON line (rank 0).  Under torchrun each rank runs its own
replica of the workload on its own GPU (weak scaling, no collective on the data path);
the timing is the max over ranks.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "MSA decode queries/s and achieved HBM GB/s (vs ~8 TB/s) at 128K ctx, 1 GB300"
FALLBACK_HBM_GBS = 6800.0
L2_FLUSH_BYTES = 512 << 20       # > 2x the 129 MB L2


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


FALLBACK_BF16_TFLOPS = 1900.0


def measured_tensor_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except Exception:
        return FALLBACK_BF16_TFLOPS, "fallback"


KERNEL_SOURCES = {
    "indexer_half_kernel": ["indexer.cu", "indexer_tile.cuh", "msa_device.cuh", "msa_kernels.h"],
    "spec_indexer_kernel": ["spec_indexer.cu", "msa_device.cuh", "msa_kernels.h", "umma.cuh"],
    "prefill_indexer_kernel": ["prefill.cu", "msa_device.cuh", "msa_kernels.h", "umma.cuh"],
    "bm_attn_kernel": ["prefill_attn.cu", "msa_device.cuh", "msa_kernels.h", "umma.cuh"],
    "attention_kernel": ["attention.cu", "attention_team.cuh", "attention_tile.cuh", "msa_device.cuh", "msa_kernels.h"],
}


def indexer_kernel_for(q_len: int, groups: int) -> str:
    """The indexer kernel msa_indexer_scores launches for T query tokens x G groups per sequence."""
    rows = q_len * groups
    if rows <= 8:
        return "indexer_half_kernel"
    return "spec_indexer_kernel" if rows < 64 else "prefill_indexer_kernel"


def decode_path(batch: int, q_len: int, groups: int, max_blocks: int):
    """The attention form msa_decode takes and the kernels it launches per step.

    From 64 query tokens on: the block-major attention (CSR count with the f16 queries beside
    it, scan and scatter, tcgen05 block attention, log-sum-exp merge) after the indexer and the
    selection.
    A small batch (at most 128 token x group rows of at most 256 blocks): the indexer, the
    attention whose producers select their rows, and the merge.  Otherwise the indexer, the
    selection, the team attention and its merge.
    """
    if q_len >= 64:
        return "block-major (K-to-Q CSR, tcgen05)", 7
    if batch * q_len * groups <= 128 and max_blocks <= 256:
        return "query-major teams (mma.sync), selection in the attention's producers", 3
    return "query-major teams (mma.sync)", 4

def kernel_source_hash(kernel: str) -> str:
    import hashlib
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "block_sparse_attention_indexer_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def step_distribution(ms):
    """Median, p10, p90, minimum and maximum of the per-step device times (ms)."""
    import numpy as np
    a = np.asarray(ms, dtype=np.float64)
    return {"median": float(np.median(a)), "p10": float(np.percentile(a, 10)), "p90": float(np.percentile(a, 90)),
            "min": float(a.min()), "max": float(a.max()), "n": int(a.size)}


def measured_traffic(kernel: str, workload: str):
    """DRAM bytes (read + write) per launch from the committed ncu summary, or None when the
    kernel's sources changed since those counters were taken."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            entry = json.load(f)[kernel]
    except Exception:
        return None
    if entry.get("source_hash") != kernel_source_hash(kernel):
        return None
    return entry.get("bytes_per_launch", {}).get(workload)


class ClockSampler:
    """nvidia-smi SM clock / throttle-reason sampling during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def replica_workload(name: str, rank: int):
    """Rank r decodes its own replica of the named workload: same shapes, its own seed."""
    from workloads import synthetic as syn
    w0 = syn.WORKLOADS[name]
    return syn.Workload(**{**w0.__dict__, "seed": w0.seed + 7919 * rank})


def reduce_max(values, world_size: int, device=None):
    """Element-wise max of a list of floats over all ranks (the job's time is its slowest rank)."""
    if world_size <= 1:
        return list(values)
    import torch
    import torch.distributed as dist
    t = torch.tensor(list(values), dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def representative_sequences(lens, n: int):
    """n sequences at evenly spaced quantiles of the context lengths (the (i + 1/2) / n-th
    shortest, i < n), so that the sample's mean length tracks the workload's."""
    import numpy as np
    order = np.argsort(np.asarray(lens), kind="stable")
    n = min(n, len(order))
    return sorted(int(order[int((i + 0.5) * len(order) / n)]) for i in range(n))


class OracleSample:
    """The CPU oracle on a bounded sample of a workload: a few sequences at evenly spaced
    quantiles of its context lengths, all their query tokens (the last 64 for prefill),
    caches quantised once before any timing."""

    def __init__(self, workload_name: str, n_seqs: int, rank_seed_offset: int = 0):
        from oracle import cache as OC
        from workloads import synthetic as syn

        w = syn.WORKLOADS[workload_name]
        self.w = syn.Workload(**{**w.__dict__, "seed": w.seed + rank_seed_offset})
        _, self.table, self.lens = syn.layout(self.w)
        self.seqs = representative_sequences(self.lens, n_seqs)
        self.cache, _, _, _ = OC.build_cache(self.w, self.lens, self.seqs, threads=os.cpu_count() or 1)
        self.q, self.qi = OC.encode_queries(self.w, self.seqs)
        T = self.w.q_len
        self.tokens = list(range(T)) if T <= 64 else list(range(T - 64, T))

    def run_one(self, b: int) -> int:
        import numpy as np
        from oracle import msa as OM

        w, T = self.w, self.w.q_len
        s = OM.block_scores(self.qi, self.cache[4], self.cache[5], self.table, self.lens, tokens=self.tokens,
                            sequences=[b])
        sel = np.full((w.batch, T, 4, 16), -1, np.int32)
        for t in self.tokens:
            for g in range(4):
                sel[b, t, g] = OM.select_row(s[b, t, g], int(self.lens[b]) - T + t)
        OM.sparse_attention(self.q, *self.cache[:4], self.table, self.lens, sel, w.heads_per_group,
                            tokens=self.tokens, sequences=[b])
        return len(self.tokens)

    def timed(self, budget_s: float):
        """Runs whole sequences of the sample (cycling) until budget_s; (queries/s, info)."""
        t_total, rows, done = 0.0, 0, []
        k = 0
        while t_total < budget_s or len(done) % len(self.seqs) != 0:  # whole cycles of the sample
            b = self.seqs[k % len(self.seqs)]
            t0 = time.perf_counter()
            rows += self.run_one(b)
            t_total += time.perf_counter() - t0
            done.append(b)
            k += 1
        return rows / t_total, {"sequences": sorted(set(done)), "sequence_runs": len(done), "query_rows": rows,
                                "seconds": round(t_total, 3)}


def run_reference(args):
    ws, rank, _ = dist_env()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")
        if rank != 0:
            dist.barrier()
            dist.destroy_process_group()
            return
    from workloads import synthetic as syn
    w = syn.WORKLOADS[args.workload]
    sample = OracleSample(args.workload, n_seqs=4)
    per_step = max(0.5, args.ref_budget / (args.steps + args.warmup))
    for _ in range(args.warmup):
        sample.timed(per_step)
    vals, info = [], None
    for _ in range(args.steps):
        v, info = sample.timed(per_step)
        vals.append(v)
    value = statistics.median(vals)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "queries/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * w.batch * w.q_len / value,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "batch": w.batch, "q_len": w.q_len, "heads": w.num_heads,
                       "kv_groups": 4, "head_dim": 128, "top_k": 16, "block": 128},
            "cpu_baseline": {"value": value, "unit": "queries/s", "cores": os.cpu_count(), "kind": "oracle",
                             "sample": f"float64 numpy oracle (BLAS threads) on whole sequences of the workload "
                                       f"(prebuilt cache), ~{per_step:.1f} s per step; last step {info}"},
            "e2e": {"value": value, "unit": "queries/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


def measure_workload(name, args, rank, dev, flush, peak, bf16_peak):
    """One more workload through msa_decode, measured like the headline: its own seeded
    replica, a CUDA graph of one msa_decode call replayed per step, L2 flushed between steps,
    CUDA events on the stream, clocks sampled around the timed region; then each stage alone
    for its kernel's roofline.  Frees its device memory before returning."""
    import numpy as np
    import torch

    import block_sparse_attention_indexer_gb300 as msa
    from oracle import msa as OM  # byte accounting of the oracle (host arithmetic, not the GPU path)
    from workloads import device

    w = replica_workload(name, rank)
    t0 = time.perf_counter()
    dw = device.upload(w)
    setup_s = time.perf_counter() - t0
    B, T, H = w.batch, w.q_len, w.num_heads
    out = torch.zeros(B, T, H, 128, dtype=torch.bfloat16, device=dev)
    lse = torch.zeros(B, T, H, dtype=torch.float32, device=dev)
    sel = torch.zeros(B, T, 4, 16, dtype=torch.int32, device=dev)
    wsp = msa.alloc_workspace(msa.MSA_OP_DECODE, dw.cfg, dw.batch, device=dev)
    scores = torch.empty(B, T, 4, dw.batch.max_blocks, dtype=torch.float32, device=dev)
    ws_idx = msa.alloc_workspace(msa.MSA_OP_INDEXER_SCORES, dw.cfg, dw.batch, device=dev)
    ws_att = msa.alloc_workspace(msa.MSA_OP_SPARSE_ATTN, dw.cfg, dw.batch, device=dev)
    stream = torch.cuda.current_stream()

    def graphed(fn):
        if args.no_graph:
            return fn
        fn()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        torch.cuda.synchronize()
        return g.replay

    def timed(fn, n, dist=None):
        run = graphed(fn)
        for _ in range(args.warmup):
            run()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        for i, (a, b) in enumerate(ev):
            flush.fill_(i & 0xFF)
            a.record(stream)
            run()
            b.record(stream)
        torch.cuda.synchronize()
        ms_list = [a.elapsed_time(b) for a, b in ev]
        if dist is not None:
            dist.extend(ms_list)
        return statistics.mean(ms_list)

    clocks = ClockSampler(dev.index if dev.index is not None else 0)
    clocks.start()
    time.sleep(0.3)
    step_list = []
    ms = timed(lambda: msa.msa_decode(dw.cfg, dw.cache, dw.batch, dw.q, dw.qi, out, lse, sel, wsp, None), args.steps,
               step_list)
    idx_ms = timed(lambda: msa.msa_indexer_scores(dw.cfg, dw.cache, dw.batch, dw.qi, scores, ws_idx, None),
                   args.steps)
    sel_ms = timed(lambda: msa.msa_select_blocks(dw.cfg, dw.batch, scores, sel, None), args.steps)
    att_ms = timed(lambda: msa.msa_sparse_attn_decode(dw.cfg, dw.cache, dw.batch, dw.q, sel, out, lse, ws_att, None),
                   args.steps)
    clk = clocks.stop()
    assert msa.msa_read_device_error(wsp) == 0

    sel_h = sel.cpu().numpy()
    idx_bytes, kv_bytes = OM.decode_step_bytes(dw.lens, sel_h)
    queries = B * T
    step_gbs = (idx_bytes + kv_bytes) / (ms / 1e3) / 1e9
    pos = dw.lens[:, None] - T + np.arange(T)[None, :]
    vis = np.clip(pos[:, :, None, None] - 128 * sel_h.astype(np.int64) + 1, 0, 128) * (sel_h >= 0)
    att_flops = 4.0 * 128 * (H // 4) * float(np.sum(vis))
    idx_kernel = indexer_kernel_for(T, 4)
    form, n_launch = decode_path(B, T, 4, dw.batch.max_blocks)
    if idx_kernel == "prefill_indexer_kernel":
        idx_flops = 2.0 * 128 * 4 * float(np.sum(pos + 1))
        tf = idx_flops / (idx_ms / 1e3) / 1e12
        roof = {"bound": "tensor", "kernel": idx_kernel, "achieved": tf, "peak": bf16_peak, "unit": "TFLOP/s",
                "frac": tf / bf16_peak, "algorithmic_flops": idx_flops, "traffic": measured_traffic(idx_kernel, name)}
    else:
        gbs = idx_bytes / (idx_ms / 1e3) / 1e9
        roof = {"bound": "hbm", "kernel": idx_kernel, "achieved": gbs, "peak": peak, "unit": "GB/s",
                "frac": gbs / peak, "algorithmic_bytes": idx_bytes, "traffic": measured_traffic(idx_kernel, name)}
    res = {"config": {"batch": B, "q_len": T, "heads": H, "mean_ctx": float(np.mean(dw.lens)),
                      "tokens_in_cache": int(np.sum(dw.lens))},
           "ms_per_step": ms, "step_ms_dist": step_distribution(step_list), "queries_per_s": queries / (ms / 1e3),
           "step_roofline": {"bound": "hbm", "algorithmic_bytes": idx_bytes + kv_bytes, "achieved": step_gbs,
                             "unit": "GB/s", "frac": step_gbs / peak, "frac_of_8tbs": step_gbs / 8000.0},
           "roofline": roof,
           "stages_ms": {"indexer": idx_ms, "select": sel_ms, "attention": att_ms,
                         "attention_gbs": kv_bytes / (att_ms / 1e3) / 1e9, "attention_bytes": kv_bytes},
           "attention_form": form,
           "attention_tflops": att_flops / (att_ms / 1e3) / 1e12,
           "launches_per_step": n_launch,
           "clocks": clk, "setup_s": round(setup_s, 1)}
    del dw, out, lse, sel, wsp, scores, ws_idx, ws_att
    torch.cuda.empty_cache()
    return res


def run_ours(args):
    import numpy as np
    import torch

    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    import block_sparse_attention_indexer_gb300 as msa
    from oracle import msa as OM  # byte accounting of the oracle (host arithmetic, not the GPU path)
    from workloads import device
    from workloads import synthetic as syn

    w0 = syn.WORKLOADS[args.workload]
    w = replica_workload(args.workload, rank)      # weak scaling: one replica per rank
    t_setup = time.perf_counter()
    dw = device.upload(w)
    setup_s = time.perf_counter() - t_setup
    B, T, H = w.batch, w.q_len, w.num_heads
    dev = torch.device("cuda", local)
    out = torch.zeros(B, T, H, 128, dtype=torch.bfloat16, device=dev)
    lse = torch.zeros(B, T, H, dtype=torch.float32, device=dev)
    sel = torch.zeros(B, T, 4, 16, dtype=torch.int32, device=dev)
    wsp = msa.alloc_workspace(msa.MSA_OP_DECODE, dw.cfg, dw.batch, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def step():
        # stream=None: the binding uses torch's current stream (the capture stream when graphed)
        msa.msa_decode(dw.cfg, dw.cache, dw.batch, dw.q, dw.qi, out, lse, sel, wsp, None)

    def graphed(fn):
        """fn captured once into a CUDA graph (the launches are capture-safe: no host sync, no
        allocation, fixed grids); returns the replay callable, or fn itself with --no-graph."""
        if args.no_graph:
            return fn
        fn()  # first call outside capture: per-device set-up (shared-memory limits)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        torch.cuda.synchronize()
        return g.replay

    step_run = graphed(step)
    for _ in range(args.warmup):
        step_run()
    torch.cuda.synchronize()
    assert msa.msa_read_device_error(wsp) == 0

    # ---- timed region: K steps, L2 flushed between steps (outside the events)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    clocks = ClockSampler(local)
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    wall0 = time.perf_counter()
    for i in range(args.steps):
        flush.fill_(i & 0xFF)
        starts[i].record(stream)
        step_run()
        ends[i].record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    if ws > 1:
        torch.distributed.barrier()
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]

    # ---- stage timing (same stream, same arguments) for the roofline of each kernel
    scores = torch.empty(B, T, 4, dw.batch.max_blocks, dtype=torch.float32, device=dev)
    ws_idx = msa.alloc_workspace(msa.MSA_OP_INDEXER_SCORES, dw.cfg, dw.batch, device=dev)
    ws_att = msa.alloc_workspace(msa.MSA_OP_SPARSE_ATTN, dw.cfg, dw.batch, device=dev)

    def timed(fn, n):
        run = graphed(fn)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        for a, b in ev:
            flush.fill_(1)
            a.record(stream)
            run()
            b.record(stream)
        torch.cuda.synchronize()
        return statistics.mean(a.elapsed_time(b) for a, b in ev)

    idx_ms = timed(lambda: msa.msa_indexer_scores(dw.cfg, dw.cache, dw.batch, dw.qi, scores, ws_idx, None),
                   args.steps)
    sel_ms = timed(lambda: msa.msa_select_blocks(dw.cfg, dw.batch, scores, sel, None), args.steps)
    att_ms = timed(lambda: msa.msa_sparse_attn_decode(dw.cfg, dw.cache, dw.batch, dw.q, sel, out, lse, ws_att,
                                                      None), args.steps)
    clk = clocks.stop()

    # ---- end to end through the public API with host buffers (pinned), every step:
    # H2D of the step's queries, index queries, block table and lengths, staged the way a
    # serving loop stages them: one pinned host buffer, one copy into one device buffer whose
    # 256-byte aligned views are the call's arguments; D2H of the output
    src = (dw.q, dw.qi, dw.batch.block_table, dw.batch.seq_lens)
    offs, off = [], 0
    for s_ in src:
        offs.append(off)
        off += (s_.numel() * s_.element_size() + 255) // 256 * 256
    h_stage = torch.empty(off, dtype=torch.uint8).pin_memory()
    d_stage = torch.empty(off, dtype=torch.uint8, device=dev)

    def view(buf, o, like):
        n = like.numel() * like.element_size()
        return buf[o:o + n].view(like.dtype).view(like.shape)

    for s_, o in zip(src, offs):
        view(h_stage, o, s_).copy_(s_.cpu())
    d_q, d_qi, d_table, d_lens = (view(d_stage, o, s_) for s_, o in zip(src, offs))
    h_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    e_batch = msa.Batch(d_table, d_lens, T)
    h2d = h_stage.numel()  # the bytes the copy moves: the inputs plus their 256-byte alignment padding
    d2h = h_out.numel() * h_out.element_size()

    def e2e_step():
        d_stage.copy_(h_stage, non_blocking=True)
        msa.msa_decode(dw.cfg, dw.cache, e_batch, d_q, d_qi, out, lse, None, wsp, None)  # current stream
        h_out.copy_(out, non_blocking=True)

    # the step as a serving loop runs it: one CUDA graph of the copies in, the msa_decode call
    # and the copy out, replayed per step (eager launches with --no-graph)
    e2e_run = graphed(e2e_step)
    for _ in range(args.warmup):
        e2e_run()
    torch.cuda.synchronize()
    e2e_times = []
    for i in range(args.steps):
        flush.fill_(i & 0xFF)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        e2e_run()
        torch.cuda.current_stream().synchronize()
        e2e_times.append(time.perf_counter() - t0)
    assert msa.msa_read_device_error(wsp) == 0

    # ---- the NVFP4 cache write (quantise + paged insert, msa_nvfp4_insert): the K rows of a
    # 65,536-token prefill (4 KV heads x 128 dims, float32, N(0, 1)) into a scratch pool of
    # shuffled pages; HBM bytes = float32 in + slots + E2M1 codes and E4M3 scales out
    ins_tokens, ins_rows = 65536, 4
    ins_pages = ins_tokens // 128
    gen = torch.Generator(device=dev)
    gen.manual_seed(1000 + ins_tokens)
    ins_x = torch.randn(ins_tokens, ins_rows, 128, generator=gen, device=dev)
    ins_perm = torch.randperm(ins_pages, generator=gen, device=dev)
    tok_idx = torch.arange(ins_tokens, device=dev)
    ins_slots = (ins_perm[tok_idx // 128] * 128 + tok_idx % 128).to(torch.int64)
    ins_data = torch.empty(ins_pages, ins_rows, 128, 64, dtype=torch.uint8, device=dev)
    ins_scale = torch.empty(ins_pages, ins_rows, 128, 8, dtype=torch.uint8, device=dev)
    ins_ms = timed(lambda: msa.msa_nvfp4_insert(ins_x, ins_slots, ins_data, ins_scale, 128, None), args.steps)
    ins_bytes = (ins_x.numel() * 4 + ins_slots.numel() * 8 + ins_data.numel() + ins_scale.numel())

    # ---- the other workloads (same process, same L2 flush and clock sampling), each freed after
    peak_gbs, _ = measured_peaks()
    bf16_tf, _ = measured_tensor_peak()
    extra = {}
    if not args.headline_only:
        del ins_x, ins_slots, ins_data, ins_scale, ins_perm, tok_idx
        for name in [n for n in syn.WORKLOADS if n != w0.name]:
            extra[name] = measure_workload(name, args, rank, dev, flush, peak_gbs, bf16_tf)

    # ---- aggregate over ranks (max time)
    ms_step = statistics.mean(step_ms)
    e2e_s = statistics.mean(e2e_times)
    ms_step, e2e_s, idx_ms, att_ms, ins_ms = reduce_max([ms_step, e2e_s, idx_ms, att_ms, ins_ms], ws, dev)
    if rank != 0:
        torch.distributed.destroy_process_group()
        return

    peak, peak_kind = measured_peaks()
    sel_h = sel.cpu().numpy()
    idx_bytes, kv_bytes = OM.decode_step_bytes(dw.lens, sel_h)
    queries = B * T
    value = ws * queries / (ms_step / 1e3)
    idx_gbs = idx_bytes / (idx_ms / 1e3) / 1e9
    att_gbs = kv_bytes / (att_ms / 1e3) / 1e9
    step_gbs = (idx_bytes + kv_bytes) / (ms_step / 1e3) / 1e9
    # the block-major form's counter memset is not a kernel
    form, launches_per_step = decode_path(B, T, 4, dw.batch.max_blocks)
    # attention FLOPs: QK and PV, 2 * 128 each, per (query head, visible selected key)
    pos_bt = dw.lens[:, None] - T + np.arange(T)[None, :]
    vis = np.clip(pos_bt[:, :, None, None] - 128 * sel_h.astype(np.int64) + 1, 0, 128) * (sel_h >= 0)
    att_flops = 4.0 * 128 * (H // 4) * float(np.sum(vis))
    idx_kernel = indexer_kernel_for(T, 4)
    traffic = measured_traffic(idx_kernel, w.name)
    if idx_kernel == "prefill_indexer_kernel":
        # the long-chunk indexer is a dense causal GEMM: tensor-pipe bound, counted in FLOPs
        # (2 * 128 per visible (row, key) pair; whole-block work past the diagonal not counted)
        pos = dw.lens[:, None] - T + np.arange(T)[None, :]
        idx_flops = 2.0 * 128 * 4 * float(np.sum(pos + 1))
        tflops = idx_flops / (idx_ms / 1e3) / 1e12
        bf16_peak, bf16_kind = measured_tensor_peak()
        roofline = {"bound": "tensor", "kernel": idx_kernel, "achieved": tflops, "peak": bf16_peak,
                    "unit": "TFLOP/s", "frac": tflops / bf16_peak, "traffic": traffic,
                    "algorithmic_flops": idx_flops, "peak_kind": f"{bf16_kind} (bf16 burst; f16 runs at the same rate)"}
    else:
        roofline = {"bound": "hbm", "kernel": idx_kernel, "achieved": idx_gbs, "peak": peak, "unit": "GB/s",
                    "frac": idx_gbs / peak, "traffic": traffic, "algorithmic_bytes": idx_bytes,
                    "peak_kind": f"{peak_kind} (burst copy)"}
    line = {
        "metric": METRIC, "value": value, "unit": "queries/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "step_ms_dist": step_distribution(step_ms),
        "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f16", "accumulate": "f32", "operands": "NVFP4 cache and FP8 queries widened exactly to f16", "data": "synthetic",
        "config": {"workload": w.name, "batch": B, "q_len": T, "heads": H, "kv_groups": 4, "head_dim": 128,
                   "index_dim": 128, "top_k": 16, "block": 128, "mean_ctx": float(np.mean(dw.lens)),
                   "tokens_in_cache": int(np.sum(dw.lens)), "l2": "flushed between timed steps (512 MiB write)",
                   "launch": "eager" if args.no_graph else "cuda graph of one msa_decode call, replayed per step",
                   "parallelism": f"replicas x{ws}"},
        "achieved_hbm_gbs": step_gbs,
        "step_roofline": {"bound": "hbm", "algorithmic_bytes": idx_bytes + kv_bytes, "achieved": step_gbs,
                          "peak": peak, "unit": "GB/s", "frac": step_gbs / peak, "peak_kind": peak_kind,
                          "frac_of_8tbs": step_gbs / 8000.0},
        "roofline": roofline,
        "stages_ms": {"indexer": idx_ms, "select": sel_ms, "attention": att_ms,
                      "attention_gbs": att_gbs, "attention_bytes": kv_bytes},
        "attention_form": form,
        "attention_tflops": att_flops / (att_ms / 1e3) / 1e12,
        "e2e": {"value": ws * queries / e2e_s, "unit": "queries/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "launch": "eager" if args.no_graph else
                "cuda graph: one H2D copy of the step's inputs staged in pinned memory, msa_decode, D2H copy of the output",
                "timing": "host wall clock from before the launch to after the stream synchronize"},
        "cache_insert": {"workload": f"{ins_tokens} tokens x {ins_rows} KV heads x 128 dims float32 -> NVFP4 "
                                     "pages (shuffled), msa_nvfp4_insert",
                         "ms": ins_ms, "bound": "hbm", "algorithmic_bytes": ins_bytes,
                         "achieved": ins_bytes / (ins_ms / 1e3) / 1e9, "peak": peak, "unit": "GB/s",
                         "frac": ins_bytes / (ins_ms / 1e3) / 1e9 / peak},
        "gpu_launches": launches_per_step * args.steps,
        "workloads": extra,
        "clocks": clk,
        "setup_s": round(setup_s, 1),
        "wall_s_timed_region": wall,
    }
    if ws == 1 and not args.no_cpu_baseline:
        sample = OracleSample(w0.name, n_seqs=4)
        v, info = sample.timed(args.cpu_budget)
        line["cpu_baseline"] = {"value": v, "unit": "queries/s", "cores": os.cpu_count(), "kind": "oracle",
                                "sample": f"float64 numpy oracle (BLAS threads) on whole sequences of the same "
                                          f"workload, cache prebuilt: {info}"}
    print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="ragged64_128k")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--ref-budget", type=float, default=120.0, help="seconds of oracle work for --impl reference")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-graph", action="store_true", help="launch eagerly instead of replaying a CUDA graph")
    ap.add_argument("--headline-only", action="store_true", help="skip the other workloads' measurements")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
