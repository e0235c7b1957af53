"""Host-side logic of bench.py that its roofline line depends on (no GPU needed): which
indexer kernel a shape launches, and when a committed DRAM-traffic figure may be reported."""
import json
import os
import re
import shutil

import bench

CSRC = os.path.join(bench.ROOT, "block_sparse_attention_indexer_gb300", "csrc")


def _dispatch_thresholds():
    # the library's own thresholds, read from its sources: rows >= kPrefillMinRows -> prefill
    # GEMM, rows > 8 -> speculative kernel, else the streaming decode kernel
    api = open(os.path.join(CSRC, "api.cu")).read()
    body = api[api.index("cudaError_t run_indexer("):]
    body = body[:body.index("\n}\n")]
    assert "launch_prefill_indexer" in body and "launch_spec_indexer" in body and "launch_indexer" in body
    spec_gt = int(re.search(r"if \(rows > (\d+)\) return launch_spec_indexer", body).group(1))
    consts = "".join(open(os.path.join(CSRC, f)).read() for f in os.listdir(CSRC) if f.endswith((".h", ".cuh", ".cu")))
    prefill_min = int(re.search(r"kPrefillMinRows\s*=\s*(\d+)", consts).group(1))
    return spec_gt, prefill_min


def test_indexer_kernel_for_matches_the_library_dispatch():
    spec_gt, prefill_min = _dispatch_thresholds()
    for groups in (1, 2, 4, 8):
        for q_len in range(1, 130):
            rows = q_len * groups
            want = ("prefill_indexer_kernel" if rows >= prefill_min else
                    "spec_indexer_kernel" if rows > spec_gt else "indexer_half_kernel")
            assert bench.indexer_kernel_for(q_len, groups) == want, (q_len, groups)


def test_every_timed_kernel_has_its_sources_listed():
    for kernel, files in bench.KERNEL_SOURCES.items():
        assert files, kernel
        for f in files:
            assert os.path.exists(os.path.join(CSRC, f)), (kernel, f)
        src = "".join(open(os.path.join(CSRC, f)).read() for f in files if f.endswith(".cu"))
        assert any("__global__" in line and re.search(r"\b%s\s*\(" % kernel, line) for line in src.splitlines()), kernel


def test_traffic_is_reported_only_for_unchanged_sources(tmp_path, monkeypatch):
    root = tmp_path / "repo"
    shutil.copytree(CSRC, root / "block_sparse_attention_indexer_gb300" / "csrc")
    (root / "profiles").mkdir()
    monkeypatch.setattr(bench, "ROOT", str(root))
    kernel = "indexer_half_kernel"
    entry = {kernel: {"source_hash": bench.kernel_source_hash(kernel),
                      "bytes_per_launch": {"ragged64_128k": 123}}}
    (root / "profiles" / "traffic.json").write_text(json.dumps(entry))
    assert bench.measured_traffic(kernel, "ragged64_128k") == 123
    assert bench.measured_traffic(kernel, "other_workload") is None
    assert bench.measured_traffic("spec_indexer_kernel", "ragged64_128k") is None
    # any edit to one of the kernel's sources drops the figure
    src = root / "block_sparse_attention_indexer_gb300" / "csrc" / bench.KERNEL_SOURCES[kernel][0]
    src.write_text(src.read_text() + "\n// edited\n")
    assert bench.measured_traffic(kernel, "ragged64_128k") is None


def test_cpu_sample_tracks_the_mean_context():
    """The CPU baseline's sample sequences sit at evenly spaced length quantiles, so their mean
    context is within a few percent of the workload's (the first sequences need not be)."""
    import numpy as np
    from workloads import synthetic as syn
    _, _, lens = syn.layout(syn.WORKLOADS["ragged64_128k"])
    picks = bench.representative_sequences(lens, 4)
    assert len(set(picks)) == 4
    assert abs(np.mean(lens[picks]) / np.mean(lens) - 1) < 0.05
    assert bench.representative_sequences(lens, 100) == sorted(range(len(lens)))
    assert bench.representative_sequences(np.array([5, 1, 3]), 1) == [2]


def test_decode_path_matches_the_library_dispatch():
    """bench.py's launch count per step follows msa_decode's own choice: block-major from
    kBlockMajorMinTokens query tokens, the attention selecting its own rows for at most
    kFusedSelectMaxRows rows of at most kFusedSelectMaxBlocks blocks, else the selection
    kernel; the thresholds are read from the library's sources."""
    consts = "".join(open(os.path.join(CSRC, f)).read() for f in os.listdir(CSRC) if f.endswith((".h", ".cuh", ".cu")))
    bm_min = int(re.search(r"kBlockMajorMinTokens\s*=\s*(\d+)", consts).group(1))
    max_rows = int(re.search(r"kFusedSelectMaxRows\s*=\s*(\d+)", consts).group(1))
    max_blocks = int(re.search(r"kFusedSelectMaxBlocks\s*=\s*(\d+)", consts).group(1))
    api = open(os.path.join(CSRC, "api.cu")).read()
    assert "rows_tg(batch, cfg) <= kFusedSelectMaxRows" in api and "batch->max_blocks <= kFusedSelectMaxBlocks" in api
    for batch in (1, 8, 32, 33, 64):
        for q_len in (1, 2, 8, 63, 64, 100):
            for mb in (32, max_blocks, max_blocks + 1, 1024):
                form, n = bench.decode_path(batch, q_len, 4, mb)
                if q_len >= bm_min:
                    assert n == 7 and form.startswith("block-major")
                elif batch * q_len * 4 <= max_rows and mb <= max_blocks:
                    assert n == 3
                else:
                    assert n == 4
