"""msa_sparse_attn_decode_noalloc: the sparse-attention stage for callers that cannot allocate
device memory (for example a plugin whose host application owns the whole device memory
pool, or code that must not allocate between decode steps).  Its scratch is the library's
own fixed 8 MiB device array instead of a caller workspace.

Checked through the C ABI against the regular msa_sparse_attn_decode (which takes a
workspace), on two calls in a row (the array keeps the previous call's contents), plus the
size bound.  This file is collected last so that a failure here does not stop the rest of
the suite from running first."""
import numpy as np
import pytest

from gpu_util import OM, OUT_MAX_ABS, OUT_MEAN_ABS, bf16_to_np, device_workload, need_gpu, oracle_inputs, syn, to_np

pytestmark = pytest.mark.gpu


def test_noalloc_matches_workspace_entry_point_twice():
    need_gpu()
    import torch
    import block_sparse_attention_indexer_gb300 as msa
    # 6 sequences x 2 tokens x 4 groups = 48 rows over ~450 teams: every row is cut by team
    # boundaries, so the scratch holds partial states
    w, lens = syn.custom("noalloc", 31, 6, 2, 8, [5000, 129, 20000, 300, 2048, 4096 + 3], shuffled=True)
    dw = device_workload(w, lens)
    cache, table, lens, q, qi = oracle_inputs(w, lens)
    sel = torch.from_numpy(OM.select_blocks(OM.block_scores(qi, cache[4], cache[5], table, lens), lens)).cuda()
    B, T, H = w.batch, w.q_len, w.num_heads

    out_ws = torch.zeros(B, T, H, 128, dtype=torch.bfloat16, device="cuda")
    lse_ws = torch.zeros(B, T, H, dtype=torch.float32, device="cuda")
    ws = msa.alloc_workspace(msa.MSA_OP_SPARSE_ATTN, dw.cfg, dw.batch)
    msa.msa_sparse_attn_decode(dw.cfg, dw.cache, dw.batch, dw.q, sel, out_ws, lse_ws, ws)
    torch.cuda.synchronize()
    ref_o, ref_l = bf16_to_np(out_ws), to_np(lse_ws)

    for _ in range(2):
        out = torch.full((B, T, H, 128), 9.0, dtype=torch.bfloat16, device="cuda")
        lse = torch.zeros(B, T, H, dtype=torch.float32, device="cuda")
        msa.msa_sparse_attn_decode_noalloc(dw.cfg, dw.cache, dw.batch, dw.q, sel, out, lse)
        torch.cuda.synchronize()
        err = np.abs(bf16_to_np(out) - ref_o)
        assert err.max() <= OUT_MAX_ABS and err.mean() <= OUT_MEAN_ABS
        assert np.allclose(to_np(lse), ref_l, rtol=1e-5, atol=1e-5)


def test_noalloc_scratch_covers_every_batch():
    need_gpu()
    import torch
    import block_sparse_attention_indexer_gb300 as msa
    # the attention's scratch does not grow with the batch, so the largest batch the ABI
    # accepts fits the 8 MiB array, for any group / head configuration
    for g, hg in [(4, 8), (8, 8), (1, 1)]:
        cfg = msa.Config(num_kv_groups=g, heads_per_group=hg)
        big = msa.Batch(torch.zeros(2048, 4, dtype=torch.int32, device="cuda"),
                        torch.full((2048,), 512, dtype=torch.int32, device="cuda"), 65535 // 2048)
        assert msa.msa_workspace_bytes(msa.MSA_OP_SPARSE_ATTN, cfg, big) <= 8 << 20
