"""The failure path of the kernels' bounded waits, exercised on the GPU without a fault.

The streaming indexer is launched through the test hook msa_test_indexer_stall: its page
copies are withheld and every wait is capped at a few polls, so each warp's first wait on its
page ring runs out.  The kernel must return (no hang), set MSA_DEVERR_TIMEOUT in the
workspace error word, and leave the context usable: regular calls right after it, on the
same workspace, match the oracle."""
import numpy as np
import pytest

from gpu_util import (OC, OM, assert_out_close, assert_scores_close, bf16_to_np, device_workload, need_gpu,
                      oracle_inputs, score_bound, selection_diffs, syn, to_np)

pytestmark = pytest.mark.gpu


def _stalled_then_regular(spin_limit):
    import torch
    import block_sparse_attention_indexer_gb300 as msa
    w, lens = syn.custom("stall", 21, 3, 1, 8, [5000, 20000, 129], shuffled=True)
    dw = device_workload(w, lens)
    B = w.batch
    scores = torch.zeros(B, 1, 4, dw.batch.max_blocks, dtype=torch.float32, device="cuda")
    ws = msa.alloc_workspace(msa.MSA_OP_INDEXER_SCORES, dw.cfg, dw.batch)
    msa.msa_test_indexer_stall(dw.cfg, dw.cache, dw.batch, dw.qi, scores, ws, spin_limit)
    torch.cuda.synchronize()
    flags = msa.msa_read_device_error(ws)
    assert flags & msa.MSA_DEVERR_TIMEOUT, flags
    assert not flags & (msa.MSA_DEVERR_BAD_PAGE | msa.MSA_DEVERR_BAD_SEQLEN), flags

    # the same context and workspace, regular calls: oracle parity, no error
    msa.msa_clear_device_error(ws)
    scores.fill_(7.0)
    msa.msa_indexer_scores(dw.cfg, dw.cache, dw.batch, dw.qi, scores, ws)
    torch.cuda.synchronize()
    assert msa.msa_read_device_error(ws) == 0
    cache, table, lens, q, qi = oracle_inputs(w, lens)
    ref = OM.block_scores(qi, cache[4], cache[5], table, lens)
    bound = score_bound(qi, cache[4], cache[5], table, lens, table.shape[1])
    assert_scores_close(to_np(scores), ref, bound)

    out = torch.zeros(B, 1, w.num_heads, 128, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros(B, 1, w.num_heads, dtype=torch.float32, device="cuda")
    sel = torch.zeros(B, 1, 4, 16, dtype=torch.int32, device="cuda")
    wsd = msa.alloc_workspace(msa.MSA_OP_DECODE, dw.cfg, dw.batch)
    msa.msa_decode(dw.cfg, dw.cache, dw.batch, dw.q, dw.qi, out, lse, sel, wsd)
    torch.cuda.synchronize()
    assert msa.msa_read_device_error(wsd) == 0
    ref_sel = OM.select_blocks(ref, lens)
    diff = selection_diffs(to_np(sel), ref_sel, ref, lens, 1)
    out_ref, lse_ref = OM.sparse_attention(q, *cache[:4], table, lens, ref_sel, w.heads_per_group)
    mask = np.ones((B, 1), bool)
    for (b, t, g) in diff:
        mask[b, t] = False
    assert_out_close(bf16_to_np(out)[mask], out_ref[mask])


@pytest.mark.parametrize("spin_limit", [1, 64])
def test_indexer_wait_runs_out_and_context_survives(spin_limit):
    need_gpu()
    _stalled_then_regular(spin_limit)


def test_stall_hook_host_validation():
    need_gpu()
    import torch
    import block_sparse_attention_indexer_gb300 as msa
    w, lens = syn.custom("stallval", 22, 2, 4, 8, [3000, 3000])
    dw = device_workload(w, lens)
    scores = torch.zeros(2, 4, 4, dw.batch.max_blocks, dtype=torch.float32, device="cuda")
    ws = msa.alloc_workspace(msa.MSA_OP_INDEXER_SCORES, dw.cfg, dw.batch)
    # 4 tokens x 4 groups = 16 rows: not the streaming kernel
    with pytest.raises(msa.MsaError, match="UNSUPPORTED"):
        msa.msa_test_indexer_stall(dw.cfg, dw.cache, dw.batch, dw.qi, scores, ws, 64)
    b1 = msa.Batch(dw.batch.block_table, dw.batch.seq_lens, 1)
    with pytest.raises(msa.MsaError, match="UNSUPPORTED"):   # a zero limit would never wait
        msa.msa_test_indexer_stall(dw.cfg, dw.cache, b1, dw.qi[:, :1].contiguous(), scores[:, :1].contiguous(),
                                   ws, 0)
