"""The failure path of the kernels' bounded waits, exercised on the GPU without a fault.

The streaming indexer and the team attention are launched through the test hooks
msa_test_indexer_stall and msa_test_attention_stall: their page copies are withheld (the
attention's slots armed for their bytes but never filled) and every wait is capped at a few
polls, so the waits run out with no copy in flight.  The kernels must return (no hang), set
MSA_DEVERR_TIMEOUT in the workspace error word, and leave the context usable: regular calls
right after them, on the same workspace, match the oracle."""
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


@pytest.mark.parametrize("spin_limit", [1, 64])
def test_attention_wait_runs_out_and_context_survives(spin_limit):
    """The team attention through msa_test_attention_stall: every page slot is armed but never
    filled, so the consumers' waits run out, then the producers'.  The launch returns with
    MSA_DEVERR_TIMEOUT set, and a regular attention call on the same context and workspace
    then matches the oracle."""
    need_gpu()
    import torch
    import block_sparse_attention_indexer_gb300 as msa
    w, lens = syn.custom("astall", 23, 3, 2, 8, [5000, 20000, 129], shuffled=True)
    dw = device_workload(w, lens)
    B, T, H = w.batch, w.q_len, w.num_heads
    cache, table, lens_o, q, qi = oracle_inputs(w, lens)
    ref_s = OM.block_scores(qi, cache[4], cache[5], table, lens_o)
    sel_np = OM.select_blocks(ref_s, lens_o)
    sel = torch.from_numpy(sel_np).cuda()
    out = torch.zeros(B, T, H, 128, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros(B, T, H, dtype=torch.float32, device="cuda")
    ws = msa.alloc_workspace(msa.MSA_OP_SPARSE_ATTN, dw.cfg, dw.batch)
    msa.msa_test_attention_stall(dw.cfg, dw.cache, dw.batch, dw.q, sel, out, lse, ws, spin_limit)
    torch.cuda.synchronize()
    flags = msa.msa_read_device_error(ws)
    assert flags & msa.MSA_DEVERR_TIMEOUT, flags
    assert not flags & (msa.MSA_DEVERR_BAD_PAGE | msa.MSA_DEVERR_BAD_SEQLEN), flags

    msa.msa_clear_device_error(ws)
    out.zero_()
    msa.msa_sparse_attn_decode(dw.cfg, dw.cache, dw.batch, dw.q, sel, out, lse, ws)
    torch.cuda.synchronize()
    assert msa.msa_read_device_error(ws) == 0
    out_ref, lse_ref = OM.sparse_attention(q, *cache[:4], table, lens_o, sel_np, w.heads_per_group)
    assert_out_close(bf16_to_np(out), out_ref)
    assert np.allclose(to_np(lse), lse_ref, rtol=1e-4, atol=1e-4)


def test_attention_stall_hook_host_validation():
    need_gpu()
    import torch
    import block_sparse_attention_indexer_gb300 as msa
    w, lens = syn.custom("astallval", 24, 2, 1, 8, [3000, 3000])
    dw = device_workload(w, lens)
    sel = torch.zeros(2, 1, 4, 16, dtype=torch.int32, device="cuda")
    out = torch.zeros(2, 1, w.num_heads, 128, dtype=torch.bfloat16, device="cuda")
    ws = msa.alloc_workspace(msa.MSA_OP_SPARSE_ATTN, dw.cfg, dw.batch)
    with pytest.raises(msa.MsaError, match="UNSUPPORTED"):   # a zero limit would never wait
        msa.msa_test_attention_stall(dw.cfg, dw.cache, dw.batch, dw.q, sel, out, None, ws, 0)
    with pytest.raises(msa.MsaError, match="WORKSPACE"):
        msa.msa_test_attention_stall(dw.cfg, dw.cache, dw.batch, dw.q, sel, out, None, ws[:100], 64)
