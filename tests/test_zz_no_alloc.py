"""msa_sparse_attn_decode_noalloc: the sparse-attention stage for callers that cannot allocate
device memory (for example a plugin whose host application owns the whole device memory
pool, or code that must not allocate between decode steps).  Its scratch is the library's
own fixed 8 MiB device array instead of a caller workspace, and that array keeps whatever
the previous call left in it.

Checked through the C ABI against the float64 oracle and against the regular
msa_sparse_attn_decode (which takes a workspace):
  * two checked calls with a differently shaped call between them, so that the shared array
    holds other partial states when the second checked call starts;
  * the largest batch the ABI accepts, and a query chunk of 64 tokens (where the regular
    entry point switches to the block-major form and this one does not), on sampled rows;
  * its device error word: a bad block-table entry is reported, and the next clean call
    clears it.
This file is collected last so that a failure here does not stop the rest of the suite from
running first; every test builds its own inputs, so it also passes alone in a fresh process."""
import numpy as np
import pytest

from gpu_util import (OC, OM, OUT_MAX_ABS, OUT_MEAN_ABS, assert_out_close, bf16_to_np, device_workload, need_gpu,
                      oracle_inputs, syn, to_np)

pytestmark = pytest.mark.gpu


def _selection_all_blocks(lens, T, G=4):
    """Every row selects blocks 0 .. r (contexts of at most 16 blocks: the selection is forced)."""
    B = len(lens)
    sel = np.full((B, T, G, 16), -1, np.int32)
    for b in range(B):
        for t in range(T):
            r = (int(lens[b]) - T + t) // 128
            sel[b, t, :, :r + 1] = np.arange(r + 1)
    return sel


def _noalloc(dw, sel_dev, fill=9.0):
    import torch
    import block_sparse_attention_indexer_gb300 as msa
    w = dw.w
    B, T, H = w.batch, w.q_len, w.num_heads
    out = torch.full((B, T, H, 128), fill, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros(B, T, H, dtype=torch.float32, device="cuda")
    msa.msa_sparse_attn_decode_noalloc(dw.cfg, dw.cache, dw.batch, dw.q, sel_dev, out, lse)
    torch.cuda.synchronize()
    return bf16_to_np(out), to_np(lse)


def test_noalloc_matches_oracle_and_workspace_entry_with_other_calls_between():
    need_gpu()
    import torch
    import block_sparse_attention_indexer_gb300 as msa
    # 6 sequences x 2 tokens x 4 groups = 48 rows over ~450 teams: every row is cut by team
    # boundaries, so the scratch holds partial states
    w, lens = syn.custom("noalloc", 31, 6, 2, 8, [5000, 129, 20000, 300, 2048, 4096 + 3], shuffled=True)
    dw = device_workload(w, lens)
    cache, table, lens, q, qi = oracle_inputs(w, lens)
    sel_np = OM.select_blocks(OM.block_scores(qi, cache[4], cache[5], table, lens), lens)
    sel = torch.from_numpy(sel_np).cuda()
    ref_o, ref_l = OM.sparse_attention(q, *cache[:4], table, lens, sel_np, w.heads_per_group)
    B, T, H = w.batch, w.q_len, w.num_heads

    out_ws = torch.zeros(B, T, H, 128, dtype=torch.bfloat16, device="cuda")
    lse_ws = torch.zeros(B, T, H, dtype=torch.float32, device="cuda")
    ws = msa.alloc_workspace(msa.MSA_OP_SPARSE_ATTN, dw.cfg, dw.batch)
    msa.msa_sparse_attn_decode(dw.cfg, dw.cache, dw.batch, dw.q, sel, out_ws, lse_ws, ws)
    torch.cuda.synchronize()

    # a differently shaped call (more rows, other selections, 4 heads per group) to run
    # between the two checked calls, so that the array holds its partial states
    w2, lens2 = syn.custom("noalloc_other", 32, 9, 3, 4, [9000, 300, 70000, 129, 4000, 33000, 1000, 640, 20000],
                           shuffled=True)
    dw2 = device_workload(w2, lens2)
    c2, t2, l2, q2, qi2 = oracle_inputs(w2, lens2)
    sel2_np = OM.select_blocks(OM.block_scores(qi2, c2[4], c2[5], t2, l2), l2)
    sel2 = torch.from_numpy(sel2_np).cuda()

    for i in range(2):
        if i == 1:
            o2, lse2 = _noalloc(dw2, sel2)
            ref2_o, ref2_l = OM.sparse_attention(q2, *c2[:4], t2, l2, sel2_np, w2.heads_per_group)
            assert_out_close(o2, ref2_o)
            assert np.allclose(lse2, ref2_l, rtol=1e-4, atol=1e-4)
        o, l = _noalloc(dw, sel)
        assert_out_close(o, ref_o)
        assert np.allclose(l, ref_l, rtol=1e-4, atol=1e-4)
        err = np.abs(o - bf16_to_np(out_ws))
        assert err.max() <= OUT_MAX_ABS and err.mean() <= OUT_MEAN_ABS
        assert np.allclose(l, to_np(lse_ws), rtol=1e-5, atol=1e-5)
        assert msa.msa_noalloc_read_device_error() == 0


@pytest.mark.parametrize("batch,q_len,ctx", [(2048, 31, 160), (1023, 64, 300)],
                         ids=["largest_batch", "chunk64"])
def test_noalloc_at_the_abi_limits(batch, q_len, ctx):
    """The largest batch the ABI accepts (2,048 sequences, batch x q_len <= 65,535) and a
    64-token chunk (the regular entry point goes block-major there; this one stays
    query-major, whose scratch does not grow with the batch): MSA_OK and oracle parity on
    sampled sequences, every token."""
    need_gpu()
    import torch
    w, lens = syn.custom(f"noalloc_{batch}", 33, batch, q_len, 8, [ctx] * batch, shuffled=True)
    dw = device_workload(w, lens)
    sel_np = _selection_all_blocks(lens, q_len)
    o, l = _noalloc(dw, torch.from_numpy(sel_np).cuda())
    seqs = [0, batch // 2, batch - 1]
    cache, table, lens, P = OC.build_cache(w, lens, seqs, threads=16)
    q, _ = OC.encode_queries(w, seqs)
    ref_o, ref_l = OM.sparse_attention(q, *cache[:4], table, lens, sel_np, w.heads_per_group, sequences=seqs)
    assert_out_close(o[seqs], ref_o[seqs])
    assert np.allclose(l[seqs], ref_l[seqs], rtol=1e-4, atol=1e-4)


def test_noalloc_reports_a_bad_page_then_clears():
    need_gpu()
    import torch
    import block_sparse_attention_indexer_gb300 as msa
    w, lens = syn.custom("noalloc_bad", 34, 3, 1, 8, [3000, 5000, 129], shuffled=False)
    dw = device_workload(w, lens)
    sel_np = np.full((3, 1, 4, 16), -1, np.int32)
    for b in range(3):
        r = (int(lens[b]) - 1) // 128
        sel_np[b, 0, :, :min(16, r + 1)] = np.arange(max(0, r - 15), r + 1)[-16:]
    sel = torch.from_numpy(sel_np).cuda()
    table = dw.batch.block_table.clone()
    table[1, int(sel_np[1, 0, 0, 3])] = dw.num_pages + 5      # a selected block points past the pool
    bad = msa.Batch(table, dw.batch.seq_lens, 1)
    out = torch.zeros(3, 1, 32, 128, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros(3, 1, 32, dtype=torch.float32, device="cuda")
    msa.msa_sparse_attn_decode_noalloc(dw.cfg, dw.cache, bad, dw.q, sel, out, lse)
    torch.cuda.synchronize()
    assert msa.msa_noalloc_read_device_error() & msa.MSA_DEVERR_BAD_PAGE
    assert np.isfinite(bf16_to_np(out)).all()
    # a call rejected on the host launches nothing and leaves the word as it was
    with pytest.raises(msa.MsaError, match="INVALID_ARG"):
        msa.msa_sparse_attn_decode_noalloc(dw.cfg, dw.cache, bad, dw.q, sel, None, lse)
    assert msa.msa_noalloc_read_device_error() & msa.MSA_DEVERR_BAD_PAGE
    # the next clean call starts from a zero word and reports nothing
    o, l = _noalloc(dw, sel)
    assert msa.msa_noalloc_read_device_error() == 0
    cache, table_np, lens, q, qi = oracle_inputs(w, lens)
    ref_o, ref_l = OM.sparse_attention(q, *cache[:4], table_np, lens, sel_np, w.heads_per_group)
    assert_out_close(o, ref_o)
