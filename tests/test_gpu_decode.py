"""End-to-end parity of the fused msa_decode entry point with the oracle, on the five
workloads at their full sizes (sampled rows where the oracle would be slow), plus the
device-side error paths.  msa_decode runs with exactly the launch configuration bench.py
times."""
import numpy as np
import pytest

from gpu_util import (OC, OM, assert_out_close, assert_scores_close, bf16_to_np, device_workload, need_gpu,
                      score_bound, selection_diffs, syn, to_np)

pytestmark = pytest.mark.gpu


def _run_decode(dw):
    import torch
    import block_sparse_attention_indexer_gb300 as msa
    w = dw.w
    B, T, H = w.batch, w.q_len, w.num_heads
    out = torch.zeros(B, T, H, 128, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros(B, T, H, dtype=torch.float32, device="cuda")
    sel = torch.zeros(B, T, 4, 16, dtype=torch.int32, device="cuda")
    ws = msa.alloc_workspace(msa.MSA_OP_DECODE, dw.cfg, dw.batch)
    msa.msa_decode(dw.cfg, dw.cache, dw.batch, dw.q, dw.qi, out, lse, sel, ws)
    scores = torch.zeros(B, T, 4, dw.batch.max_blocks, dtype=torch.float32, device="cuda")
    ws2 = msa.alloc_workspace(msa.MSA_OP_INDEXER_SCORES, dw.cfg, dw.batch)
    msa.msa_indexer_scores(dw.cfg, dw.cache, dw.batch, dw.qi, scores, ws2)
    torch.cuda.synchronize()
    assert msa.msa_read_device_error(ws) == 0
    return bf16_to_np(out), to_np(lse), to_np(sel), to_np(scores)


def _check(w, dw, sequences=None, tokens=None):
    """msa_decode's scores, selections, outputs and lse against the oracle on the given
    sequences x tokens (default: all).  The oracle quantises the index keys of those
    sequences and, for the attention, K and V of the blocks its own selection picks."""
    out, lse, sel, scores = _run_decode(dw)
    seqs = list(range(w.batch)) if sequences is None else list(sequences)
    cache, table, lens, P = OC.build_cache(w, dw.lens, seqs, threads=16, index_only=True)
    q, qi = OC.encode_queries(w, seqs)
    toks = list(range(w.q_len)) if tokens is None else list(tokens)
    ref_s = OM.block_scores(qi, cache[4], cache[5], table, lens, tokens=toks, sequences=seqs)
    bound = score_bound(qi, cache[4], cache[5], table, lens, table.shape[1])
    rows = np.zeros(scores.shape[:2], bool)
    for b in seqs:
        rows[b, toks] = True
    assert_scores_close(scores[rows], ref_s[rows], bound[rows])
    ref_sel = np.full(sel.shape, -1, np.int32)
    for b in seqs:
        L = int(lens[b])
        for t in toks:
            for g in range(4):
                ref_sel[b, t, g] = OM.select_row(ref_s[b, t, g], L - w.q_len + t)
    diff = selection_diffs(np.where(rows[:, :, None, None], sel, -1), ref_sel, ref_s, lens, w.q_len)
    OC.add_kv_blocks(cache, w, table, {(b, int(n)) for b in seqs for n in ref_sel[b].ravel() if n >= 0}, threads=16)
    out_ref, lse_ref = OM.sparse_attention(q, *cache[:4], table, lens, ref_sel, w.heads_per_group, tokens=toks,
                                           sequences=seqs)
    mask = rows.copy()
    for (b, t, g) in diff:      # a near-tie selection legitimately changes that row's output
        mask[b, t] = False
    assert len(diff) <= max(2, 0.02 * rows.sum() * 4), f"{len(diff)} near-tie rows"
    err = assert_out_close(out[mask], out_ref[mask])
    assert np.allclose(lse[mask], lse_ref[mask], rtol=1e-4, atol=1e-4)
    return err, len(diff)


def test_tiny_full():
    need_gpu()
    w = syn.WORKLOADS["tiny"]
    _check(w, device_workload(w))


def test_b8_32k_full():
    need_gpu()
    w = syn.WORKLOADS["b8_32k"]
    _check(w, device_workload(w))


def test_ragged64_128k_full():
    """The headline workload, every one of its 64 sequences (4.6 M cached tokens)."""
    need_gpu()
    w = syn.WORKLOADS["ragged64_128k"]
    _check(w, device_workload(w))


def test_spec4_512k_full():
    """Speculative decode, all 4 sequences x 8 query tokens."""
    need_gpu()
    w = syn.WORKLOADS["spec4_512k"]
    _check(w, device_workload(w))


def test_prefill_4k_on_64k_sampled():
    """Chunked prefill on 520 of the 4,096 new tokens: the first and last token of every
    128-token block the chunk covers, plus a seeded sample of the rest."""
    need_gpu()
    w = syn.WORKLOADS["prefill_4k_on_64k"]
    dw = device_workload(w)
    T = w.q_len
    pos0 = int(dw.lens[0]) - T
    edges = {t for t in range(T) if (pos0 + t) % 128 in (0, 127)}
    rng = np.random.default_rng(0)
    rest = [t for t in range(T) if t not in edges]
    toks = sorted(edges | {0, T - 1} | set(int(x) for x in rng.choice(rest, 520 - len(edges | {0, T - 1}),
                                                                        replace=False)))
    assert len(toks) == 520
    _check(w, dw, tokens=toks)


def test_one_million_token_context():
    """A context of 1,048,576 + 77 tokens (8,193 blocks a row) next to a short one: more
    candidates than the selection holds in registers (its shares are re-read from L2) and a
    block-table row longer than it stages for the attention (which then looks the pages up
    itself); every row checked against the oracle."""
    need_gpu()
    w, lens = syn.custom("ctx1m", 161, 2, 1, 8, [1048576 + 77, 20000], shuffled=True)
    dw = device_workload(w, lens)
    _check(w, dw)


def test_deterministic_reruns():
    """Bitwise-identical reruns (a race would show up as nondeterminism)."""
    need_gpu()
    w, lens = syn.custom("det", 11, 6, 2, 8, [5000, 129, 20000, 7, 300, 4096], shuffled=True)
    dw = device_workload(w, lens)
    a = _run_decode(dw)
    b = _run_decode(dw)
    for x, y in zip(a, b):
        assert np.array_equal(x, y, equal_nan=True)


@pytest.mark.parametrize("T", [2, 8, 80], ids=["t2", "t8_speculative", "t80_block_major"])
def test_padding_rows_and_bad_inputs_flag_errors(T):
    """Padding rows, a length below q_len and a bad page: flagged, defined outputs, no fault --
    for two query tokens, for eight (32 query rows: the speculative tcgen05 indexer, whose bad
    page is never copied and whose block scores there are -inf) and for 80 (the tcgen05
    prefill indexer and the block-major plan, which must skip the bad page's entries)."""
    need_gpu()
    import torch
    import block_sparse_attention_indexer_gb300 as msa
    w, lens = syn.custom("bad", 12, 4, T, 8, [3000, 3000, 3000, 3000], shuffled=False)
    dw = device_workload(w, lens)
    B, H = 4, 32
    # sequence 1 is a padding row, sequence 2 is shorter than q_len, sequence 3 has a bad page
    seq = dw.batch.seq_lens.clone()
    seq[1] = 0
    seq[2] = 1
    table = dw.batch.block_table.clone()
    table[3, 5] = dw.num_pages + 10
    batch = msa.Batch(table, seq, T)
    out = torch.full((B, T, H, 128), 3.0, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros(B, T, H, dtype=torch.float32, device="cuda")
    sel = torch.zeros(B, T, 4, 16, dtype=torch.int32, device="cuda")
    ws = msa.alloc_workspace(msa.MSA_OP_DECODE, dw.cfg, batch)
    msa.msa_decode(dw.cfg, dw.cache, batch, dw.q, dw.qi, out, lse, sel, ws)
    torch.cuda.synchronize()
    flags = msa.msa_read_device_error(ws)
    assert flags & msa.MSA_DEVERR_BAD_SEQLEN and flags & msa.MSA_DEVERR_BAD_PAGE
    o, l, s = bf16_to_np(out), to_np(lse), to_np(sel)
    for b in (1, 2):
        assert (o[b] == 0).all() and np.isneginf(l[b]).all() and (s[b] == -1).all()
    assert np.isfinite(o[0]).all() and np.isfinite(o[3]).all()
    msa.msa_clear_device_error(ws)
    assert msa.msa_read_device_error(ws) == 0


def test_host_validation_rejects_before_launch():
    need_gpu()
    import torch
    import block_sparse_attention_indexer_gb300 as msa
    w, lens = syn.custom("val", 13, 2, 1, 8, [1000, 2000])
    dw = device_workload(w, lens)
    out = torch.zeros(2, 1, 32, 128, dtype=torch.bfloat16, device="cuda")
    small = torch.zeros(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(msa.MsaError, match="WORKSPACE"):
        msa.msa_decode(dw.cfg, dw.cache, dw.batch, dw.q, dw.qi, out, None, None, small)
    bad_cfg = msa.Config(heads_per_group=8, top_k=17)
    ws = msa.alloc_workspace(msa.MSA_OP_DECODE, dw.cfg, dw.batch)
    with pytest.raises(msa.MsaError, match="UNSUPPORTED"):
        msa.msa_decode(bad_cfg, dw.cache, dw.batch, dw.q, dw.qi, out, None, None, ws)
    # a query pointer that is not 16-byte aligned is rejected on the host
    buf = torch.zeros(dw.q.numel() + 16, dtype=torch.uint8, device="cuda")
    q_mis = buf[1:1 + dw.q.numel()].view(dw.q.shape)
    with pytest.raises(msa.MsaError, match="INVALID_ARG"):
        msa.msa_decode(dw.cfg, dw.cache, dw.batch, q_mis, dw.qi, out, None, None, ws)


def test_inputs_written_by_the_kernel_just_before_are_seen():
    """On the decode step the selection reads seq_lens and the block table before its wait on
    the indexer (the step's inputs were written before its first kernel, which waits for the
    writer).  Inputs written by kernels queued on the same stream right before msa_decode,
    with no synchronisation, must give bit-for-bit the result of the same inputs written
    beforehand; the old inputs give a different one."""
    need_gpu()
    import torch
    import block_sparse_attention_indexer_gb300 as msa
    lens = [20000, 9000, 3000, 129, 40000, 5000, 16 * 128 + 5, 700]
    w, lens = syn.custom("inputs_early", 131, len(lens), 1, 8, lens, shuffled=True)
    dw = device_workload(w, lens)
    B, T, H = w.batch, w.q_len, w.num_heads
    old_table, old_lens = dw.batch.block_table.clone(), dw.batch.seq_lens.clone()
    # new inputs: sequence b takes sequence b - 1's length and pages
    new_table, new_lens = torch.roll(old_table, 1, 0).contiguous(), torch.roll(old_lens, 1, 0).contiguous()

    def decode(batch):
        out = torch.zeros(B, T, H, 128, dtype=torch.bfloat16, device="cuda")
        lse = torch.zeros(B, T, H, dtype=torch.float32, device="cuda")
        sel = torch.full((B, T, 4, 16), 7, dtype=torch.int32, device="cuda")
        ws = msa.alloc_workspace(msa.MSA_OP_DECODE, dw.cfg, batch)
        torch.cuda.synchronize()
        return out, lse, sel, ws

    # reference: the new inputs in place before the call
    ref_b = msa.Batch(new_table.clone(), new_lens.clone(), 1)
    o_ref, l_ref, s_ref, ws = decode(ref_b)
    msa.msa_decode(dw.cfg, dw.cache, ref_b, dw.q, dw.qi, o_ref, l_ref, s_ref, ws)
    torch.cuda.synchronize()
    assert msa.msa_read_device_error(ws) == 0
    # the same call with the old inputs
    old_b = msa.Batch(old_table.clone(), old_lens.clone(), 1)
    o_old, l_old, s_old, ws_old = decode(old_b)
    msa.msa_decode(dw.cfg, dw.cache, old_b, dw.q, dw.qi, o_old, l_old, s_old, ws_old)
    torch.cuda.synchronize()
    assert not torch.equal(s_old, s_ref)
    # the buffers hold the old inputs; elementwise kernels write the new ones on the stream,
    # and msa_decode follows them with no synchronisation in between
    for _ in range(3):
        t_b = msa.Batch(old_table.clone(), old_lens.clone(), 1)
        o, l, s, ws_t = decode(t_b)
        torch.add(new_table, 0, out=t_b.block_table)
        torch.add(new_lens, 0, out=t_b.seq_lens)
        msa.msa_decode(dw.cfg, dw.cache, t_b, dw.q, dw.qi, o, l, s, ws_t)
        torch.cuda.synchronize()
        assert msa.msa_read_device_error(ws_t) == 0
        assert torch.equal(s, s_ref)
        assert torch.equal(o, o_ref) and torch.equal(l, l_ref)


@pytest.mark.parametrize("T,lens", [
    (1, [20000, 9000, 3000, 129, 40000, 5000, 16 * 128 + 5, 700]),   # streaming indexer, team attention
    (8, [30000, 70000, 2100]),                                       # tcgen05 speculative indexer
    (96, [8000, 3000]),                                              # prefill indexer, block-major attention
], ids=["decode", "spec", "prefill"])
def test_page_relabelling_leaves_every_output_bitwise_unchanged(T, lens):
    """The pages are reached only through the block table: moving every page of the six pools
    to a new id (a seeded permutation) and rewriting the table to match leaves the block
    scores, selections, outputs and lse bit-for-bit unchanged, on each indexer and attention
    form."""
    need_gpu()
    import torch
    import block_sparse_attention_indexer_gb300 as msa
    w, lens = syn.custom(f"relabel_{T}", 141 + T, len(lens), T, 8, lens, shuffled=True)
    dw = device_workload(w, lens)
    B, H = w.batch, w.num_heads

    def run(cache, batch):
        out = torch.zeros(B, T, H, 128, dtype=torch.bfloat16, device="cuda")
        lse = torch.zeros(B, T, H, dtype=torch.float32, device="cuda")
        sel = torch.zeros(B, T, 4, 16, dtype=torch.int32, device="cuda")
        scores = torch.zeros(B, T, 4, batch.max_blocks, dtype=torch.float32, device="cuda")
        ws = msa.alloc_workspace(msa.MSA_OP_DECODE, dw.cfg, batch)
        ws_i = msa.alloc_workspace(msa.MSA_OP_INDEXER_SCORES, dw.cfg, batch)
        msa.msa_decode(dw.cfg, cache, batch, dw.q, dw.qi, out, lse, sel, ws)
        msa.msa_indexer_scores(dw.cfg, cache, batch, dw.qi, scores, ws_i)
        torch.cuda.synchronize()
        assert msa.msa_read_device_error(ws) == 0 and msa.msa_read_device_error(ws_i) == 0
        return out, lse, sel, scores

    base = run(dw.cache, dw.batch)
    P = dw.cache.num_pages
    perm = torch.randperm(P, generator=torch.Generator().manual_seed(5)).to("cuda")  # page p -> perm[p]
    moved = msa.PagedCache(P, 4, 128, 128, 128)
    for old, new in zip(dw.cache.tensors(), moved.tensors()):
        new[perm] = old
    tab = dw.batch.block_table
    new_tab = torch.where(tab >= 0, perm[tab.clamp(min=0).long()].to(torch.int32), tab).contiguous()
    assert not torch.equal(new_tab, tab)
    relabelled = run(moved, msa.Batch(new_tab, dw.batch.seq_lens.clone(), T))
    for name, a, b in zip(("out", "lse", "selection", "scores"), base, relabelled):
        assert torch.equal(a, b), name


@pytest.mark.parametrize("T,lens", [(1, [9000, 300, 40000, 2200]), (8, [30000, 5000]), (80, [6000])],
                         ids=["decode", "spec", "prefill"])
def test_optional_outputs_change_nothing(T, lens):
    """selection_out and lse are optional: with or without them msa_decode gives the same
    output bit for bit (without selection_out the selection stays in the workspace), and the
    selection it hands out is the one msa_select_blocks makes from the same scores."""
    need_gpu()
    import torch
    import block_sparse_attention_indexer_gb300 as msa
    w, lens = syn.custom(f"optional_{T}", 151 + T, len(lens), T, 8, lens, shuffled=True)
    dw = device_workload(w, lens)
    B, H = w.batch, w.num_heads
    results = []
    for with_sel, with_lse in ((True, True), (False, True), (True, False), (False, False)):
        out = torch.zeros(B, T, H, 128, dtype=torch.bfloat16, device="cuda")
        lse = torch.zeros(B, T, H, dtype=torch.float32, device="cuda") if with_lse else None
        sel = torch.full((B, T, 4, 16), 9, dtype=torch.int32, device="cuda") if with_sel else None
        ws = msa.alloc_workspace(msa.MSA_OP_DECODE, dw.cfg, dw.batch)
        msa.msa_decode(dw.cfg, dw.cache, dw.batch, dw.q, dw.qi, out, lse, sel, ws)
        torch.cuda.synchronize()
        assert msa.msa_read_device_error(ws) == 0
        results.append((out, lse, sel))
    for out, lse, sel in results[1:]:
        assert torch.equal(out, results[0][0])
        if lse is not None:
            assert torch.equal(lse, results[0][1])
    assert torch.equal(results[0][2], results[2][2])
    scores = torch.zeros(B, T, 4, dw.batch.max_blocks, dtype=torch.float32, device="cuda")
    msa.msa_indexer_scores(dw.cfg, dw.cache, dw.batch, dw.qi, scores,
                           msa.alloc_workspace(msa.MSA_OP_INDEXER_SCORES, dw.cfg, dw.batch))
    sel2 = torch.zeros(B, T, 4, 16, dtype=torch.int32, device="cuda")
    msa.msa_select_blocks(dw.cfg, dw.batch, scores, sel2)
    torch.cuda.synchronize()
    assert torch.equal(sel2, results[0][2])
