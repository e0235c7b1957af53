"""The query-major sparse attention (msa_sparse_attn_decode below 64 query tokens per
sequence) on the edges of its work split, against the float64 oracle.

The (row, selection entry) pairs of all rows are cut into equal ranges, one per team of four
warps, and rows cut by ranges are merged from partial states by a second kernel.  Covered
here: a single row, few rows, ragged contexts, speculative tokens sharing pages, rows with
empty entries (top_k < 16, short contexts, padding rows, a bad page), 16,384 rows, and
bitwise repeatability; the no-allocation entry point (the same kernel on its fixed scratch)
gives bit-identical results."""
import numpy as np
import pytest

from gpu_util import OC, OM, assert_out_close, bf16_to_np, device_workload, need_gpu, oracle_inputs, syn, to_np

pytestmark = pytest.mark.gpu


def _both(dw, sel_np, cfg=None, batch=None):
    import torch
    import block_sparse_attention_indexer_gb300 as msa
    w = dw.w
    cfg = cfg or dw.cfg
    batch = batch or dw.batch
    B, T, H = w.batch, w.q_len, w.num_heads
    sel = torch.from_numpy(sel_np).cuda()
    out_s = torch.full((B, T, H, 128), 7.0, dtype=torch.bfloat16, device="cuda")
    lse_s = torch.zeros(B, T, H, dtype=torch.float32, device="cuda")
    ws = msa.alloc_workspace(msa.MSA_OP_SPARSE_ATTN, cfg, batch)
    msa.msa_sparse_attn_decode(cfg, dw.cache, batch, dw.q, sel, out_s, lse_s, ws)
    out_t = torch.full((B, T, H, 128), 7.0, dtype=torch.bfloat16, device="cuda")
    lse_t = torch.zeros(B, T, H, dtype=torch.float32, device="cuda")
    msa.msa_sparse_attn_decode_noalloc(cfg, dw.cache, batch, dw.q, sel, out_t, lse_t)
    torch.cuda.synchronize()
    flags = msa.msa_read_device_error(ws)
    return (bf16_to_np(out_s), to_np(lse_s)), (bf16_to_np(out_t), to_np(lse_t)), flags


def _agree(a, b):
    """The workspace entry point and the no-allocation one run the same kernel on the same
    split: bit-identical outputs and lse."""
    (oa, la), (ob, lb) = a, b
    assert np.array_equal(oa, ob)
    assert np.array_equal(la, lb, equal_nan=True)


def _oracle(w, lens, sel_np, out, lse, sequences=None):
    seqs = list(range(w.batch)) if sequences is None else list(sequences)
    cache, table, lens, _ = OC.build_cache(w, lens, seqs, threads=16)
    q, _ = OC.encode_queries(w, seqs)
    ref_o, ref_l = OM.sparse_attention(q, *cache[:4], table, lens, sel_np, w.heads_per_group, sequences=seqs)
    assert_out_close(out[seqs], ref_o[seqs])
    assert np.allclose(lse[seqs], ref_l[seqs], rtol=1e-4, atol=1e-4)


def _oracle_selection(w, lens, top_k=16, init=0, local=1):
    """The oracle's selection, padded with -1 to the ABI's 16 entries per row."""
    cache, table, lens, q, qi = oracle_inputs(w, lens)
    s = OM.block_scores(qi, cache[4], cache[5], table, lens)
    sel = OM.select_blocks(s, lens, top_k, init, local)
    out = np.full(sel.shape[:3] + (16,), -1, np.int32)
    out[..., :top_k] = sel
    return out


@pytest.mark.parametrize("name,B,T,hg,lens", [
    ("one_row", 1, 1, 1, [700]),                                  # one row cut across many teams
    ("few_rows", 2, 1, 8, [20000, 129]),
    ("ragged", 9, 1, 8, [5000, 129, 20000, 7, 300, 4096, 130000, 2049, 16 * 128 + 1]),
    ("spec_t8", 2, 8, 8, [40000, 3000]),                           # tokens share pages (L2 policy)
    ("t3_hg4", 5, 3, 4, [9000, 40000, 3000, 129, 20000]),
])
def test_attention_edges_vs_oracle(name, B, T, hg, lens):
    need_gpu()
    w, lens = syn.custom(f"attn_{name}", 81 + B + T, B, T, hg, lens, shuffled=True)
    dw = device_workload(w, lens)
    sel = _oracle_selection(w, lens)
    ws_res, noalloc_res, flags = _both(dw, sel)
    assert flags == 0
    _agree(ws_res, noalloc_res)
    _oracle(w, lens, sel, *ws_res)


def test_attention_empty_entries_padding_and_bad_page():
    """top_k 5 with init 1 / local 1 (most entries empty), a padding row, a row shorter than
    q_len, and a bad block-table entry: flagged, defined outputs, oracle parity elsewhere."""
    need_gpu()
    import block_sparse_attention_indexer_gb300 as msa
    w, lens = syn.custom("attn_edges", 91, 5, 2, 8, [9000, 3000, 20000, 5000, 2000], shuffled=True)
    dw = device_workload(w, lens)
    sel = _oracle_selection(w, lens, top_k=5, init=1, local=1)
    cfg = msa.Config(top_k=5, init_blocks=1, local_blocks=1)
    seq = dw.batch.seq_lens.clone()
    seq[1] = 0                         # padding row
    seq[3] = 1                         # shorter than q_len
    table = dw.batch.block_table.clone()
    table[4, int(sel[4, 0, 2, 1])] = dw.num_pages + 3
    bad = msa.Batch(table, seq, 2)
    ws_res, noalloc_res, flags = _both(dw, sel, cfg, bad)
    assert flags & msa.MSA_DEVERR_BAD_PAGE
    _agree(ws_res, noalloc_res)
    o, l = ws_res
    for b in (1, 3):
        assert (o[b] == 0).all() and np.isneginf(l[b]).all()
    _oracle(w, lens, sel, o, l, sequences=[0, 2])


def test_attention_many_rows_and_repeatability():
    """2,048 sequences x 2 tokens x 4 groups (16,384 rows, short contexts): sampled oracle rows,
    and five calls bit-identical."""
    need_gpu()
    import torch
    import block_sparse_attention_indexer_gb300 as msa
    rng = np.random.default_rng(9)
    lens = (rng.integers(2, 24, size=2048) * 128 + rng.integers(0, 128, size=2048)).astype(np.int32)
    w, lens = syn.custom("attn_many", 93, 2048, 2, 8, lens, shuffled=True)
    dw = device_workload(w, lens)
    sel = np.full((2048, 2, 4, 16), -1, np.int32)
    for b in range(2048):                      # the recent block and up to 15 others, ascending
        for t in range(2):
            r = (int(lens[b]) - 2 + t) // 128
            for g in range(4):
                others = rng.choice(r, size=min(15, r), replace=False) if r > 0 else np.zeros(0, int)
                ids = np.sort(np.append(others, r))
                sel[b, t, g, :len(ids)] = ids
    ws_res, noalloc_res, flags = _both(dw, sel)
    assert flags == 0
    _agree(ws_res, noalloc_res)
    _oracle(w, lens, sel, *ws_res, sequences=[0, 1, 777, 2047])
    B, T, H = 2048, 2, 32
    ws = msa.alloc_workspace(msa.MSA_OP_SPARSE_ATTN, dw.cfg, dw.batch)
    sel_d = torch.from_numpy(sel).cuda()
    outs = []
    for _ in range(5):
        out = torch.zeros(B, T, H, 128, dtype=torch.bfloat16, device="cuda")
        lse = torch.zeros(B, T, H, dtype=torch.float32, device="cuda")
        msa.msa_sparse_attn_decode(dw.cfg, dw.cache, dw.batch, dw.q, sel_d, out, lse, ws)
        torch.cuda.synchronize()
        outs.append((bf16_to_np(out), to_np(lse)))
    for o, l in outs[1:]:
        assert np.array_equal(o, outs[0][0]) and np.array_equal(l, outs[0][1])
