"""Decode context parallelism on one GPU ("vLLM liefert Day-0-Unterstützung für
MiniMax-M3.1-Flash", §NVFP4-Indexer-DCP): S virtual shards, each a range of logical blocks of
every sequence, run msa_dcp_local_candidates; msa_dcp_merge combines their lists.  The exchange
between GPUs is not exercised here (one GPU per box); the two halves are:
  * every shard's block scores are bit-identical to msa_indexer_scores over its range and -inf
    elsewhere;
  * every shard's candidate list is bit-identical to the oracle's dcp_local_candidates run on
    those fp32 scores;
  * the merged selection is bit-identical to msa_select_blocks on the unsharded scores, to the
    oracle's dcp_merge of the same lists, and agrees with the float64 oracle's selection up
    to near ties."""
import numpy as np
import pytest

from gpu_util import OM, device_workload, need_gpu, oracle_inputs, selection_diffs, syn, to_np

pytestmark = pytest.mark.gpu


def _shards(dw, cuts, cfg=None):
    import torch
    import block_sparse_attention_indexer_gb300 as msa
    w = dw.w
    cfg = cfg or dw.cfg
    B, T, MB = w.batch, w.q_len, dw.batch.max_blocks
    ws = msa.alloc_workspace(msa.MSA_OP_INDEXER_SCORES, cfg, dw.batch)
    full = torch.zeros(B, T, 4, MB, dtype=torch.float32, device="cuda")
    msa.msa_indexer_scores(cfg, dw.cache, dw.batch, dw.qi, full, ws)
    sel_full = torch.zeros(B, T, 4, 16, dtype=torch.int32, device="cuda")
    msa.msa_select_blocks(cfg, dw.batch, full, sel_full)
    S = len(cuts) - 1
    part = torch.full((S, B, T, 4, MB), 7.0, dtype=torch.float32, device="cuda")
    cs = torch.zeros(S, B, T, 4, 15, dtype=torch.float32, device="cuda")
    cb = torch.zeros(S, B, T, 4, 15, dtype=torch.int32, device="cuda")
    for i in range(S):
        msa.msa_dcp_local_candidates(cfg, dw.cache, dw.batch, dw.qi, int(cuts[i]), int(cuts[i + 1]), part[i], cs[i],
                                     cb[i], ws)
    sel = torch.full((B, T, 4, 16), 99, dtype=torch.int32, device="cuda")
    msa.msa_dcp_merge(cfg, dw.batch, cs, cb, sel)
    torch.cuda.synchronize()
    assert msa.msa_read_device_error(ws) == 0
    return to_np(full), to_np(sel_full), to_np(part), to_np(cs), to_np(cb), to_np(sel)


def _check(w, dw, cuts):
    full, sel_full, part, cs, cb, sel = _shards(dw, cuts)
    lens, T = dw.lens, w.q_len
    for i in range(len(cuts) - 1):
        lo, hi = int(cuts[i]), int(cuts[i + 1])
        inside = np.zeros(full.shape[-1], bool)
        inside[lo:hi] = True
        assert np.array_equal(part[i][..., inside], full[..., inside]), f"shard {i} scores"
        assert np.isneginf(part[i][..., ~inside]).all(), f"shard {i} outside its range"
    for b in range(w.batch):
        for t in range(T):
            pos = int(lens[b]) - T + t
            for g in range(4):
                lists = []
                for i in range(len(cuts) - 1):
                    want = OM.dcp_local_candidates(full[b, t, g].astype(np.float64), pos, int(cuts[i]), int(cuts[i + 1]))
                    n = len(want)
                    assert list(cb[i, b, t, g, :n]) == [blk for _, blk in want], (i, b, t, g)
                    assert np.array_equal(cs[i, b, t, g, :n].astype(np.float64), np.array([sc for sc, _ in want])), (i, b, t, g)
                    assert (cb[i, b, t, g, n:] == -1).all() and np.isneginf(cs[i, b, t, g, n:]).all()
                    lists.append(want)
                assert np.array_equal(sel[b, t, g], OM.dcp_merge(lists, pos)), (b, t, g)
    assert np.array_equal(sel, sel_full), "merged selection differs from msa_select_blocks"
    return sel


@pytest.mark.parametrize("T,lens,cuts", [
    (1, [5000, 129, 20000, 7, 300, 4096, 70000, 2049], [0, 140, 300, 547]),       # uneven, 3 shards
    (1, [5000, 129, 20000, 7, 300, 4096, 70000, 2049], [0, 547]),                 # one shard = unsharded
    (2, [9000, 3000, 128, 40000, 16 * 128, 16 * 128 + 1], [0, 10, 20, 100, 313]),  # 4 shards, some empty rows
    (1, [131072, 65536], [0, 256, 512, 768, 1024]),                                # 4 equal shards, 128K context
], ids=["s3_uneven", "s1", "s4_t2_edges", "s4_128k"])
def test_dcp_shards_merge_exactly(T, lens, cuts):
    need_gpu()
    w, lens = syn.custom(f"dcp_{len(cuts)}_{T}", 101 + T, len(lens), T, 8, lens, shuffled=True)
    dw = device_workload(w, lens)
    sel = _check(w, dw, cuts)
    # and the float64 oracle's own selection, up to near ties
    cache, table, lens_o, q, qi = oracle_inputs(w, lens)
    ref_s = OM.block_scores(qi, cache[4], cache[5], table, lens_o)
    ref_sel = OM.select_blocks(ref_s, lens_o)
    diff = selection_diffs(sel, ref_sel, ref_s, lens_o, T)
    assert len(diff) <= 2


def test_dcp_shard_order_and_padding_row():
    """Shard lists may arrive in any order; a padding row selects nothing."""
    need_gpu()
    import torch
    import block_sparse_attention_indexer_gb300 as msa
    w, lens = syn.custom("dcp_order", 111, 4, 1, 8, [9000, 0, 20000, 3000], shuffled=True)
    dw = device_workload(w, lens)
    full, sel_full, part, cs, cb, sel = _shards(dw, [0, 50, 90, 157])
    assert np.array_equal(sel, sel_full)
    assert (sel[1] == -1).all()
    sel2 = torch.zeros(4, 1, 4, 16, dtype=torch.int32, device="cuda")
    msa.msa_dcp_merge(dw.cfg, dw.batch, torch.from_numpy(cs[::-1].copy()).cuda(), torch.from_numpy(cb[::-1].copy()).cuda(),
                      sel2)
    torch.cuda.synchronize()
    assert np.array_equal(to_np(sel2), sel)


def test_dcp_host_validation():
    need_gpu()
    import torch
    import block_sparse_attention_indexer_gb300 as msa
    w, lens = syn.custom("dcp_val", 112, 2, 1, 8, [3000, 3000])
    dw = device_workload(w, lens)
    ws = msa.alloc_workspace(msa.MSA_OP_INDEXER_SCORES, dw.cfg, dw.batch)
    sc = torch.zeros(2, 1, 4, dw.batch.max_blocks, dtype=torch.float32, device="cuda")
    cs = torch.zeros(2, 1, 4, 15, dtype=torch.float32, device="cuda")
    cb = torch.zeros(2, 1, 4, 15, dtype=torch.int32, device="cuda")
    with pytest.raises(msa.MsaError, match="INVALID_ARG"):
        msa.msa_dcp_local_candidates(dw.cfg, dw.cache, dw.batch, dw.qi, 5, 5, sc, cs, cb, ws)
    with pytest.raises(msa.MsaError, match="UNSUPPORTED"):     # the recipe's forced blocks only
        msa.msa_dcp_local_candidates(msa.Config(init_blocks=1), dw.cache, dw.batch, dw.qi, 0, 5, sc, cs, cb, ws)
    sel = torch.zeros(2, 1, 4, 16, dtype=torch.int32, device="cuda")
    with pytest.raises(msa.MsaError, match="UNSUPPORTED"):     # at most 8 shards
        msa.msa_dcp_merge(dw.cfg, dw.batch, torch.zeros(9, 2, 1, 4, 15, device="cuda"),
                          torch.zeros(9, 2, 1, 4, 15, dtype=torch.int32, device="cuda"), sel)
