"""Parity of the configuration variants the pages name with the oracle, through the C ABI:
the block-score reduction (max or log-sum-exp) and the forced blocks of the selection
(init_blocks leading, local_blocks trailing) with top_k below 16 ("MiniMax M3 x vLLM：百万
token 多模态推理的 Day-0 部署", §Prefill 执行 step 2 and §MSA 机制细节)."""
import dataclasses

import numpy as np
import pytest

from gpu_util import (OM, NEAR_TIE_REL, assert_out_close, bf16_to_np, device_workload, need_gpu, oracle_inputs,
                      score_bound, syn, to_np)

pytestmark = pytest.mark.gpu

CASES = [
    # name, lens, q_len, heads_per_group, shuffled  (q_len x 4 groups picks the indexer kernel)
    ("v_ragged_t1", [1, 127, 129, 1000, 4096 + 5, 16 * 128 + 1], 1, 8, True),   # half-page kernel
    ("v_spec_t3", [300, 5000, 3 * 128], 3, 4, True),                           # speculative tcgen05 kernel
    ("v_chunked_t20", [640, 3000], 20, 8, True),                               # tcgen05 GEMM kernel
]
VARIANTS = [  # top_k, init_blocks, local_blocks
    (16, 0, 1), (8, 2, 2), (4, 0, 0), (12, 3, 1), (16, 1, 3), (1, 0, 1), (5, 5, 0),
]


def _lse_tol(bound, ref):
    # float32 accumulation of each key score, then a float32 sum of up to 128 exponentials
    # and one log: the scores' bound plus a few float32 ulps of the result
    return bound * 2.0 ** -16 + 1e-5 + 1e-6 * np.abs(ref)


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_indexer_log_sum_exp(case):
    need_gpu()
    import torch
    import block_sparse_attention_indexer_gb300 as msa
    name, lens, q_len, hg, shuffled = case
    w, lens = syn.custom(name, 91 + len(name), len(lens), q_len, hg, lens, shuffled=shuffled)
    dw = device_workload(w, lens)
    cache, table, lens, q, qi = oracle_inputs(w, lens)
    cfg = dataclasses.replace(dw.cfg, score_type=msa.MSA_SCORE_LSE)
    B, T, MB = w.batch, w.q_len, table.shape[1]
    scores = torch.full((B, T, 4, MB), 7.0, dtype=torch.float32, device="cuda")
    ws = msa.alloc_workspace(msa.MSA_OP_INDEXER_SCORES, cfg, dw.batch)
    msa.msa_indexer_scores(cfg, dw.cache, dw.batch, dw.qi, scores, ws)
    torch.cuda.synchronize()
    assert msa.msa_read_device_error(ws) == 0
    got = to_np(scores).astype(np.float64)
    ref = OM.block_scores(qi, cache[4], cache[5], table, lens, pooling="lse")
    assert np.array_equal(np.isneginf(got), np.isneginf(ref))
    fin = np.isfinite(ref)
    bound = score_bound(qi, cache[4], cache[5], table, lens, MB)
    err = np.abs(got[fin] - ref[fin])
    assert (err <= _lse_tol(bound[fin], ref[fin])).all(), float(err.max())


def _pad16(sel):
    out = np.full(sel.shape[:-1] + (16,), -1, np.int32)
    out[..., : sel.shape[-1]] = sel
    return out


@pytest.mark.parametrize("variant", VARIANTS, ids=[f"k{v[0]}_i{v[1]}_l{v[2]}" for v in VARIANTS])
@pytest.mark.parametrize("case", CASES[:2], ids=[c[0] for c in CASES[:2]])
def test_select_variants_bit_exact_on_oracle_scores(case, variant):
    need_gpu()
    import torch
    import block_sparse_attention_indexer_gb300 as msa
    name, lens, q_len, hg, shuffled = case
    k, init, local = variant
    w, lens = syn.custom(name, 5, len(lens), q_len, hg, lens, shuffled=shuffled)
    cache, table, lens, q, qi = oracle_inputs(w, lens)
    ref_scores = OM.block_scores(qi, cache[4], cache[5], table, lens).astype(np.float32)
    want = _pad16(OM.select_blocks(ref_scores.astype(np.float64), lens, k, init, local))
    batch = msa.Batch(torch.from_numpy(table).cuda(), torch.from_numpy(lens).cuda(), w.q_len)
    cfg = msa.Config(heads_per_group=hg, top_k=k, init_blocks=init, local_blocks=local)
    sel = torch.full(want.shape, 99, dtype=torch.int32, device="cuda")
    msa.msa_select_blocks(cfg, batch, torch.from_numpy(ref_scores).cuda(), sel)
    torch.cuda.synchronize()
    assert np.array_equal(to_np(sel), want)


def test_select_variants_on_long_rows_and_ties():
    """4,096-candidate rows (the staged path) and rows made of exact ties."""
    need_gpu()
    import torch
    import block_sparse_attention_indexer_gb300 as msa
    rng = np.random.default_rng(44)
    R, MB = 24, 4200
    scores = rng.standard_normal((R, 1, 1, MB)).astype(np.float32)
    scores[8:16] = np.round(scores[8:16])                       # many exact ties
    scores[16:, 0, 0, ::3] = np.float32(np.nan)
    lens = np.array([int(rng.integers(1, MB * 128)) for _ in range(R)], np.int32)
    for k, init, local in [(16, 0, 1), (9, 2, 3), (16, 4, 0)]:
        want = np.stack([_pad16(OM.select_row(scores[i, 0, 0].astype(np.float64), int(lens[i]) - 1, k, init, local))
                         for i in range(R)])
        sc4 = np.repeat(scores, 4, axis=2)                        # 4 groups, identical rows
        table = np.zeros((R, MB), np.int32)
        batch = msa.Batch(torch.from_numpy(table).cuda(), torch.from_numpy(lens).cuda(), 1)
        cfg = msa.Config(top_k=k, init_blocks=init, local_blocks=local)
        sel = torch.full((R, 1, 4, 16), 99, dtype=torch.int32, device="cuda")
        msa.msa_select_blocks(cfg, batch, torch.from_numpy(np.ascontiguousarray(sc4)).cuda(), sel)
        torch.cuda.synchronize()
        got = to_np(sel)
        for g in range(4):
            assert np.array_equal(got[:, 0, g], want), (k, init, local)


@pytest.mark.parametrize("case", [("v_e2e", 2, [3000, 9000, 700]), ("v_e2e_chunk", 80, [2000, 9000])],
                         ids=["decode_t2", "chunk_t80"])
def test_decode_variant_end_to_end(case):
    """msa_decode with top_k 8, init_blocks 2, local_blocks 2 and log-sum-exp pooling: two
    query tokens (streaming indexer, team attention), and 80 (the tcgen05 prefill indexer and
    the block-major attention, half of whose selection slots are then empty)."""
    need_gpu()
    import torch
    import block_sparse_attention_indexer_gb300 as msa
    k, init, local = 8, 2, 2
    name, q_len, ctx = case
    w, lens = syn.custom(name, 303, len(ctx), q_len, 4, ctx, shuffled=True)
    dw = device_workload(w, lens)
    cfg = dataclasses.replace(dw.cfg, top_k=k, init_blocks=init, local_blocks=local, score_type=msa.MSA_SCORE_LSE)
    B, T, H = w.batch, w.q_len, w.num_heads
    out = torch.zeros(B, T, H, 128, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros(B, T, H, dtype=torch.float32, device="cuda")
    sel = torch.zeros(B, T, 4, 16, dtype=torch.int32, device="cuda")
    ws = msa.alloc_workspace(msa.MSA_OP_DECODE, cfg, dw.batch)
    msa.msa_decode(cfg, dw.cache, dw.batch, dw.q, dw.qi, out, lse, sel, ws)
    torch.cuda.synchronize()
    assert msa.msa_read_device_error(ws) == 0
    out, lse, sel = bf16_to_np(out), to_np(lse), to_np(sel)
    cache, table, lens, q, qi = oracle_inputs(w, lens)
    ref_s = OM.block_scores(qi, cache[4], cache[5], table, lens, pooling="lse")
    ref_sel = _pad16(OM.select_blocks(ref_s, lens, k, init, local))
    same = np.ones((B, T), bool)
    for b in range(B):
        for t in range(T):
            r = (int(lens[b]) - T + t) // 128
            for g in range(4):
                a, e = set(int(x) for x in sel[b, t, g] if x >= 0), set(int(x) for x in ref_sel[b, t, g] if x >= 0)
                assert len(a) == len(e) == min(k, r + 1)
                forced = set(range(min(init, r + 1))) | set(range(max(0, r - local + 1), r + 1))
                assert forced <= a
                if a != e:     # only near ties among the ranked blocks may differ
                    same[b, t] = False
                    thr = min(ref_s[b, t, g, n] for n in e - forced)
                    for n in a ^ e:
                        assert abs(ref_s[b, t, g, n] - thr) <= NEAR_TIE_REL * abs(thr), (b, t, g, n)
    assert same.sum() >= same.size - max(1, same.size // 50)
    out_ref, lse_ref = OM.sparse_attention(q, *cache[:4], table, lens, ref_sel[..., :k], w.heads_per_group)
    assert_out_close(out[same], out_ref[same])
    assert np.allclose(lse[same], lse_ref[same], rtol=1e-4, atol=1e-4)
