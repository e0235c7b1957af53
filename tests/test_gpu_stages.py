"""Stage-by-stage parity of the CUDA path with the oracle, through the C ABI.

Each stage is fed inputs the oracle computed itself (never outputs of another CUDA
stage): the indexer gets the seeded workload, the selection gets the oracle's scores
rounded to float32, the attention gets the oracle's selection."""
import numpy as np
import pytest

from gpu_util import (OF, OM, assert_out_close, assert_scores_close, bf16_to_np, device_workload, need_gpu,
                      oracle_inputs, score_bound, syn, to_np)

pytestmark = pytest.mark.gpu

CASES = [
    # name, lens, q_len, heads_per_group, shuffled
    ("ragged_t1", [1, 127, 128, 129, 1000, 4096 + 5, 2048, 16 * 128 + 1], 1, 8, True),
    ("spec_t3", [300, 5000, 3 * 128], 3, 4, True),           # 12 rows: speculative tcgen05 indexer, N 16
    ("spec_t8", [8, 2100, 7777], 8, 8, False),               # 32 rows: N 32
    ("spec_t15", [15, 1111, 6000 + 3], 15, 4, True),         # 60 rows: N 64, the widest speculative case
    ("chunked_t20", [640, 3000], 20, 8, True),               # 80 rows: tcgen05 GEMM indexer
    ("chunked_t12", [1500, 999, 260], 12, 4, True),          # 48 rows: speculative indexer, N 48
    ("prefill_t300", [300, 5000 + 77, 40000], 300, 8, True),  # 1,200 rows: several GEMM row tiles
    ("prefill_t96", [96, 3000 + 5], 96, 8, True),            # 384 rows: the last CTA has one full tile
    ("hg4_t1", [4096] * 3, 1, 4, False),
    ("many_rows_t4", [300 + 37 * i for i in range(64)], 4, 8, True),     # 1024 rows: no split
    ("rows256_t2", [2500 + 101 * i for i in range(32)], 2, 8, True),      # 256 rows: 4 splits
    # the dispatch edges: 64 rows (the GEMM indexer's first shape), 63 query tokens (the team
    # attention's last), 64 query tokens (the block-major attention's first), each with a
    # sequence exactly as long as its new tokens
    ("edge_t16", [16, 700, 4000 + 9], 16, 8, True),
    ("edge_t63", [63, 3000], 63, 8, True),
    ("edge_t64", [64, 2000 + 3], 64, 8, True),
    ("prefill_hg4_t80", [80, 3000 + 1], 80, 4, True),       # block-major with 4 heads per group: 32 tokens a tile
]


def _setup(name, lens, q_len, hg, shuffled):
    w, lens = syn.custom(name, 77 + len(name), len(lens), q_len, hg, lens, shuffled=shuffled)
    dw = device_workload(w, lens)
    cache, table, lens, q, qi = oracle_inputs(w, lens)
    return w, dw, cache, table, lens, q, qi


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_indexer_scores(case):
    need_gpu()
    import torch
    import block_sparse_attention_indexer_gb300 as msa
    w, dw, cache, table, lens, q, qi = _setup(*case)
    # both sides quantised the same fp32 values: identical bytes
    assert np.array_equal(to_np(dw.cache.idx_data), cache[4]) and np.array_equal(to_np(dw.cache.idx_scale), cache[5])
    assert np.array_equal(to_np(dw.qi), qi)
    B, T, MB = w.batch, w.q_len, table.shape[1]
    scores = torch.full((B, T, 4, MB), 7.0, dtype=torch.float32, device="cuda")
    ws = msa.alloc_workspace(msa.MSA_OP_INDEXER_SCORES, dw.cfg, dw.batch)
    msa.msa_indexer_scores(dw.cfg, dw.cache, dw.batch, dw.qi, scores, ws)
    torch.cuda.synchronize()
    assert msa.msa_read_device_error(ws) == 0
    ref = OM.block_scores(qi, cache[4], cache[5], table, lens)
    bound = score_bound(qi, cache[4], cache[5], table, lens, MB)
    assert_scores_close(to_np(scores), ref, bound)


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_select_bit_exact_on_oracle_scores(case):
    need_gpu()
    import torch
    import block_sparse_attention_indexer_gb300 as msa
    w, lens = syn.custom(case[0], 5, len(case[1]), case[2], case[3], case[1], shuffled=case[4])
    cache, table, lens, q, qi = oracle_inputs(w, lens)
    ref_scores = OM.block_scores(qi, cache[4], cache[5], table, lens).astype(np.float32)
    want = OM.select_blocks(ref_scores.astype(np.float64), lens)
    batch = msa.Batch(torch.from_numpy(table).cuda(), torch.from_numpy(lens).cuda(), w.q_len)
    cfg = msa.Config(heads_per_group=w.heads_per_group)
    sel = torch.full(want.shape, 99, dtype=torch.int32, device="cuda")
    msa.msa_select_blocks(cfg, batch, torch.from_numpy(ref_scores).cuda(), sel)
    torch.cuda.synchronize()
    assert np.array_equal(to_np(sel), want)


def _select_synthetic(rows_scores, pos_per_row, max_blocks):
    """Runs the GPU select on hand-made score rows (one sequence per row, q_len 1)."""
    import torch
    import block_sparse_attention_indexer_gb300 as msa
    R = len(rows_scores)
    scores = np.full((R, 1, 1, max_blocks), -np.inf, dtype=np.float32)
    for i, s in enumerate(rows_scores):
        scores[i, 0, 0, :len(s)] = s
    lens = np.asarray(pos_per_row, dtype=np.int32) + 1
    table = np.zeros((R, max_blocks), dtype=np.int32)
    batch = msa.Batch(torch.from_numpy(table).cuda(), torch.from_numpy(lens).cuda(), 1)
    cfg = msa.Config(num_kv_groups=1, heads_per_group=1)
    sel = torch.full((R, 1, 1, 16), 99, dtype=torch.int32, device="cuda")
    msa.msa_select_blocks(cfg, batch, torch.from_numpy(scores).cuda(), sel)
    torch.cuda.synchronize()
    got = to_np(sel)[:, 0, 0]
    want = np.stack([OM.select_row(scores[i, 0, 0].astype(np.float64), int(pos_per_row[i])) for i in range(R)])
    return got, want


def test_select_ties_nan_inf_and_edges():
    need_gpu()
    rng = np.random.default_rng(1)
    rows, poss = [], []
    MB = 4096
    for r in [0, 1, 5, 15, 16, 17, 31, 32, 33, 100, 1000, 4095]:
        s = rng.integers(-3, 4, size=MB).astype(np.float32)      # heavy ties
        rows.append(s)
        poss.append(r * 128 + int(rng.integers(0, 128)))
    s = rng.standard_normal(MB).astype(np.float32)
    s[rng.random(MB) < 0.3] = np.nan
    s[rng.random(MB) < 0.3] = -np.inf
    rows.append(s)
    poss.append(3000 * 128)
    s = np.full(MB, np.nan, dtype=np.float32)
    s[::97] = -np.inf
    rows.append(s)
    poss.append(2000 * 128 + 5)
    s = rng.standard_normal(MB).astype(np.float32)
    s[5] = -0.0
    s[6] = 0.0
    s[7] = 0.0
    rows.append(s)
    poss.append(40 * 128)
    got, want = _select_synthetic(rows, poss, MB)
    assert np.array_equal(got, want)


def test_select_overflow_fallback():
    need_gpu()
    # lanes 0..14 of the warp hold all the large scores, lane l's values all above lane
    # l+1's, so thousands of keys pass the first filter and the full-row path runs
    MB = 4096
    s = np.zeros(MB, dtype=np.float32)
    for n in range(MB):
        lane = n % 32
        s[n] = (1000.0 - 10 * lane + n / 8192.0) if lane < 15 else -float(n)
    got, want = _select_synthetic([s], [MB * 128 - 1], MB)
    assert np.array_equal(got, want)


@pytest.mark.parametrize("MB", [576, 768, 1024])
def test_select_warp_per_row_edges(MB):
    """More than 2,048 rows of at most 1,024 candidates take the warp-per-row kernel, whose
    instance holds 18, 24 or 32 candidates per lane by the row length: heavy ties, NaN and
    -inf, signed zeros, rows whose survivors of the first filter exceed 32 (the arg-max
    rounds) or the buffer (all scores equal: the full-row rounds), and every recent-block
    position class; 1,050 sequences x 2 KV groups, each row compared with the oracle's."""
    need_gpu()
    import torch
    import block_sparse_attention_indexer_gb300 as msa
    rng = np.random.default_rng(MB)
    B, G = 1050, 2
    scores = np.zeros((B, 1, G, MB), dtype=np.float32)
    for i in range(B * G):
        kind = i % 6
        if kind == 0:
            s = rng.integers(-3, 4, size=MB).astype(np.float32)
        elif kind == 1:
            s = rng.standard_normal(MB).astype(np.float32)
            s[rng.random(MB) < 0.3] = np.nan
            s[rng.random(MB) < 0.3] = -np.inf
        elif kind == 2:
            lane = np.arange(MB) % 32
            s = np.where(lane < 15, 1000.0 - 10 * lane + np.arange(MB) / 8192.0, -np.arange(MB, dtype=np.float64))
            s = s.astype(np.float32)
        elif kind == 3:
            s = np.zeros(MB, dtype=np.float32)
            s[rng.random(MB) < 0.5] = -0.0
        else:
            s = rng.standard_normal(MB).astype(np.float32)
        scores[i // G, 0, i % G] = s
    r = np.array([[0, 15, 16, 31, MB - 1][b % 5] if b % 6 else int(rng.integers(0, MB)) for b in range(B)])
    pos = r * 128 + rng.integers(0, 128, size=B)
    lens = (pos + 1).astype(np.int32)
    table = np.zeros((B, MB), dtype=np.int32)
    batch = msa.Batch(torch.from_numpy(table).cuda(), torch.from_numpy(lens).cuda(), 1)
    cfg = msa.Config(num_kv_groups=G, heads_per_group=1)
    sel = torch.full((B, 1, G, 16), 99, dtype=torch.int32, device="cuda")
    msa.msa_select_blocks(cfg, batch, torch.from_numpy(scores).cuda(), sel)
    torch.cuda.synchronize()
    got = to_np(sel)
    for b in range(B):
        for g in range(G):
            want = OM.select_row(scores[b, 0, g].astype(np.float64), int(pos[b]))
            assert np.array_equal(got[b, 0, g], want), (b, g)


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_attention_on_oracle_selection(case):
    need_gpu()
    import torch
    import block_sparse_attention_indexer_gb300 as msa
    w, dw, cache, table, lens, q, qi = _setup(*case)
    for i in range(4):
        assert np.array_equal(to_np(dw.cache.tensors()[i]), cache[i])
    assert np.array_equal(to_np(dw.q), q)
    ref_scores = OM.block_scores(qi, cache[4], cache[5], table, lens)
    sel = OM.select_blocks(ref_scores, lens)
    out_ref, lse_ref = OM.sparse_attention(q, *cache[:4], table, lens, sel, w.heads_per_group)
    B, T, H = w.batch, w.q_len, w.num_heads
    out = torch.zeros(B, T, H, 128, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros(B, T, H, dtype=torch.float32, device="cuda")
    ws = msa.alloc_workspace(msa.MSA_OP_SPARSE_ATTN, dw.cfg, dw.batch)
    msa.msa_sparse_attn_decode(dw.cfg, dw.cache, dw.batch, dw.q, torch.from_numpy(sel).cuda(), out, lse, ws)
    torch.cuda.synchronize()
    assert msa.msa_read_device_error(ws) == 0
    assert_out_close(bf16_to_np(out), out_ref)
    assert np.allclose(to_np(lse), lse_ref, rtol=1e-4, atol=1e-4)


def test_attention_uniform_values_equal_value_row():
    need_gpu()
    import torch
    import block_sparse_attention_indexer_gb300 as msa
    w, lens = syn.custom("uni", 3, 2, 2, 8, [3000, 700])
    dw = device_workload(w, lens)
    # the expected row: the oracle's own quantisation of value token 5, head 0 of block 0
    _, v, _ = syn.gen_block_fp32(w, 0, 0)
    d_ref, s_ref = OF.nvfp4_quantize(v[5, 0][None, :])
    row = OF.nvfp4_dequantize(d_ref, s_ref)[0]
    page0 = int(dw.table[0, 0])
    assert np.array_equal(to_np(dw.cache.v_data[page0, 0, 5]), d_ref[0])
    dw.cache.v_data[:] = dw.cache.v_data[page0, 0, 5].clone()
    dw.cache.v_scale[:] = dw.cache.v_scale[page0, 0, 5].clone()
    out = torch.zeros(2, 2, 32, 128, dtype=torch.bfloat16, device="cuda")
    sel_out = torch.zeros(2, 2, 4, 16, dtype=torch.int32, device="cuda")
    ws = msa.alloc_workspace(msa.MSA_OP_DECODE, dw.cfg, dw.batch)
    msa.msa_decode(dw.cfg, dw.cache, dw.batch, dw.q, dw.qi, out, None, sel_out, ws)
    torch.cuda.synchronize()
    want = torch.tensor(row, dtype=torch.float32).to(torch.bfloat16).float().numpy()
    got = bf16_to_np(out)
    assert np.abs(got - want[None, None, None, :]).max() <= 2.0 ** -8 * np.abs(want).max()


@pytest.mark.parametrize("case", [c for c in CASES if c[2] >= 64], ids=[c[0] for c in CASES if c[2] >= 64])
def test_block_major_attention_repeatable_and_matches_team_kernel(case):
    """From 64 query tokens on the attention runs block-major (CSR plan, tcgen05 tiles, partial
    states, merge).  Every partial is computed on its own and merged in slot order, so repeated
    calls must give bit-identical results (a race between the kernel's warp roles shows up as a
    difference); the query-major team kernel (the no-allocation entry point always runs it)
    computes the same attention."""
    need_gpu()
    import torch
    import block_sparse_attention_indexer_gb300 as msa
    w, dw, cache, table, lens, q, qi = _setup(*case)
    ref_scores = OM.block_scores(qi, cache[4], cache[5], table, lens)
    sel = torch.from_numpy(OM.select_blocks(ref_scores, lens)).cuda()
    B, T, H = w.batch, w.q_len, w.num_heads
    ws = msa.alloc_workspace(msa.MSA_OP_SPARSE_ATTN, dw.cfg, dw.batch)
    outs = []
    for _ in range(5):
        out = torch.zeros(B, T, H, 128, dtype=torch.bfloat16, device="cuda")
        lse = torch.zeros(B, T, H, dtype=torch.float32, device="cuda")
        msa.msa_sparse_attn_decode(dw.cfg, dw.cache, dw.batch, dw.q, sel, out, lse, ws)
        outs.append((out, lse))
    torch.cuda.synchronize()
    assert msa.msa_read_device_error(ws) == 0
    for out, lse in outs[1:]:
        assert torch.equal(out, outs[0][0]) and torch.equal(lse, outs[0][1])
    team = torch.zeros(B, T, H, 128, dtype=torch.bfloat16, device="cuda")
    team_lse = torch.zeros(B, T, H, dtype=torch.float32, device="cuda")
    msa.msa_sparse_attn_decode_noalloc(dw.cfg, dw.cache, dw.batch, dw.q, sel, team, team_lse)
    torch.cuda.synchronize()
    err = np.abs(bf16_to_np(outs[0][0]) - bf16_to_np(team))
    assert err.max() <= 2e-2 and err.mean() <= 2e-3
    assert np.allclose(to_np(outs[0][1]), to_np(team_lse), rtol=1e-4, atol=1e-4)


def test_block_major_plan_wide_table():
    """The block-major plan counts each 128-token chunk's blocks in a shared-memory histogram
    when a row has at most 12,288 blocks and with global atomics beyond: the same sequences
    with the block table padded to 12,289 columns (-1 past each sequence) take the second
    form and must give bit-identical outputs, both matching the oracle."""
    need_gpu()
    import torch
    import block_sparse_attention_indexer_gb300 as msa
    w, dw, cache, table, lens, q, qi = _setup("prefill_hg4_t80", [80, 3000 + 1], 80, 4, True)
    ref_scores = OM.block_scores(qi, cache[4], cache[5], table, lens)
    sel_np = OM.select_blocks(ref_scores, lens)
    out_ref, lse_ref = OM.sparse_attention(q, *cache[:4], table, lens, sel_np, w.heads_per_group)
    sel = torch.from_numpy(sel_np).cuda()
    B, T, H = w.batch, w.q_len, w.num_heads
    wide = torch.full((B, 12289), -1, dtype=torch.int32, device="cuda")
    wide[:, :table.shape[1]] = dw.batch.block_table
    batches = [dw.batch, msa.Batch(wide, dw.batch.seq_lens, T)]
    res = []
    for batch in batches:
        out = torch.zeros(B, T, H, 128, dtype=torch.bfloat16, device="cuda")
        lse = torch.zeros(B, T, H, dtype=torch.float32, device="cuda")
        ws = msa.alloc_workspace(msa.MSA_OP_SPARSE_ATTN, dw.cfg, batch)
        msa.msa_sparse_attn_decode(dw.cfg, dw.cache, batch, dw.q, sel, out, lse, ws)
        torch.cuda.synchronize()
        assert msa.msa_read_device_error(ws) == 0
        assert_out_close(bf16_to_np(out), out_ref)
        assert np.allclose(to_np(lse), lse_ref, rtol=1e-4, atol=1e-4)
        res.append((out, lse))
    assert torch.equal(res[0][0], res[1][0]) and torch.equal(res[0][1], res[1][1])
