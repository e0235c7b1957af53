"""The usage example of the README, run as written: a paged NVFP4 cache filled with
msa_nvfp4_insert, FP8 queries from msa_fp8_quantize, one msa_decode step.  Its output must be
finite and agree with the three stage calls on the same inputs."""
import pytest

from gpu_util import need_gpu

pytestmark = pytest.mark.gpu


def test_readme_example_runs():
    need_gpu()
    # ---- begin README example
    import torch
    import block_sparse_attention_indexer_gb300 as msa

    cfg = msa.Config(num_kv_groups=4, heads_per_group=8)       # 32 query heads, 4 KV heads
    P, B, L = 1024, 2, 20000                                   # pages, sequences, tokens each
    cache = msa.PagedCache(P)                                  # NVFP4 K, V and index-key pools
    nb = -(-L // 128)
    table = torch.arange(B * nb, dtype=torch.int32, device="cuda").view(B, nb)  # block -> page
    lens = torch.full((B,), L, dtype=torch.int32, device="cuda")
    # every token's K, V (4 KV heads) and index key (one head) into its page slot
    slots = (table.long()[:, :, None] * 128 + torch.arange(128, device="cuda")).view(B, -1)[:, :L].reshape(-1)
    msa.msa_nvfp4_insert(torch.randn(B * L, 4, 128, device="cuda"), slots, cache.k_data, cache.k_scale)
    msa.msa_nvfp4_insert(torch.randn(B * L, 4, 128, device="cuda"), slots, cache.v_data, cache.v_scale)
    msa.msa_nvfp4_insert(torch.randn(B * L, 1, 128, device="cuda"), slots,
                         cache.idx_data.view(P, 1, 128, 64), cache.idx_scale.view(P, 1, 128, 8))
    # one decode step: FP8 queries (32 heads) and index queries (one per KV group)
    batch = msa.Batch(table, lens, q_len=1)
    q = torch.empty(B, 1, 32, 128, dtype=torch.uint8, device="cuda")
    qi = torch.empty(B, 1, 4, 128, dtype=torch.uint8, device="cuda")
    msa.msa_fp8_quantize(torch.randn(B, 1, 32, 128, device="cuda"), q)
    msa.msa_fp8_quantize(torch.randn(B, 1, 4, 128, device="cuda"), qi)
    out = torch.empty(B, 1, 32, 128, dtype=torch.bfloat16, device="cuda")
    ws = msa.alloc_workspace(msa.MSA_OP_DECODE, cfg, batch)
    msa.msa_decode(cfg, cache, batch, q, qi, out, None, None, ws)  # indexer -> top-16 -> sparse attention
    assert msa.msa_read_device_error(ws) == 0
    # ---- end README example
    assert torch.isfinite(out.float()).all()
    scores = torch.empty(B, 1, 4, nb, dtype=torch.float32, device="cuda")
    msa.msa_indexer_scores(cfg, cache, batch, qi, scores, msa.alloc_workspace(msa.MSA_OP_INDEXER_SCORES, cfg, batch))
    sel = torch.empty(B, 1, 4, 16, dtype=torch.int32, device="cuda")
    msa.msa_select_blocks(cfg, batch, scores, sel)
    out2 = torch.empty_like(out)
    msa.msa_sparse_attn_decode(cfg, cache, batch, q, sel, out2, None,
                               msa.alloc_workspace(msa.MSA_OP_SPARSE_ATTN, cfg, batch))
    torch.cuda.synchronize()
    assert torch.equal(out, out2)
