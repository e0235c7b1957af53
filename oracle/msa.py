"""Plain CPU oracle of MiniMax Sparse Attention (MSA) decode over an NVFP4 paged cache.

TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and bench.py's
cpu_baseline / reference leg may import this module.  It shares no code with the CUDA
path (block_sparse_attention_indexer_gb300) and never imports it.

Everything is computed in float64 from the exact values of the cache bytes.  Each
function restates one step of the method as the pages define it:

  * scoring: every cached key is scored with one index query per GQA group against a
    single shared index-key head; scores are max-pooled to one score per 128-token
    block; attention runs exactly over the top-16 blocks, the most recent block always
    kept, so at most 2,048 keys per query
    ("vLLM liefert Day-0-Unterstützung für MiniMax-M3.1-Flash", §MSA-Grundlagen);
  * block rules: init_blocks = 0, local_blocks = 1; the incomplete tail block is masked,
    the causal boundary inside a block is respected, a local block that also makes the
    top-k is not counted twice, requests have different valid block ranges
    ("MiniMax M3 x vLLM：百万 token 多模态推理的 Day-0 部署", §MSA 机制细节);
  * selection per query token and KV group, then sparse GQA equal to dense attention
    restricted to the selected set (same page, §Prefill 执行, steps 2-4);
  * configuration variants the pages name: the block-score reduction is max or
    log-sum-exp by model configuration (same page, §Prefill 执行 step 2); init_blocks
    leading and local_blocks trailing blocks are kept by rule, the rest come from the top-k
    of the indexer scores, none counted twice (same page, §MSA 机制细节);
  * speculative tokens flattened request-major, each with its own causal position
    (same page, §Decode Kernel 中的投机解码);
  * decode context parallelism: local top-16 per shard, merged exactly by the owner
    (first page, §NVFP4-Indexer-DCP).

Readings where the pages are silent (all listed in the design notes): the query
position of token t of sequence b is pos = L_b - T + t (the new tokens are already in
the cache); key j is visible iff j <= pos; the recent block is r = pos // 128 and is
counted inside the 16; ties in the block ranking go to the lower block index; the
softmax scale is 1/sqrt(128); query head h belongs to KV group h // Hg.
"""
from __future__ import annotations

import math
from typing import List, Sequence, Tuple

import numpy as np

from .formats import E4M3_TABLE, nvfp4_dequantize

BLOCK = 128
TOP_K = 16


# --------------------------------------------------------------------------------------
# cache access
# --------------------------------------------------------------------------------------
def index_keys(idx_data, idx_scale, block_table_row, length: int) -> np.ndarray:
    """Exact index keys of one sequence, [length, Di] float64 (pages looked up through the
    block table, then concatenated in logical order)."""
    nb = -(-length // BLOCK)
    pages = np.asarray(block_table_row[:nb], dtype=np.int64)
    keys = nvfp4_dequantize(idx_data[pages], idx_scale[pages])      # [nb, 128, Di]
    return keys.reshape(nb * BLOCK, -1)[:length]


def kv_rows(data, scale, block_table_row, group: int, blocks: Sequence[int]) -> np.ndarray:
    """Exact K (or V) rows of KV head `group` for the given logical blocks,
    [len(blocks)*128, D] float64."""
    pages = np.asarray([block_table_row[n] for n in blocks], dtype=np.int64)
    if len(pages) == 0:
        return np.zeros((0, data.shape[-1] * 2))
    rows = nvfp4_dequantize(data[pages, group], scale[pages, group])  # [nsel, 128, D]
    return rows.reshape(len(pages) * BLOCK, -1)


def query_positions(length: int, q_len: int) -> np.ndarray:
    return np.arange(length - q_len, length, dtype=np.int64)


# --------------------------------------------------------------------------------------
# stage 1: indexer score + block max-pool
# --------------------------------------------------------------------------------------
def pool_block(values: np.ndarray, pooling: str, axis: int) -> np.ndarray:
    """One score per block from its keys' scores (-inf = not visible): their maximum, or
    their log-sum-exp ln(sum_j e^{s_j}) (natural log); -inf for a block with no visible key."""
    m = values.max(axis=axis)
    if pooling == "max":
        return m
    assert pooling == "lse", pooling
    mk = np.expand_dims(np.where(np.isfinite(m), m, 0.0), axis)
    with np.errstate(divide="ignore"):
        return np.where(np.isfinite(m), np.squeeze(mk, axis) + np.log(np.exp(values - mk).sum(axis=axis)), m)


def block_scores(qi_codes, idx_data, idx_scale, block_table, seq_lens, max_blocks: int | None = None,
                 rows_per_matmul: int = 256, tokens=None, sequences=None, pooling: str = "max") -> np.ndarray:
    """Block scores S[b, t, g, n] = pool over visible keys j of block n of qi[b,t,g] . k_j,
    pool = max (the recipe) or log-sum-exp.

    qi_codes: uint8 E4M3 [B, T, G, Di].  A block with no visible key scores -inf (every
    block after the query's own block, and every block past the sequence end).
    Returns float64 [B, T, G, max_blocks].  `tokens` / `sequences` restrict the work to
    those query-token indices / sequences (the other rows stay -inf).
    """
    B, T, G, _ = qi_codes.shape
    if max_blocks is None:
        max_blocks = block_table.shape[1]
    out = np.full((B, T, G, max_blocks), -np.inf)
    ts_all = np.arange(T) if tokens is None else np.asarray(sorted(tokens), dtype=np.int64)
    step = max(1, rows_per_matmul // G)
    for b in (range(B) if sequences is None else sequences):
        L = int(seq_lens[b])
        if L <= 0:
            continue
        keys = index_keys(idx_data, idx_scale, block_table[b], L)    # [L, Di]
        nb = -(-L // BLOCK)
        qi = E4M3_TABLE[qi_codes[b]]                                  # [T, G, Di]
        pos_all = query_positions(L, T)
        for c0 in range(0, len(ts_all), step):
            ts = ts_all[c0:c0 + step]
            s = keys @ qi[ts].reshape(-1, qi.shape[-1]).T             # [L, len(ts)*G]
            s = s.reshape(L, len(ts), G)
            padded = np.full((nb * BLOCK, len(ts), G), -np.inf)
            padded[:L] = s
            j = np.arange(nb * BLOCK)[:, None]
            visible = j <= pos_all[ts][None, :]                       # [nb*128, len(ts)]
            padded = np.where(visible[:, :, None], padded, -np.inf)
            pooled = pool_block(padded.reshape(nb, BLOCK, len(ts), G), pooling, axis=1)  # [nb, len(ts), G]
            out[b, ts, :, :nb] = pooled.transpose(1, 2, 0)
    return out


# --------------------------------------------------------------------------------------
# stage 2: top-k block selection with the recent block forced
# --------------------------------------------------------------------------------------
def rank_key(score: float, n: int):
    """Sort key of candidate block n: higher score first, then lower index; NaN ranks
    below every number (including -inf)."""
    if math.isnan(score):
        return (1, 0.0, n)
    return (0, -score, n)


def select_row(scores_row: np.ndarray, pos: int, top_k: int = TOP_K, init_blocks: int = 0,
               local_blocks: int = 1) -> np.ndarray:
    """Selected logical blocks of one (query token, KV group), min(top_k, r + 1) of them with
    r = pos // 128 the recent block: the first init_blocks blocks and the last local_blocks
    blocks up to r are kept by rule (each once), and the remaining places go to the best of
    the other blocks up to r; ascending; -1 padded.  The recipe (init 0, local 1) is the
    recent block plus the top-(k-1) of the blocks before it."""
    assert init_blocks + local_blocks <= top_k
    r = pos // BLOCK
    forced = set(range(min(init_blocks, r + 1))) | set(range(max(0, r - local_blocks + 1), r + 1))
    cands = sorted((n for n in range(r + 1) if n not in forced), key=lambda n: rank_key(float(scores_row[n]), n))
    chosen = sorted(forced | set(cands[: max(0, top_k - len(forced))]))
    out = np.full(top_k, -1, dtype=np.int32)
    out[: len(chosen)] = chosen
    return out


def select_blocks(scores, seq_lens, top_k: int = TOP_K, init_blocks: int = 0, local_blocks: int = 1) -> np.ndarray:
    """sel[b, t, g, :] for every row; scores [B, T, G, max_blocks]."""
    B, T, G, _ = scores.shape
    sel = np.full((B, T, G, top_k), -1, dtype=np.int32)
    for b in range(B):
        L = int(seq_lens[b])
        if L <= 0:
            continue
        for t, pos in enumerate(query_positions(L, T)):
            for g in range(G):
                sel[b, t, g] = select_row(scores[b, t, g], int(pos), top_k, init_blocks, local_blocks)
    return sel


# --------------------------------------------------------------------------------------
# stage 3: exact sparse GQA attention over the selected blocks
# --------------------------------------------------------------------------------------
def sparse_attention(q_codes, k_data, k_scale, v_data, v_scale, block_table, seq_lens, sel,
                     heads_per_group: int, softmax_scale: float | None = None, tokens=None, sequences=None):
    """Attention of every query head over the visible keys of its group's selected blocks.

    q_codes: uint8 E4M3 [B, T, H, D]; sel: int32 [B, T, G, k].
    Returns (out float64 [B, T, H, D], lse float64 [B, T, H]) with lse the natural log of
    the softmax denominator including the row max.  `tokens` / `sequences` restrict the
    work to those rows (the others stay 0 / -inf).
    """
    B, T, H, D = q_codes.shape
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(D)
    out = np.zeros((B, T, H, D))
    lse = np.full((B, T, H), -np.inf)
    for b in (range(B) if sequences is None else sequences):
        L = int(seq_lens[b])
        if L <= 0:
            continue
        q = E4M3_TABLE[q_codes[b]]                                     # [T, H, D]
        positions = query_positions(L, T)
        for t in (range(T) if tokens is None else tokens):
            pos = int(positions[t])
            for g in range(sel.shape[2]):
                blocks = [int(n) for n in sel[b, t, g] if n >= 0]
                K = kv_rows(k_data, k_scale, block_table[b], g, blocks)
                V = kv_rows(v_data, v_scale, block_table[b], g, blocks)
                j = np.concatenate([np.arange(n * BLOCK, (n + 1) * BLOCK) for n in blocks]) if blocks \
                    else np.zeros(0, dtype=np.int64)
                keep = (j <= pos) & (j < L)
                K, V = K[keep], V[keep]
                for h in range(g * heads_per_group, (g + 1) * heads_per_group):
                    logits = (K @ q[t, h]) * softmax_scale
                    m = logits.max()
                    p = np.exp(logits - m)
                    l = p.sum()
                    out[b, t, h] = (p @ V) / l
                    lse[b, t, h] = m + math.log(l)
    return out, lse


def dense_causal_attention(q_codes, k_data, k_scale, v_data, v_scale, block_table, seq_lens,
                           heads_per_group: int, softmax_scale: float | None = None):
    """Ordinary causal GQA attention over the whole cache (no block selection), written
    independently of sparse_attention; MSA must equal it whenever a query has at most
    16 blocks to choose from."""
    from scipy.special import logsumexp, softmax

    B, T, H, D = q_codes.shape
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(D)
    out = np.zeros((B, T, H, D))
    lse = np.zeros((B, T, H))
    for b in range(B):
        L = int(seq_lens[b])
        nb = -(-L // BLOCK)
        pages = np.asarray(block_table[b, :nb], dtype=np.int64)
        q = E4M3_TABLE[q_codes[b]]
        for h in range(H):
            g = h // heads_per_group
            K = nvfp4_dequantize(k_data[pages, g], k_scale[pages, g]).reshape(nb * BLOCK, D)[:L]
            V = nvfp4_dequantize(v_data[pages, g], v_scale[pages, g]).reshape(nb * BLOCK, D)[:L]
            for t in range(T):
                pos = L - T + t
                logits = K[: pos + 1] @ q[t, h] * softmax_scale
                out[b, t, h] = softmax(logits) @ V[: pos + 1]
                lse[b, t, h] = logsumexp(logits)
    return out, lse


def msa_decode(q_codes, qi_codes, cache, block_table, seq_lens, heads_per_group: int,
               top_k: int = TOP_K, init_blocks: int = 0, local_blocks: int = 1, pooling: str = "max"):
    """The whole decode step: scores -> selection -> attention.
    cache = (k_data, k_scale, v_data, v_scale, idx_data, idx_scale)."""
    k_data, k_scale, v_data, v_scale, idx_data, idx_scale = cache
    s = block_scores(qi_codes, idx_data, idx_scale, block_table, seq_lens, pooling=pooling)
    sel = select_blocks(s, seq_lens, top_k, init_blocks, local_blocks)
    out, lse = sparse_attention(q_codes, k_data, k_scale, v_data, v_scale, block_table, seq_lens, sel,
                                heads_per_group)
    return s, sel, out, lse


# --------------------------------------------------------------------------------------
# split-K merge of partial attention states
# --------------------------------------------------------------------------------------
def merge_partials(parts: List[Tuple[float, float, np.ndarray]]):
    """Combine partial softmax states (m_s, l_s, o_s) over disjoint key subsets, where
    o_s = sum_j exp(x_j - m_s) v_j and l_s = sum_j exp(x_j - m_s):
    out = sum_s e^{m_s - M} o_s / sum_s e^{m_s - M} l_s, lse = M + log(sum_s e^{m_s - M} l_s)."""
    M = max(m for m, _, _ in parts)
    num = sum(math.exp(m - M) * o for m, _, o in parts)
    den = sum(math.exp(m - M) * l for m, l, _ in parts)
    return num / den, M + math.log(den)


# --------------------------------------------------------------------------------------
# decode context parallelism: local top-k per context shard, exact merge at the owner
# --------------------------------------------------------------------------------------
def dcp_local_candidates(scores_row: np.ndarray, pos: int, lo: int, hi: int, top_k: int = TOP_K):
    """A shard owning blocks [lo, hi) keeps its best top_k-1 candidates among the blocks
    before the recent one, as (score, block) pairs ranked like select_row."""
    r = pos // BLOCK
    cands = [n for n in range(lo, min(hi, r))]
    cands.sort(key=lambda n: rank_key(float(scores_row[n]), n))
    return [(float(scores_row[n]), n) for n in cands[: top_k - 1]]


def dcp_merge(candidate_lists, pos: int, top_k: int = TOP_K) -> np.ndarray:
    """The owner merges the shards' candidate lists into the final selection."""
    allc = [c for lst in candidate_lists for c in lst]
    allc.sort(key=lambda sn: rank_key(sn[0], sn[1]))
    chosen = sorted([n for _, n in allc[: top_k - 1]] + [pos // BLOCK])
    out = np.full(top_k, -1, dtype=np.int32)
    out[: len(chosen)] = chosen
    return out


# --------------------------------------------------------------------------------------
# byte accounting (algorithmic HBM bytes of one decode step)
# --------------------------------------------------------------------------------------
NVFP4_BYTES_PER_ELEMENT = 0.5 + 1.0 / 16.0          # 4-bit value + one 8-bit scale per 16


def index_key_bytes_per_token(index_dim: int = 128) -> int:
    return int(index_dim * NVFP4_BYTES_PER_ELEMENT)


def kv_bytes_per_token_per_head(head_dim: int = 128) -> int:
    """K plus V of one KV head."""
    return int(2 * head_dim * NVFP4_BYTES_PER_ELEMENT)


def decode_step_bytes(seq_lens, sel, index_dim: int = 128, head_dim: int = 128):
    """(index-key bytes, selected K/V bytes) of one decode step: the indexer reads every
    cached index key once per sequence; attention reads, per (sequence, KV group), every
    block selected by any of the sequence's query tokens once."""
    idx = sum(int(L) for L in seq_lens) * index_key_bytes_per_token(index_dim)
    kv = 0
    B, T, G, _ = sel.shape
    for b in range(B):
        for g in range(G):
            union = {int(n) for n in sel[b, :, g].ravel() if n >= 0}
            kv += len(union) * BLOCK * kv_bytes_per_token_per_head(head_dim)
    return idx, kv
