"""Pins of the oracle's MSA steps against things other than its own formulas: exact
rational brute force on tiny inputs, special cases with closed forms, subset brute force
for the selection, an independently written dense attention (scipy softmax), structural
invariants the pages state, and the byte counts the pages print."""
import itertools
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

from oracle import cache as C
from oracle import formats as F
from oracle import msa as M
from workloads import synthetic as syn

GOLD = os.path.join(os.path.dirname(__file__), "golden")
FACTS = json.load(open(os.path.join(GOLD, "page_facts.json")))


def small_case(lens, q_len=1, hg=4, seed=5, shuffled=True, offset_std=2.0):
    w, lens = syn.custom("t", seed, len(lens), q_len, hg, lens, shuffled=shuffled, offset_std=offset_std)
    cache, table, lens, P = C.build_cache(w, lens)
    q, qi = C.encode_queries(w)
    return w, cache, table, lens, q, qi


# ------------------------------------------------------------------ page facts / bytes
def test_constants_match_page_facts():
    assert M.BLOCK == FACTS["block_size_tokens"]["value"]
    assert M.TOP_K == FACTS["top_k_blocks"]["value"]
    assert M.BLOCK * M.TOP_K == FACTS["max_keys_per_query"]["value"]


def test_byte_accounting_matches_pages():
    fp8_idx = FACTS["index_key_bytes_per_token_fp8"]["value"]
    fp8_kv = FACTS["dense_kv_bytes_per_token_fp8"]["value"]
    heads = FACTS["kv_heads"]["value"]
    d = FACTS["head_dim"]["value"]
    assert fp8_idx == d * 1 and fp8_kv == heads * d * 2 * 1          # FP8: one byte per element
    nv_idx = M.index_key_bytes_per_token()
    nv_kv = heads * M.kv_bytes_per_token_per_head()
    assert (nv_idx, nv_kv) == (72, 576)
    assert Fraction(nv_idx, nv_kv) == Fraction(fp8_idx, fp8_kv) == Fraction(FACTS["index_to_dense_ratio"]["value"])
    # decode traffic vs dense tends to 1/8 for long contexts (the pages' "about 12.5%")
    L = 1 << 22
    sel = np.tile(np.arange(16, dtype=np.int32), (1, 1, 4, 1))
    idx, kv = M.decode_step_bytes([L], sel)
    frac = (idx + kv) / (L * nv_kv)
    assert abs(frac - FACTS["long_context_traffic_fraction"]["value"]) < 2e-3
    idx, kv = M.decode_step_bytes([131072], sel)
    # at 128K the 16 selected blocks of 4 groups add 4*2048*144 / (576*131072) = 1/64
    assert abs((idx + kv) / (131072 * nv_kv) - (0.125 + 1 / 64)) < 1e-12


# ------------------------------------------------------------------ stage 1 pins
def _exact_scores_bruteforce(qi_codes, cache, table, lens):
    """Pure-Python exact rational block scores, decoding nibbles bit by bit."""
    _, _, _, _, idx_data, idx_scale = cache

    def e2m1(c):
        s, e, m = c >> 3, (c >> 1) & 3, c & 1
        mag = Fraction(m, 2) if e == 0 else Fraction(2) ** (e - 1) * (1 + Fraction(m, 2))
        return -mag if s else mag

    def e4m3(c):
        s, e, m = c >> 7, (c >> 3) & 15, c & 7
        mag = Fraction(m, 8) * Fraction(1, 64) if e == 0 else (1 + Fraction(m, 8)) * Fraction(2) ** (e - 7)
        return -mag if s else mag

    B, T, G, Di = qi_codes.shape
    out = {}
    for b in range(B):
        L = int(lens[b])
        for t in range(T):
            pos = L - T + t
            for g in range(G):
                q = [e4m3(int(c)) for c in qi_codes[b, t, g]]
                for n in range(-(-L // 128)):
                    page = int(table[b, n])
                    best = None
                    for i in range(128):
                        j = n * 128 + i
                        if j > pos or j >= L:
                            continue
                        row = idx_data[page, i]
                        sc = idx_scale[page, i]
                        s = Fraction(0)
                        for d in range(Di):
                            byte = int(row[d // 2])
                            code = byte & 15 if d % 2 == 0 else byte >> 4
                            s += q[d] * e2m1(code) * e4m3(int(sc[d // 16]))
                        best = s if best is None or s > best else best
                    out[(b, t, g, n)] = best
    return out


def test_block_scores_match_exact_rational_bruteforce():
    # two sequences, ragged tail (300 = 2 blocks + 44 tokens), two query tokens
    w, cache, table, lens, q, qi = small_case([300, 200], q_len=2, hg=1, seed=21)
    s = M.block_scores(qi, cache[4], cache[5], table, lens)
    ref = _exact_scores_bruteforce(qi[:, :, :1], cache, table, lens)   # one group keeps it fast
    for (b, t, g, n), v in ref.items():
        if v is None:
            assert s[b, t, g, n] == -np.inf
        else:
            assert abs(s[b, t, g, n] - float(v)) <= 1e-9 * max(1.0, abs(float(v)))


def test_identical_keys_block_score_is_the_dot_product():
    w, cache, table, lens, q, qi = small_case([512], q_len=1, seed=3)
    idx_data, idx_scale = cache[4], cache[5]
    page = table[0, 1]
    idx_data[page] = idx_data[page, 7]            # every key of block 1 equals key 7 of it
    idx_scale[page] = idx_scale[page, 7]
    s = M.block_scores(qi, idx_data, idx_scale, table, lens)
    k = F.nvfp4_dequantize(idx_data[page, 7], idx_scale[page, 7])
    for g in range(4):
        assert s[0, 0, g, 1] == pytest.approx(float(F.e4m3_decode(qi[0, 0, g]) @ k), rel=1e-12)


def test_causal_and_tail_masking():
    # a key planted far above the rest must win its block only where it is visible
    w, cache, table, lens, q, qi = small_case([260], q_len=8, seed=4)
    idx_data, idx_scale = cache[4], cache[5]
    qi[0, :, 0] = qi[0, 0, 0]                        # the same index query at every position
    qv = F.e4m3_decode(qi[0, 0, 0])
    j = 255                                          # position 255: block 1, last slot
    p, i = table[0, j // 128], j % 128
    big = np.sign(qv).astype(np.float32) * 6.0
    d, sc = F.nvfp4_quantize((big * 100).astype(np.float32)[None, :])
    idx_data[p, i], idx_scale[p, i] = d[0], sc[0]
    # garbage past the sequence end (tokens 260..383 of block 2) must never count
    p2 = table[0, 2]
    idx_data[p2, 10:], idx_scale[p2, 10:] = d[0], sc[0]
    s = M.block_scores(qi, idx_data, idx_scale, table, lens)
    pos = np.arange(260 - 8, 260)                    # 252 .. 259
    k_big = float(qv @ F.nvfp4_dequantize(d[0], sc[0]))
    for t in range(8):
        if pos[t] >= j:
            assert s[0, t, 0, 1] == pytest.approx(k_big, rel=1e-12)
        else:
            assert s[0, t, 0, 1] < k_big / 2
        assert s[0, t, 0, 2] == -np.inf if pos[t] < 256 else np.isfinite(s[0, t, 0, 2])
        if pos[t] >= 256:
            assert s[0, t, 0, 2] < k_big / 2         # the garbage tail stayed masked
        assert (s[0, t, 0, 3:] == -np.inf).all()


def test_page_relabelling_invariance():
    w, cache, table, lens, q, qi = small_case([700, 333], q_len=3, seed=8)
    s1 = M.block_scores(qi, cache[4], cache[5], table, lens)
    P = cache[4].shape[0]
    perm = np.random.default_rng(0).permutation(P)
    inv = np.argsort(perm)
    cache2 = tuple(a[perm] for a in cache)             # physical page p moves to inv[p]
    table2 = np.where(table >= 0, inv[np.maximum(table, 0)], -1).astype(np.int32)
    s2 = M.block_scores(qi, cache2[4], cache2[5], table2, lens)
    assert np.array_equal(s1, s2)


# ------------------------------------------------------------------ stage 2 pins
def _subset_bruteforce(scores_row, r, k):
    """All subsets of the blocks before r of size min(k-1, r): the one with the largest
    score sum, ties to the lexicographically smallest; then add r."""
    best = None
    m = min(k - 1, r)
    for sub in itertools.combinations(range(r), m):
        tot = sum(scores_row[n] for n in sub)
        if best is None or tot > best[0] or (tot == best[0] and sub < best[1]):
            best = (tot, sub)
    return sorted(list(best[1]) + [r])


def test_select_equals_subset_bruteforce_with_ties():
    rng = np.random.default_rng(2)
    k = 4
    for trial in range(300):
        r = int(rng.integers(0, 9))
        row = rng.integers(-3, 4, size=12).astype(np.float64)    # many exact ties
        got = M.select_row(row, r * 128 + int(rng.integers(0, 128)), top_k=k)
        want = _subset_bruteforce(row, r, k)
        assert [int(x) for x in got if x >= 0] == want
        assert (got[len(want):] == -1).all()


def test_select_invariants_and_nan_rank():
    rng = np.random.default_rng(9)
    for _ in range(200):
        nb = int(rng.integers(1, 60))
        row = rng.standard_normal(64)
        row[rng.random(64) < 0.1] = -np.inf
        pos = int(rng.integers(0, nb * 128))
        sel = M.select_row(row, pos)
        r = pos // 128
        chosen = sel[sel >= 0]
        assert len(chosen) == min(16, r + 1)
        assert r in chosen and (chosen <= r).all()
        assert (np.diff(chosen) > 0).all()
        assert len(chosen) * 128 <= FACTS["max_keys_per_query"]["value"]
    row = np.array([np.nan, -np.inf, 1.0, np.nan, 0.0])
    sel = M.select_row(row, 5 * 128, top_k=4)        # r = 5; 3 picks among 0..4
    assert sel.tolist() == [1, 2, 4, 5]               # 1.0, 0.0, -inf beat the NaNs


# ------------------------------------------------------------------ stage 3 pins
def test_sparse_equals_dense_when_at_most_16_blocks():
    w, cache, table, lens, q, qi = small_case([2048, 1000], q_len=3, hg=2, seed=13)
    s, sel, out, lse = M.msa_decode(q, qi, cache, table, lens, heads_per_group=2)
    ref, ref_lse = M.dense_causal_attention(q, *cache[:4], table, lens, heads_per_group=2)
    assert np.allclose(out, ref, rtol=1e-12, atol=1e-12)
    assert np.allclose(lse, ref_lse, rtol=1e-12, atol=1e-12)


def test_sparse_equals_dense_restricted_to_selected_set():
    from scipy.special import softmax
    w, cache, table, lens, q, qi = small_case([4096 + 77], q_len=2, hg=2, seed=17)
    s, sel, out, lse = M.msa_decode(q, qi, cache, table, lens, heads_per_group=2)
    L = int(lens[0])
    nb = -(-L // 128)
    pages = table[0, :nb]
    for t in range(2):
        pos = L - 2 + t
        for h in range(8):
            g = h // 2
            K = F.nvfp4_dequantize(cache[0][pages, g], cache[1][pages, g]).reshape(-1, 128)[:L]
            V = F.nvfp4_dequantize(cache[2][pages, g], cache[3][pages, g]).reshape(-1, 128)[:L]
            logits = K @ F.e4m3_decode(q[0, t, h]) / math.sqrt(128)
            allowed = np.zeros(L, bool)
            for n in sel[0, t, g]:
                if n >= 0:
                    allowed[n * 128:(n + 1) * 128] = True
            allowed[pos + 1:] = False
            logits = np.where(allowed, logits, -np.inf)
            assert np.allclose(out[0, t, h], softmax(logits) @ V, rtol=1e-10, atol=1e-12)


def test_uniform_values_and_single_key():
    w, cache, table, lens, q, qi = small_case([3000], q_len=1, seed=19)
    v_data, v_scale = cache[2], cache[3]
    v_data[:] = v_data[0, 0, 5]                       # every value row identical
    v_scale[:] = v_scale[0, 0, 5]
    s, sel, out, lse = M.msa_decode(q, qi, cache, table, lens, heads_per_group=4)
    row = F.nvfp4_dequantize(v_data[0, 0, 5], v_scale[0, 0, 5])
    assert np.allclose(out, row[None, None, None, :], rtol=1e-12, atol=1e-12)
    # a sequence of one token: the output is that token's value row, lse its logit
    w, cache, table, lens, q, qi = small_case([1], q_len=1, seed=20)
    s, sel, out, lse = M.msa_decode(q, qi, cache, table, lens, heads_per_group=4)
    for h in range(16):
        g = h // 4
        v = F.nvfp4_dequantize(cache[2][table[0, 0], g, 0], cache[3][table[0, 0], g, 0])
        k = F.nvfp4_dequantize(cache[0][table[0, 0], g, 0], cache[1][table[0, 0], g, 0])
        assert np.allclose(out[0, 0, h], v, rtol=1e-12, atol=1e-12)
        assert lse[0, 0, h] == pytest.approx(float(k @ F.e4m3_decode(q[0, 0, h])) / math.sqrt(128), rel=1e-12)


def test_split_merge_identity():
    rng = np.random.default_rng(5)
    x = rng.standard_normal(300) * 4
    v = rng.standard_normal((300, 8))
    full_p = np.exp(x - x.max())
    want = full_p @ v / full_p.sum()
    want_lse = x.max() + math.log(full_p.sum())
    for _ in range(20):
        cuts = sorted(rng.choice(np.arange(1, 300), size=int(rng.integers(1, 6)), replace=False))
        parts = []
        for a, b in zip([0] + list(cuts), list(cuts) + [300]):
            m = x[a:b].max()
            p = np.exp(x[a:b] - m)
            parts.append((m, p.sum(), p @ v[a:b]))
        got, lse = M.merge_partials(parts)
        assert np.allclose(got, want, rtol=1e-12) and lse == pytest.approx(want_lse, rel=1e-13)


def test_at_most_2048_keys_and_recent_block_present():
    w, cache, table, lens, q, qi = small_case([9000, 5000], q_len=4, seed=23)
    s, sel, out, lse = M.msa_decode(q, qi, cache, table, lens, heads_per_group=4)
    for b in range(2):
        L = int(lens[b])
        for t in range(4):
            pos = L - 4 + t
            for g in range(4):
                chosen = sel[b, t, g][sel[b, t, g] >= 0]
                assert len(chosen) == 16 and pos // 128 in chosen
                visible = sum(min(128, pos + 1 - n * 128) for n in chosen)
                assert visible <= FACTS["max_keys_per_query"]["value"]


# ------------------------------------------------------------------ DCP merge
def test_dcp_merge_is_exact():
    rng = np.random.default_rng(31)
    for _ in range(200):
        nb = int(rng.integers(2, 300))
        row = np.round(rng.standard_normal(nb) * 3, 1)    # rounding creates ties
        pos = int(rng.integers(0, nb * 128))
        shards = int(rng.integers(1, 6))
        cuts = np.linspace(0, nb, shards + 1).astype(int)
        lists = [M.dcp_local_candidates(row, pos, int(a), int(b)) for a, b in zip(cuts[:-1], cuts[1:])]
        assert np.array_equal(M.dcp_merge(lists, pos), M.select_row(row, pos))


# ------------------------------------------------------------------ configuration variants
# (block rules: "MiniMax M3 x vLLM：百万 token 多模态推理的 Day-0 部署", §MSA 机制细节 for init /
# local blocks, §Prefill 执行 step 2 for the max or log-sum-exp block reduction)
def _variant_bruteforce(scores_row, r, k, init_blocks, local_blocks):
    """Forced blocks (the first init_blocks and the last local_blocks up to r, each once)
    plus, among every subset of the other blocks up to r of the remaining size, the one with
    the largest score sum, ties to the lexicographically smallest."""
    forced = set(range(min(init_blocks, r + 1))) | set(range(max(0, r - local_blocks + 1), r + 1))
    others = [n for n in range(r + 1) if n not in forced]
    m = min(max(0, k - len(forced)), len(others))
    best = None
    for sub in itertools.combinations(others, m):
        tot = sum(scores_row[n] for n in sub)
        if best is None or tot > best[0] or (tot == best[0] and sub < best[1]):
            best = (tot, sub)
    return sorted(forced | set(best[1]))


def test_select_variants_equal_subset_bruteforce():
    rng = np.random.default_rng(17)
    for trial in range(400):
        k = int(rng.integers(1, 7))
        init = int(rng.integers(0, k + 1))
        local = int(rng.integers(0, k - init + 1))
        r = int(rng.integers(0, 11))
        row = rng.integers(-3, 4, size=12).astype(np.float64)   # many exact ties
        got = M.select_row(row, r * 128 + int(rng.integers(0, 128)), top_k=k, init_blocks=init, local_blocks=local)
        want = _variant_bruteforce(row, r, k, init, local)
        assert [int(x) for x in got if x >= 0] == want, (k, init, local, r)
        assert len(want) == min(k, r + 1)
        assert (got[len(want):] == -1).all()


def test_select_recipe_is_the_default_variant():
    rng = np.random.default_rng(23)
    for _ in range(100):
        row = rng.standard_normal(40)
        pos = int(rng.integers(0, 40 * 128))
        assert np.array_equal(M.select_row(row, pos), M.select_row(row, pos, 16, 0, 1))


def test_lse_pooling_equals_library_logsumexp_of_exact_scores():
    from scipy.special import logsumexp
    w, cache, table, lens, q, qi = small_case([300, 130], q_len=2, hg=1, seed=29)
    s = M.block_scores(qi, cache[4], cache[5], table, lens, pooling="lse")
    _, _, _, _, idx_data, idx_scale = cache
    for b in range(2):
        L = int(lens[b])
        keys = np.concatenate([F.nvfp4_dequantize(idx_data[table[b, n]], idx_scale[table[b, n]])
                               for n in range(-(-L // 128))])[:L]
        for t in range(2):
            pos = L - 2 + t
            for g in range(4):
                qv = F.e4m3_decode(qi[b, t, g])
                for n in range(-(-L // 128)):
                    js = [j for j in range(n * 128, min((n + 1) * 128, L)) if j <= pos]
                    if not js:
                        assert s[b, t, g, n] == -np.inf
                        continue
                    want = logsumexp([float(qv @ keys[j]) for j in js])
                    assert abs(s[b, t, g, n] - want) <= 1e-9 * max(1.0, abs(want))


def test_lse_pooling_closed_forms():
    w, cache, table, lens, q, qi = small_case([300], q_len=1, seed=31)
    idx_data, idx_scale = cache[4], cache[5]
    for n in range(3):                                # every key of each block = its key 5
        page = table[0, n]
        idx_data[page] = idx_data[page, 5]
        idx_scale[page] = idx_scale[page, 5]
    s_max = M.block_scores(qi, idx_data, idx_scale, table, lens)
    s_lse = M.block_scores(qi, idx_data, idx_scale, table, lens, pooling="lse")
    pos = 299                                         # blocks 0, 1 full; block 2 holds 44 keys
    for g in range(4):
        for n, count in [(0, 128), (1, 128), (2, pos - 256 + 1)]:
            assert s_lse[0, 0, g, n] == pytest.approx(s_max[0, 0, g, n] + math.log(count), rel=1e-12, abs=1e-12)
    # in general: max <= lse <= max + ln(visible keys)
    w, cache, table, lens, q, qi = small_case([700, 260], q_len=3, seed=37)
    a = M.block_scores(qi, cache[4], cache[5], table, lens)
    l = M.block_scores(qi, cache[4], cache[5], table, lens, pooling="lse")
    fin = np.isfinite(a)
    assert np.array_equal(fin, np.isfinite(l))
    assert (l[fin] >= a[fin] - 1e-12).all() and (l[fin] <= a[fin] + math.log(128) + 1e-12).all()
