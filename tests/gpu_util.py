"""Helpers shared by the -m gpu parity tests: building both sides' inputs from the same
seeded workload (each side quantises with its own code), tolerances, and comparisons."""
from __future__ import annotations

import math

import numpy as np
import pytest

from oracle import cache as OC
from oracle import formats as OF
from oracle import msa as OM
from workloads import synthetic as syn

# parity bar for the attention output (max-abs / mean-abs vs the float64 oracle) and the
# relative score gap below which two selections may legitimately differ
OUT_MAX_ABS = 2e-2
OUT_MEAN_ABS = 2e-3
NEAR_TIE_REL = 1e-3


def need_gpu():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def device_workload(w, lens=None, **kw):
    from workloads import device
    return device.upload(w, lens, **kw)


def oracle_inputs(w, lens=None, sequences=None):
    cache, table, lens, P = OC.build_cache(w, lens, sequences, threads=8)
    q, qi = OC.encode_queries(w, sequences)
    return cache, table, lens, q, qi


def score_bound(qi_codes, idx_data, idx_scale, table, lens, max_blocks):
    """Per (b, t, g, n): the largest sum_d |q_d k_d| over the block's keys -- the scale of the
    float32 accumulation error of one score (bound used: 2^-16 times it)."""
    qa = np.abs(OF.E4M3_TABLE[qi_codes])
    B, T, G, _ = qi_codes.shape
    out = np.zeros((B, T, G, max_blocks))
    for b in range(B):
        L = int(lens[b])
        if L <= 0:
            continue
        keys = np.abs(OM.index_keys(idx_data, idx_scale, table[b], L))
        nb = -(-L // 128)
        s = keys @ qa[b].reshape(-1, qa.shape[-1]).T            # [L, T*G]
        pad = np.zeros((nb * 128, T * G))
        pad[:L] = s
        out[b, :, :, :nb] = pad.reshape(nb, 128, T, G).max(axis=1).transpose(1, 2, 0)
    return out


def assert_scores_close(gpu, ref, bound):
    gpu = np.asarray(gpu, dtype=np.float64)
    inf_g, inf_r = np.isneginf(gpu), np.isneginf(ref)
    assert np.array_equal(inf_g, inf_r), f"-inf pattern differs at {np.argwhere(inf_g != inf_r)[:5]}"
    fin = ~inf_r
    err = np.abs(gpu[fin] - ref[fin])
    tol = bound[fin] * 2.0 ** -16 + 1e-30
    bad = err > tol
    assert not bad.any(), f"{bad.sum()} scores outside the float32 accumulation bound; worst {err.max()}"
    return float(err.max()) if err.size else 0.0


def selection_diffs(sel_gpu, sel_ref, scores_ref, lens, q_len):
    """Rows whose selections differ; each difference must be a near tie in the oracle's
    scores (every block of the symmetric difference within NEAR_TIE_REL of the weakest
    selected candidate).  Returns the set of differing rows (b, t, g)."""
    diff_rows = set()
    B, T, G, K = sel_ref.shape
    for b in range(B):
        L = int(lens[b])
        if L <= 0:
            continue
        for t in range(T):
            r = (L - T + t) // 128
            for g in range(G):
                a, e = sel_gpu[b, t, g], sel_ref[b, t, g]
                if np.array_equal(a, e):
                    continue
                sa, se = set(int(x) for x in a if x >= 0), set(int(x) for x in e if x >= 0)
                assert len(sa) == len(se) and r in sa, (b, t, g, a, e)
                cands = sorted((n for n in se if n != r), key=lambda n: -scores_ref[b, t, g, n])
                thr = scores_ref[b, t, g, cands[-1]]
                for n in sa ^ se:
                    gap = abs(scores_ref[b, t, g, n] - thr)
                    assert gap <= NEAR_TIE_REL * abs(thr), (b, t, g, n, scores_ref[b, t, g, n], thr)
                diff_rows.add((b, t, g))
    return diff_rows


def assert_out_close(out_gpu, out_ref, mask=None):
    o = np.asarray(out_gpu, dtype=np.float64)
    if mask is not None:
        o, out_ref = o[mask], out_ref[mask]
    err = np.abs(o - out_ref)
    assert err.max() <= OUT_MAX_ABS, f"max-abs {err.max()}"
    assert err.mean() <= OUT_MEAN_ABS, f"mean-abs {err.mean()}"
    rms = math.sqrt(float((out_ref ** 2).mean())) if out_ref.size else 1.0
    return float(err.max()), float(err.mean()), float(err.max()) / max(rms, 1e-30)


def to_np(t):
    return t.detach().cpu().numpy()


def bf16_to_np(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


__all__ = ["need_gpu", "device_workload", "oracle_inputs", "score_bound", "assert_scores_close",
           "selection_diffs", "assert_out_close", "to_np", "bf16_to_np", "syn", "OC", "OF", "OM"]
