"""NVFP4 insert and FP8 encode kernels: bit-exact against the oracle's quantiser."""
import numpy as np
import pytest

from gpu_util import OF, need_gpu, to_np

pytestmark = pytest.mark.gpu


def _edge_rows(rng, n, dim):
    x = rng.standard_normal((n, dim)).astype(np.float32) * rng.uniform(1e-3, 30, (n, 1)).astype(np.float32)
    x[0] = 0.0
    x[1] = -0.0
    x[2, :16] = 1e-30                     # scale rounds to zero
    x[3] = 1e6 * np.sign(x[3])            # scale saturates at 448, values at +-6
    x[4] = -1e-4                          # tiny negatives
    # exact E2M1 midpoints times a power-of-two scale: amax 6 -> scale 1
    mids = np.float32([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0])
    x[5, :16] = np.concatenate([mids, -mids])
    x[6, :16] = np.concatenate([mids, -mids]) * np.float32(2.0 ** -7)
    x[7, :] = np.float32(448 * 6 * 1.01)
    # infinite elements: the scale saturates at 448, the infinity at +-6, the rest keep their signs
    x[8, :16] = np.float32([np.inf, -3.0, 1.0, -0.0, 2.0e3, -2.0e4, 5.0, 0.5] * 2)
    x[9, 16:32] = np.float32([-np.inf, 3.0, -1.0, 0.0, -2.0e3, 2.0e4, -5.0, 7.0e5] * 2)
    return x


def test_nvfp4_insert_bit_exact():
    need_gpu()
    import torch
    import block_sparse_attention_indexer_gb300 as msa
    rng = np.random.default_rng(42)
    P, G, D, BL = 7, 4, 128, 128
    n = 3 * BL + 17
    x = _edge_rows(rng, n * G, D).reshape(n, G, D)
    slots = rng.permutation(P * BL)[:n].astype(np.int64)
    data = torch.zeros(P, G, BL, D // 2, dtype=torch.uint8, device="cuda")
    scale = torch.zeros(P, G, BL, D // 16, dtype=torch.uint8, device="cuda")
    msa.msa_nvfp4_insert(torch.from_numpy(x).cuda(), torch.from_numpy(slots).cuda(), data, scale, BL)
    torch.cuda.synchronize()
    d_ref, s_ref = OF.nvfp4_quantize(x)                     # [n, G, 64], [n, G, 8]
    d_gpu, s_gpu = to_np(data), to_np(scale)
    for i, slot in enumerate(slots):
        p, o = divmod(int(slot), BL)
        assert np.array_equal(d_gpu[p, :, o], d_ref[i]), f"token {i}"
        assert np.array_equal(s_gpu[p, :, o], s_ref[i]), f"token {i}"
    # untouched slots stay zero; out-of-range slots are skipped
    used = np.zeros(P * BL, bool)
    used[slots] = True
    flat = d_gpu.transpose(0, 2, 1, 3).reshape(P * BL, -1)
    assert (flat[~used] == 0).all()
    bad = torch.tensor([-1, P * BL], dtype=torch.int64, device="cuda")
    msa.msa_nvfp4_insert(torch.ones(2, G, D, device="cuda"), bad, data, scale, BL)
    torch.cuda.synchronize()
    assert np.array_equal(to_np(data), d_gpu)


def test_nvfp4_insert_many_passes_odd_shape():
    """A write larger than one pass of the grid, with groups per token (3 rows x 5 groups)
    that do not divide the grid's thread count: each thread's (token, group) advances across
    passes with a carry; every token's codes and scales are compared with the oracle."""
    need_gpu()
    import torch
    import block_sparse_attention_indexer_gb300 as msa
    rng = np.random.default_rng(11)
    R, D, BL = 3, 80, 64
    n = 40_000
    P = (n + BL - 1) // BL + 5
    x = (rng.standard_normal((n, R, D)) * rng.uniform(0.01, 50, (n, 1, 1))).astype(np.float32)
    x[7] = -0.0
    x[n - 1, 2, 64:] = np.inf
    slots = rng.permutation(P * BL)[:n].astype(np.int64)
    slots[123] = -5                                  # skipped
    data = torch.zeros(P, R, BL, D // 2, dtype=torch.uint8, device="cuda")
    scale = torch.zeros(P, R, BL, D // 16, dtype=torch.uint8, device="cuda")
    msa.msa_nvfp4_insert(torch.from_numpy(x).cuda(), torch.from_numpy(slots).cuda(), data, scale, BL)
    torch.cuda.synchronize()
    d_ref, s_ref = OF.nvfp4_quantize(x)              # [n, R, 40], [n, R, 5]
    d_gpu, s_gpu = to_np(data), to_np(scale)
    ok = slots >= 0
    p, o = np.divmod(slots[ok], BL)
    assert np.array_equal(d_gpu[p, :, o], d_ref[ok])
    assert np.array_equal(s_gpu[p, :, o], s_ref[ok])
    used = np.zeros(P * BL, bool)
    used[slots[ok]] = True
    flat = s_gpu.transpose(0, 2, 1, 3).reshape(P * BL, -1)
    assert (flat[~used] == 0).all()


def test_nvfp4_insert_index_layout():
    need_gpu()
    import torch
    import block_sparse_attention_indexer_gb300 as msa
    rng = np.random.default_rng(3)
    P, BL, Di = 3, 128, 128
    x = (rng.standard_normal((P * BL, Di)) * 3).astype(np.float32)
    idx_data = torch.zeros(P, BL, Di // 2, dtype=torch.uint8, device="cuda")
    idx_scale = torch.zeros(P, BL, Di // 16, dtype=torch.uint8, device="cuda")
    slots = torch.arange(P * BL, dtype=torch.int64, device="cuda")
    msa.msa_nvfp4_insert(torch.from_numpy(x).cuda().view(P * BL, 1, Di), slots, idx_data.view(P, 1, BL, Di // 2),
                         idx_scale.view(P, 1, BL, Di // 16), BL)
    torch.cuda.synchronize()
    d_ref, s_ref = OF.nvfp4_quantize(x)
    assert np.array_equal(to_np(idx_data).reshape(P * BL, -1), d_ref)
    assert np.array_equal(to_np(idx_scale).reshape(P * BL, -1), s_ref)


def test_fp8_quantize_bit_exact():
    need_gpu()
    import torch
    import block_sparse_attention_indexer_gb300 as msa
    rng = np.random.default_rng(9)
    pos = OF.E4M3_TABLE[:127]
    mids = ((pos[:-1] + pos[1:]) / 2).astype(np.float32)
    x = np.concatenate([rng.standard_normal(100000).astype(np.float32) * 4, mids, -mids,
                        np.float32([0.0, -0.0, 1e-12, -1e-12, 448, 449, 500, 1e9, -1e9])])
    out = torch.empty(x.size, dtype=torch.uint8, device="cuda")
    msa.msa_fp8_quantize(torch.from_numpy(x).cuda(), out)
    torch.cuda.synchronize()
    assert np.array_equal(to_np(out), OF.e4m3_encode(x))
