"""Pins of the oracle's number formats against things other than itself: the published
code tables (tests/golden/ocp_formats.json), PyTorch's own float8_e4m3fn conversion, exact
rational arithmetic, and the byte counts the pages print."""
import json
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import formats as F

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _gold(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


def test_e2m1_table_matches_published_codes():
    want = _gold("ocp_formats.json")["e2m1"]["values_by_code"]
    assert len(F.E2M1_TABLE) == 16
    for code, v in enumerate(want):
        assert F.E2M1_TABLE[code] == v
        assert np.signbit(F.E2M1_TABLE[code]) == (code >= 8)


def test_e4m3_table_matches_published_points_and_torch():
    g = _gold("ocp_formats.json")["e4m3"]
    for hexcode, v in g["points"].items():
        c = int(hexcode, 16)
        assert F.E4M3_TABLE[c] == v and np.signbit(F.E4M3_TABLE[c]) == np.signbit(v)
    for hexcode in g["nan_codes"]:
        assert np.isnan(F.E4M3_TABLE[int(hexcode, 16)])
    # every one of the 256 codes against PyTorch's own E4M3FN decoder
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ours = F.E4M3_TABLE
    same = (ref == ours) | (np.isnan(ref) & np.isnan(ours))
    assert same.all()


def test_e4m3_encode_matches_torch_round_to_nearest_even():
    rng = np.random.default_rng(7)
    x = np.concatenate([
        rng.standard_normal(200000).astype(np.float32) * np.float32(3.0),
        (rng.standard_normal(50000) * 100).astype(np.float32),
        (rng.standard_normal(50000) * 1e-3).astype(np.float32),
        np.float32([0.0, -0.0, 448.0, -448.0, 1e-12, -1e-12, 2.0 ** -10, -(2.0 ** -10)]),
    ])
    # exact midpoints between neighbouring codes exercise ties-to-even
    pos = F.E4M3_TABLE[:127]
    mids = ((pos[:-1] + pos[1:]) / 2).astype(np.float32)
    x = np.concatenate([x, mids, -mids])
    x = x[np.abs(x) <= 448]
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(F.e4m3_encode(x), ref)


def test_e4m3_encode_saturates():
    assert F.e4m3_encode(np.float32([449.0, 1e9, -1e9, 464.0, 500.0])).tolist() == [0x7E, 0x7E, 0xFE, 0x7E, 0x7E]


def _nearest_even_fraction(v: Fraction, grid):
    """Brute force with exact rationals: nearest grid value, ties to the even index."""
    best = None
    for i, gv in enumerate(grid):
        d = abs(v - Fraction(gv))
        if best is None or d < best[0] or (d == best[0] and i % 2 == 0):
            best = (d, i)
    return best[1]


def test_e2m1_encode_brute_force_and_ties():
    grid = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    ties = {0.25: 0, 0.75: 1.0, 1.25: 1.0, 1.75: 2.0, 2.5: 2.0, 3.5: 4.0, 5.0: 4.0}
    for v, want in ties.items():
        assert F.E2M1_TABLE[F.e2m1_encode(np.float32(v))] == want
    rng = np.random.default_rng(3)
    xs = np.concatenate([rng.uniform(-7, 7, 3000), np.arange(-7, 7.001, 0.125)]).astype(np.float32)
    codes = F.e2m1_encode(xs)
    for x, c in zip(xs, codes):
        a = min(abs(Fraction(float(x))), Fraction(6))
        i = _nearest_even_fraction(a, grid)
        assert (c & 7) == i, (x, c)
        assert (c >> 3) == int(np.signbit(x))


def test_nvfp4_quantize_nibble_order_and_scale():
    # one group whose amax is 6 -> scale 1.0 exactly, so codes are the values themselves
    row = np.float32([0.5, 1, 1.5, 2, 3, 4, 6, -6, 0, -0.5, -1, -1.5, -2, -3, -4, 0.25])
    data, scale = F.nvfp4_quantize(row[None, :])
    assert F.E4M3_TABLE[scale[0, 0]] == 1.0
    assert data.shape == (1, 8) and scale.shape == (1, 1)
    # element 0 (0.5, code 1) in the low nibble of byte 0, element 1 (1.0, code 2) high
    assert data[0, 0] == (1 | (2 << 4))
    back = F.nvfp4_dequantize(data, scale)[0]
    want = row.astype(np.float64).copy()
    want[15] = 0.0  # 0.25 is a tie between 0 and 0.5 -> even code 0
    assert np.array_equal(back, want)


def test_nvfp4_zero_group_and_byte_ratio():
    x = np.zeros((3, 32), np.float32)
    x[1, 16:] = 1e-20          # amax/6 rounds to E4M3 zero -> all codes zero
    data, scale = F.nvfp4_quantize(x)
    assert (data == 0).all() and (scale == 0).all()
    # 4.5 bits per element: 64 data bytes + 8 scale bytes per 128 elements; the pages'
    # 34,560 vs 61,440 bytes per token is the same 9/16 ratio
    facts = _gold("page_facts.json")
    x = np.ones((1, 128), np.float32)
    d, s = F.nvfp4_quantize(x)
    assert d.nbytes + s.nbytes == 72
    assert Fraction(d.nbytes + s.nbytes, 128) == Fraction(facts["nvfp4_kv_bytes_per_token_model"]["value"],
                                                          facts["fp8_kv_bytes_per_token_model"]["value"])
    assert 100 * (1 - Fraction(72, 128)) == facts["nvfp4_saving_percent"]["value"]


def test_nvfp4_round_trip_error_bound_and_idempotence():
    rng = np.random.default_rng(11)
    x = (rng.standard_normal((4000, 128)) * rng.uniform(0.01, 50, (4000, 1))).astype(np.float32)
    data, scale = F.nvfp4_quantize(x)
    back = F.nvfp4_dequantize(data, scale)
    s = F.E4M3_TABLE[scale]                                    # [4000, 8]
    err = np.abs(back - x.astype(np.float64)).reshape(4000, 8, 16)
    amax = np.abs(x).reshape(4000, 8, 16).max(-1)
    # E2M1 grid gaps are 0.5 (below 2), 1 (2..4) and 2 (4..6): half a gap is at most 1
    # scale unit; clipping at 6*scale adds at most amax - 6*scale (scale rounded down)
    bound = s[..., None] * 1.0 + np.maximum(amax - 6 * s, 0)[..., None] + 1e-12
    assert (err <= bound).all()
    # dequantised values requantise to the same bytes when the scale is recomputed exactly
    d2, s2 = F.nvfp4_quantize(back.astype(np.float32))
    same_scale = (s2 == scale)
    assert same_scale.mean() > 0.5
    rows = same_scale.all(axis=1)
    assert np.array_equal(d2[rows], data[rows])


def test_dequant_products_are_exact_in_fp16_and_bf16():
    # every E2M1 magnitude times every finite E4M3 scale: at most 6 significant bits and
    # within range, so the product is exact in fp16 and in bf16 (the GPU path relies on it)
    mags = F.E2M1_TABLE[:8]
    sc = F.E4M3_TABLE[np.isfinite(F.E4M3_TABLE)]
    prod = (mags[:, None] * sc[None, :]).ravel()
    assert np.array_equal(prod.astype(np.float16).astype(np.float64), prod)
    as_bf16 = torch.from_numpy(prod).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(as_bf16, prod)


def test_fp8_dequant_table_is_2kb_single_rounding():
    facts = _gold("page_facts.json")
    tab = F.fp8_dequant_table()
    assert tab.shape == (facts["e4m3_scale_count"]["value"], facts["e2m1_magnitude_count"]["value"])
    assert tab.nbytes == facts["fp8_dequant_table_bytes"]["value"]
    # each entry is the E4M3 rounding of the exact product (checked against torch)
    prod = F.E4M3_TABLE[:, None] * F.E2M1_TABLE[None, :8]
    prod = np.where(np.isnan(prod), 0.0, np.clip(prod, -448.0, 448.0))
    ref = torch.from_numpy(prod.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    # float32 cast of a <= 6-significant-bit product is exact, so torch sees the exact value
    assert np.array_equal(tab, ref)


@pytest.mark.parametrize("shape", [(2, 3, 128), (5, 16)])
def test_quantize_shapes(shape):
    x = np.random.default_rng(0).standard_normal(shape).astype(np.float32)
    d, s = F.nvfp4_quantize(x)
    assert d.shape == shape[:-1] + (shape[-1] // 2,) and s.shape == shape[:-1] + (shape[-1] // 16,)
