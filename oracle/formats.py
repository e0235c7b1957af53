"""Exact number formats of the MSA cache: FP4 E2M1 values, FP8 E4M3 scales and queries.

TEST INFRASTRUCTURE ONLY.  This package is the plain CPU oracle of the MSA decode path.
Only tests/, __graft_entry__.smoke() and bench.py's cpu_baseline / reference leg may import
it; the product (block_sparse_attention_indexer_gb300) never does, and shares no code
with it.

The cache is NVFP4: 4-bit E2M1 values with one E4M3 scale per 16 consecutive elements
("vLLM liefert Day-0-Unterstützung für MiniMax-M3.1-Flash", §Was ist neu in der
MiniMax-M3.1-Architektur: 34,560 instead of 61,440 bytes per token, i.e. 4.5 bits per
element = 4 value bits + 8 scale bits / 16 elements).  Queries stay FP8 E4M3
(same page, §NVIDIA-Blackwell-optimierte MSA-Kernel).  The AMD section of that page
(§NVFP4-MSA-Kernel) counts 256 possible E4M3 scales and 8 E2M1 magnitudes.

Bit fields (OCP 8-bit floating point / microscaling formats):
  E2M1: s | e1 e0 | m, exponent bias 1, e = 0 is subnormal (0.5 * m), no inf / NaN.
  E4M3 (FN): s | e3..e0 | m2..m0, bias 7, e = 0 subnormal (m/8 * 2^-6), max 448,
             s.1111.111 is NaN, no inf.

Parity pins for everything here live in tests/test_oracle_formats.py.
"""
from __future__ import annotations

import numpy as np


def e2m1_value(code: int) -> float:
    """Real value of one 4-bit E2M1 code (0..15), from its bit fields."""
    s = (code >> 3) & 1
    e = (code >> 1) & 3
    m = code & 1
    mag = 0.5 * m if e == 0 else 2.0 ** (e - 1) * (1.0 + 0.5 * m)
    return -mag if s else mag


def e4m3_value(code: int) -> float:
    """Real value of one FP8 E4M3 (FN) code (0..255), from its bit fields."""
    s = (code >> 7) & 1
    e = (code >> 3) & 15
    m = code & 7
    if e == 15 and m == 7:
        return float("nan")
    mag = (m / 8.0) * 2.0 ** -6 if e == 0 else (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return -mag if s else mag


E2M1_TABLE = np.array([e2m1_value(c) for c in range(16)], dtype=np.float64)
E4M3_TABLE = np.array([e4m3_value(c) for c in range(256)], dtype=np.float64)

# non-negative finite codes are monotone in value: E2M1 codes 0..7, E4M3 codes 0..126
_E2M1_POS = E2M1_TABLE[:8]
_E4M3_POS = E4M3_TABLE[:127]


def _round_nearest_even(a: np.ndarray, grid: np.ndarray) -> np.ndarray:
    """Index of the grid point nearest to each a >= 0 (grid ascending, index = code).

    Ties go to the even code (the one whose lowest mantissa bit is 0); values above the
    last grid point saturate to it (the 'satfinite' rule).
    """
    hi = np.searchsorted(grid, a, side="left")          # first grid point >= a
    hi = np.minimum(hi, len(grid) - 1)
    lo = np.maximum(hi - 1, 0)
    d_lo = a - grid[lo]
    d_hi = grid[hi] - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo)
    code = np.where(a >= grid[-1], len(grid) - 1, code)
    return code.astype(np.uint8)


def e4m3_encode(x) -> np.ndarray:
    """Round each value to FP8 E4M3: nearest, ties to even, saturating at +-448.

    The sign bit is copied from x (so tiny negatives become 0x80).
    """
    x = np.asarray(x, dtype=np.float64)
    code = _round_nearest_even(np.abs(x), _E4M3_POS)
    return (code | (np.signbit(x).astype(np.uint8) << 7)).astype(np.uint8)


def e2m1_encode(x) -> np.ndarray:
    """Round each value to FP4 E2M1: nearest, ties to even, saturating at +-6; sign copied."""
    x = np.asarray(x, dtype=np.float64)
    code = _round_nearest_even(np.abs(x), _E2M1_POS)
    return (code | (np.signbit(x).astype(np.uint8) << 3)).astype(np.uint8)


def e4m3_decode(codes) -> np.ndarray:
    return E4M3_TABLE[np.asarray(codes, dtype=np.uint8)]


def nvfp4_quantize(x):
    """Quantise float32 rows to NVFP4, 16 consecutive elements per scale.

    x: float32 [..., n*16].  For every group of 16:
      scale code = E4M3(amax / 6), amax and the division in float32 (correctly rounded);
      element code = E2M1(x / scale), division in float32 (correctly rounded);
      a scale that rounds to zero gives all-zero element codes.
    Returns (data uint8 [..., n*8], scales uint8 [..., n]); byte j of a row holds
    element 2j in its low nibble and element 2j+1 in its high nibble.
    """
    x = np.asarray(x, dtype=np.float32)
    lead = x.shape[:-1]
    width = x.shape[-1]
    assert width % 16 == 0
    g = x.reshape(*lead, width // 16, 16)
    amax = np.max(np.abs(g), axis=-1)
    scale_code = e4m3_encode(amax / np.float32(6.0))
    scale = E4M3_TABLE[scale_code].astype(np.float32)
    nonzero = scale > 0
    safe = np.where(nonzero, scale, np.float32(1.0)).astype(np.float32)
    ratio = g / safe[..., None]                      # float32 / float32 -> float32, correctly rounded
    codes = e2m1_encode(ratio)
    codes = np.where(nonzero[..., None], codes, np.uint8(0)).astype(np.uint8)
    codes = codes.reshape(*lead, width)
    data = (codes[..., 0::2] | (codes[..., 1::2] << 4)).astype(np.uint8)
    return data, scale_code


def nvfp4_dequantize(data, scales) -> np.ndarray:
    """Exact real values (float64) of NVFP4 rows: data uint8 [..., n*8], scales uint8 [..., n]."""
    data = np.asarray(data, dtype=np.uint8)
    scales = np.asarray(scales, dtype=np.uint8)
    lo = E2M1_TABLE[data & 0x0F]
    hi = E2M1_TABLE[data >> 4]
    vals = np.empty(data.shape[:-1] + (data.shape[-1] * 2,), dtype=np.float64)
    vals[..., 0::2] = lo
    vals[..., 1::2] = hi
    n = scales.shape[-1]
    vals = vals.reshape(*data.shape[:-1], n, 16) * E4M3_TABLE[scales][..., None]
    return vals.reshape(*data.shape[:-1], n * 16)


def fp8_dequant_table() -> np.ndarray:
    """The 256 x 8 table of every E4M3 scale times every E2M1 magnitude, each product
    rounded once to E4M3 (the pre-rounded FP8 dequantisation table of the AMD section,
    §NVFP4-MSA-Kernel: 256 scales x 8 magnitudes = 2,048 entries = 2 KB)."""
    prod = E4M3_TABLE[:, None] * _E2M1_POS[None, :]
    prod = np.where(np.isnan(prod), 0.0, prod)
    return e4m3_encode(prod)
