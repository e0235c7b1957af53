"""The cache-write kernel divides by a float32 divisor d through its correctly rounded
reciprocal y = RN(1/d): q = RN(x y), r = x - d q (exact, one fma), result RN(q + r y)
(Markstein's correction step).  The divisors are E4M3 scales and 6, whose significands are
the integers 1..15 times a power of two.  This checks, on the host, that the three steps give
the correctly rounded quotient for sampled float32 significands of x and every such divisor
significand: a restatement of the method the kernel relies on, not of the oracle."""
import numpy as np


def _rn32_of_exact_sum(hi, lo):
    # RN to float32 of the exact value hi + lo (hi float64, |lo| <= half an ulp of hi)
    s = hi.astype(np.float32)
    up = np.nextafter(s, np.float32(np.inf))
    dn = np.nextafter(s, np.float32(-np.inf))
    base = s.astype(np.float64)
    d_up = (hi - (base + up.astype(np.float64)) / 2) + lo
    d_dn = (hi - (base + dn.astype(np.float64)) / 2) + lo
    odd = (s.view(np.uint32) & 1) == 1
    out = np.where((d_up > 0) | ((d_up == 0) & odd), up, s)
    return np.where((d_dn < 0) | ((d_dn == 0) & odd), dn, out)


def _reciprocal_division(a, b):
    y = np.float32(1.0 / b)                         # RN(1/b): 1/b is never a float32 midpoint
    q = (a * np.float64(y)).astype(np.float32)      # the product is exact in float64
    r64 = a - np.float64(b) * q.astype(np.float64)  # exact
    r = r64.astype(np.float32)
    assert np.array_equal(r.astype(np.float64), r64)  # the remainder is a float32
    ry = r.astype(np.float64) * np.float64(y)       # exact
    qd = q.astype(np.float64)
    hi = qd + ry
    lo = (qd - hi) + ry                             # exact error of the sum (|qd| >= |ry|)
    return q, _rn32_of_exact_sum(hi, lo)


def test_reciprocal_division_is_correctly_rounded():
    rng = np.random.default_rng(5)
    bits = rng.integers(0, 1 << 23, size=1 << 18, dtype=np.uint32)
    bits = np.concatenate([bits, np.arange(4096, dtype=np.uint32), (1 << 23) - 1 - np.arange(4096, dtype=np.uint32)])
    a = (bits | np.uint32(127 << 23)).view(np.float32).astype(np.float64)  # significands in [1, 2)
    for b in range(1, 16):
        q, got = _reciprocal_division(a, b)
        ref = (a / b).astype(np.float32)            # a / b is a float32 midpoint only when exact
        assert np.array_equal(got, ref), b
        if b not in (1, 2, 4, 8):                   # the correction step is what makes it exact
            assert not np.array_equal(q, ref), b
