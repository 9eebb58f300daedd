"""The NVFP4 attention kernel takes the E4M3 scale of every 16 probabilities
from amax / 6 without a division: q = RN(a r), then one correction step
q' = RN(q + RN(a - 6 q) r) with r = RN(1/6), each step one fp32 multiply or
fused multiply-add.  The kernel relies on q' being the correctly rounded
quotient RN(a / 6) for every a in [2^-120, 2^30] (the probabilities lie in
(0, 1], their scale in E4M3's range; below 2^-120 both values are far under
E4M3's smallest step and give the code 0).

This test checks that claim on the CPU with the fp32 arithmetic emulated
exactly in fp64: a product of two fp32 values is exact in fp64, so casting
it rounds once; a - 6q is exact in fp64 (the two are within a few units of
each other); the final sum is rounded through an exact two-sum so that a
double rounding at an fp32 midpoint cannot go unnoticed.  The correctly
rounded quotient is found by comparing |a - 6 c| over c and its fp32
neighbours (a / 6 is never an fp32 midpoint: 6 times a 25-bit odd
significand does not fit in 24 bits).

Every fp32 value of the binades tested is checked.  Above 2^-100 every
intermediate is a normal fp32 number, so the results scale exactly by powers
of two and one binade stands for all of them; a few are checked anyway.
Below 2^-100 the residual a - 6q can be subnormal, so every binade down to
2^-120 is checked.
"""
import numpy as np
import pytest

R = np.float32(1.0) / np.float32(6.0)


def _binade(e):
    """Every fp32 value in [2^e, 2^(e+1))."""
    base = (e + 127) << 23
    return (np.arange(base, base + (1 << 23), dtype=np.uint32)).view(np.float32)


def _round_sum_f32(x, y):
    """RN32(x + y) for fp64 inputs whose exact sum may need more than 53 bits:
    two-sum gives t = RN64(x + y) and the exact error; only when t is an fp32
    midpoint does the error decide the rounding."""
    t = x + y
    bp = t - x
    err = (x - (t - bp)) + (y - bp)
    f = t.astype(np.float32)
    ff = f.astype(np.float64)
    g = np.where(t > ff, np.nextafter(f, np.float32(np.inf)), np.nextafter(f, np.float32(-np.inf)))
    gf = g.astype(np.float64)
    mid = (t != ff) & (ff + gf == 2.0 * t)
    # at a midpoint numpy rounded to even; the exact sum lies on the side of err
    up = mid & (err > 0)
    down = mid & (err < 0)
    hi = np.maximum(ff, gf).astype(np.float32)
    lo = np.minimum(ff, gf).astype(np.float32)
    return np.where(up, hi, np.where(down, lo, f))


def kernel_quotient(a):
    """The kernel's steps: q0 = RN(a r); e = RN(fma(-q0, 6, a)); q1 = RN(fma(e, r, q0))."""
    a64 = a.astype(np.float64)
    q0 = (a64 * np.float64(R)).astype(np.float32)
    e = (a64 - 6.0 * q0.astype(np.float64)).astype(np.float32)
    return _round_sum_f32(e.astype(np.float64) * np.float64(R), q0.astype(np.float64))


def ieee_quotient(a):
    a64 = a.astype(np.float64)
    c = (a64 / 6.0).astype(np.float32)
    cands = [np.nextafter(c, np.float32(-np.inf)), c, np.nextafter(c, np.float32(np.inf))]
    dist = np.stack([np.abs(a64 - 6.0 * x.astype(np.float64)) for x in cands])
    best = np.argmin(dist, axis=0)
    return np.choose(best, cands)


def test_emulation_rounds_like_fp32():
    """The emulated steps against numpy's own fp32 arithmetic where that is
    exact: a product of fp32 values rounded once, and sums that fit in fp64."""
    rng = np.random.default_rng(0)
    a = rng.uniform(1e-3, 1e3, 100000).astype(np.float32)
    assert np.array_equal((a.astype(np.float64) * np.float64(R)).astype(np.float32), a * R)
    x = rng.uniform(-1, 1, 100000).astype(np.float32)
    y = rng.uniform(-1, 1, 100000).astype(np.float32)
    assert np.array_equal(_round_sum_f32(x.astype(np.float64), y.astype(np.float64)), x + y)
    # a midpoint the error must break: 1 + 2^-24 (+/- tiny) in fp32
    t = np.array([1.0 + 2.0 ** -24] * 3)
    d = np.array([2.0 ** -80, -2.0 ** -80, 0.0])
    got = _round_sum_f32(t, d)
    assert got.tolist() == [np.float32(1.0) + np.float32(2.0 ** -23), 1.0, 1.0]
    # the quotient reference where the quotient is exact, and 1/6 itself
    q = np.array([6.0, 3.0, 1.5, 12.0, 1.0], np.float32)
    assert ieee_quotient(q).tolist() == [1.0, 0.5, 0.25, 2.0, float(R)]


@pytest.mark.parametrize("e", list(range(-120, -99)) + [-60, -1, 0, 29])
def test_corrected_quotient_is_the_ieee_quotient(e):
    a = _binade(e)
    got = kernel_quotient(a)
    want = ieee_quotient(a)
    bad = np.flatnonzero(got != want)
    assert bad.size == 0, (e, a[bad[:4]], got[bad[:4]], want[bad[:4]])


def test_plain_product_is_not_enough():
    """Without the correction step RN(a r) misses the quotient on part of
    every binade: the correction is needed, and the check above can fail."""
    a = _binade(0)
    q0 = (a.astype(np.float64) * np.float64(R)).astype(np.float32)
    assert np.count_nonzero(q0 != ieee_quotient(a)) > 0
