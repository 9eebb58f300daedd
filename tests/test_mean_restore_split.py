"""The E4M3 attention kernel adds the block means back with one bf16 MMA per 16
key blocks: each row sum rs and each scaled mean mu = mean / s_v is split into
hi = bf16(rs) and lo = bf16(rs - hi), and the MMA sums the four products
hi.hi + lo.hi + hi.lo + lo.lo in fp32.  Each product of two bf16 values has at
most 16 significant bits, so it is exact in fp32, and the split keeps about 16
bits of each factor.  This test checks those two facts on the CPU, with torch's
bf16 rounding, over factors spanning the range the kernel sees.
"""
import numpy as np
import torch


def _bf16(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16).float().numpy()


def _split(x):
    x = np.asarray(x, np.float32)
    hi = _bf16(x)
    lo = _bf16((x - hi).astype(np.float32))      # x - hi is exact in fp32
    return hi, lo


def test_split_keeps_sixteen_bits():
    rng = np.random.default_rng(0)
    x = (rng.uniform(0.5, 1.0, 200000) * 2.0 ** rng.integers(-40, 40, 200000)).astype(np.float32)
    x *= np.where(rng.random(200000) < 0.5, -1, 1).astype(np.float32)
    hi, lo = _split(x)
    rel = np.abs(x.astype(np.float64) - hi.astype(np.float64) - lo.astype(np.float64)) / np.abs(x.astype(np.float64))
    assert rel.max() <= 2.0 ** -16, rel.max()
    # values with at most 16 significant bits are split exactly
    y = (rng.integers(1 << 15, 1 << 16, 10000) * 2.0 ** rng.integers(-30, 10, 10000)).astype(np.float32)
    hy, ly = _split(y)
    assert np.array_equal(hy.astype(np.float64) + ly.astype(np.float64), y.astype(np.float64))


def test_partial_products_are_exact_and_their_sum_is_the_product():
    rng = np.random.default_rng(1)
    rs = (rng.uniform(1.0, 128.0, 100000)).astype(np.float32)            # row sums of a block
    mu = (rng.standard_normal(100000) * 2.0 ** rng.integers(-8, 8, 100000)).astype(np.float32)
    rh, rl = _split(rs)
    mh, ml = _split(mu)
    terms = [a.astype(np.float64) * b.astype(np.float64) for a, b in ((rh, mh), (rl, mh), (rh, ml), (rl, ml))]
    for t in terms:
        assert np.array_equal(t.astype(np.float32).astype(np.float64), t)   # exact in fp32
    exact = rs.astype(np.float64) * mu.astype(np.float64)
    got = sum(terms)
    assert np.all(np.abs(got - exact) <= 2.0 ** -15 * np.abs(exact))
