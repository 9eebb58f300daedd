"""The NVFP4 attention kernel runs PV as the block-scaled FP4 MMA: per group of
16 keys, the products of the E2M1 codes of P and V are summed and the sum is
scaled by P's and V's E4M3 scale factors of that group.  The result equals
the oracle's fp64 arithmetic on the decoded operands up to the fp32
accumulation across groups only if every group's contribution is exact in
fp32: a sum of 16 code products (multiples of 1/4, at most 16 x 36 = 576) times
two E4M3 scales (at most 8 significant bits together).  This checks all of
them, and that the same holds for the row-sum MMA (codes of P times 1.0, V's
scale 1.0), with P's scales limited by the lazy reference max (p <= 2^8, so
sf <= E4M3(2^8 / 6)).
"""
import numpy as np
import torch

E2M1 = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]          # OCP FP4 E2M1 magnitudes


def _e4m3_values():
    codes = torch.arange(0, 127, dtype=torch.uint8)        # non-negative, finite
    return codes.view(torch.float8_e4m3fn).double().numpy()


def _group_sums():
    """Every value a sum of 16 signed E2M1 x E2M1 products can take."""
    prods = np.unique(np.outer(E2M1, E2M1))
    assert np.all(prods * 4 == np.round(prods * 4)) and prods.max() == 36.0
    return np.arange(-16 * 36 * 4, 16 * 36 * 4 + 1) / 4.0   # every multiple of 1/4 up to 576 (a superset)


def test_every_group_contribution_is_exact_in_fp32():
    sf = _e4m3_values()
    assert sf.size == 127 and sf[1] == 2.0 ** -9 and sf[-1] == 448.0
    scale = np.unique(np.outer(sf, sf))                      # sf_p * sf_v over all pairs
    sums = _group_sums()
    for chunk in np.array_split(scale, 16):
        exact = sums[:, None] * chunk[None, :]               # fp64 holds these exactly (<= 20 bits)
        assert np.array_equal(exact.astype(np.float32).astype(np.float64), exact)


def test_the_row_sum_mma_is_exact_per_group():
    sf = _e4m3_values()
    e4m3_256_over_6 = torch.tensor(256.0 / 6.0).to(torch.float8_e4m3fn).double().item()
    p_scales = sf[sf <= e4m3_256_over_6]
    sums = np.arange(0, 16 * 6 * 2 + 1) / 2.0                # 16 codes of P times E2M1 1.0
    exact = sums[:, None] * p_scales[None, :]
    assert np.array_equal(exact.astype(np.float32).astype(np.float64), exact)
