"""The NVFP4 attention kernel runs PV as an f16 MMA on decoded operands instead
of a block-scaled FP4 MMA.  That gives the same products only if every decoded
operand is exact in f16: an E2M1 code times its E4M3 scale (the V residual
before the fp32 per-(b,h) scale, and P).  With at most 2 + 4 significant bits
and magnitudes in [2^-10, 2688], every such product must be an f16 value; this
test checks all 8 x 127 of them, and the P side's range under the lazy
reference max (p <= 2^8, so its scale is at most E4M3(2^8 / 6)).
"""
import numpy as np
import torch

E2M1 = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]          # OCP FP4 E2M1 magnitudes


def _e4m3_values():
    codes = torch.arange(0, 127, dtype=torch.uint8)        # non-negative, finite
    return codes.view(torch.float8_e4m3fn).double().numpy()


def test_every_code_times_scale_is_an_f16_value():
    sf = _e4m3_values()
    assert sf.size == 127 and sf[1] == 2.0 ** -9 and sf[-1] == 448.0
    prod = np.array(E2M1)[:, None] * sf[None, :]
    as_f16 = prod.astype(np.float16).astype(np.float64)
    assert np.array_equal(as_f16, prod)
    nz = prod[prod > 0]
    assert nz.min() == 2.0 ** -10 and nz.max() == 2688.0
    # all are normal f16 numbers (>= 2^-14) or zero
    assert np.all((prod == 0) | (prod >= 2.0 ** -14))


def test_p_scale_range_under_the_lazy_max():
    """p = 2^(s - m) <= 2^8 with the lazy reference max, so a group's scale is
    at most E4M3(2^8 / 6) and a decoded P at most 6 times that: well inside f16."""
    amax = np.float32(256.0)
    q = np.float32(amax / np.float32(6.0))
    sf = torch.tensor([float(q)]).to(torch.float8_e4m3fn).double().item()
    assert sf <= 44.0 and 6.0 * sf < 65504.0
