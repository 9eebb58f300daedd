"""Pins for the oracle's attention (online softmax with ExpCast, block-mean
restore through the per-block row sums).

Paper page, "method": V-Smooth permutes K and V together (non-causal attention
is unchanged), demeans each 128-token block and restores the mean with one
outer product from the row sums online softmax already keeps; ExpCast writes P
bytes with one FMA.  Pins:
  * with P kept unquantised (the oracle's exact-P mode) the schedule reduces to
    softmax attention over the dequantised operands: torch fp64 is the pin;
  * exact attention matches torch's scaled_dot_product_attention and is
    invariant under a joint K/V permutation;
  * a two-block worked example, derived by hand below, fixes the running-max
    schedule (codes taken against the max so far, then rescaled);
  * a constant V comes back exactly; ExpCast output stays within the pages'
    total-variation bound of the exact-P output.
"""
import math

import numpy as np
import pytest
import torch

from bit_attention_video_smooth_gb300 import inputs as I
from cases import LN2_F32, nvfp4_two_block_case, two_block_case as _two_block_case



def _f32(u16):
    return (np.asarray(u16, np.uint16).astype(np.uint32) << 16).view(np.float32)


def _prepped(seed=0, N=512, BH=2, vmode=0):
    import oracle
    w = I.with_n(I.WORKLOADS["tiny"], N, H=BH)
    q, k, v = (I.to_u16(t).reshape(BH, N, 128) for t in I.make_qkv(w, seed=seed))
    perm = I.random_perm(BH, N, seed=seed + 7).numpy()
    return (q, k, v, perm), oracle.prep(q, k, v, perm, vmode=vmode)


def _dequant(orc, p, bh):
    """Dequantised operands of one (b,h): Qhat, Khat (permuted order), Vhat."""
    BH, N, d = p["q8"].shape
    nb = N // 128
    qh = orc.e4m3_decode(p["q8"][bh]) * np.repeat(p["sq"][bh], 128)[:, None]
    kh = orc.e4m3_decode(p["k8"][bh]) * np.repeat(p["sk"][bh], 128)[:, None]
    if p["v_sf"] is None:
        r = orc.e4m3_decode(p["v_res"][bh]).transpose(0, 2, 1) * p["v_scale"][bh][None, None, :]
    else:
        byts = p["v_res"][bh]                                   # [nb][d][64]
        nib = np.stack([byts & 15, byts >> 4], axis=-1).reshape(nb, d, 128)
        sf = orc.e4m3_decode(p["v_sf"][bh]).repeat(16, axis=-1)  # [nb][d][128]
        r = (orc.e2m1_decode(nib) * sf * p["v_scale"][bh]).transpose(0, 2, 1)
    vh = r + _f32(p["v_mean"][bh])[:, None, :].astype(np.float64)
    return qh, kh, vh.reshape(N, d)


@pytest.mark.parametrize("vmode", [0, 1])
def test_exact_p_mode_is_softmax_over_dequantised_operands(orc, vmode):
    _, p = _prepped(seed=1, vmode=vmode)
    O = orc.attention(p, orc.P_EXACT)
    for bh in range(2):
        qh, kh, vh = _dequant(orc, p, bh)
        S = torch.from_numpy(qh) @ torch.from_numpy(kh).T / math.sqrt(128)
        ref = torch.softmax(S, dim=-1) @ torch.from_numpy(vh)
        got = _f32(O[bh]).astype(np.float64)
        # bf16 output rounding is the only difference
        np.testing.assert_allclose(got, ref.numpy(), rtol=2 ** -8, atol=1e-6)


def test_exact_attention_matches_sdpa_and_is_permutation_invariant(orc):
    (q, k, v, perm), _ = _prepped(seed=2, N=384)
    O = orc.attention_exact(q, k, v)
    qt, kt, vt = (torch.from_numpy(_f32(a).astype(np.float64)) for a in (q, k, v))
    scale = float(np.float32(1.0 / math.sqrt(128)))        # the oracle's fp32 default scale
    ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=scale)
    np.testing.assert_allclose(O, ref.numpy(), rtol=1e-10, atol=1e-12)
    kp = np.stack([k[b][perm[b]] for b in range(2)])
    vp = np.stack([v[b][perm[b]] for b in range(2)])
    Op = orc.attention_exact(q, kp, vp)
    np.testing.assert_allclose(Op, O, rtol=1e-12, atol=1e-13)
    rows = np.array([0, 5, 383], np.int32)
    np.testing.assert_allclose(orc.attention_exact(q, k, v, rows=rows), O[:, rows], rtol=0, atol=0)


def test_running_max_schedule_worked_example(orc):
    p = _two_block_case(orc)
    # ExpCast, t = 8(s - m) + 55.65:
    #  block 0, m = 1:   key0 t=55.65 -> 56 (1.0); key1 t=50.15 -> 50 (0.625);
    #                    zeros t=47.65 -> 48 (0.5) x126           rowsum0 = 64.625
    #  block 1, m = 4.5: alpha = 2^(1-4.5); key128 -> 56 (1.0); key129 t=35.65 -> 36
    #                    (0.1875); zeros t=19.65 -> 20 (0.046875) x126  rowsum1 = 7.09375
    a = 2.0 ** -3.5
    l = 64.625 * a + 7.09375
    ch0 = (a * (0.625 * 2.0 + 64.625 * 0.5) + 7.09375 * -0.25) / l
    ch1 = (a * (1.0 * -1.0 + 64.625 * 0.5) + (0.1875 * 1.0 + 7.09375 * -0.25)) / l
    rest = (a * 64.625 * 0.5 + 7.09375 * -0.25) / l
    O, lo = orc.attention(p, orc.P_EXPCAST, softmax_scale=LN2_F32, rows=np.array([0], np.int32), return_l=True,
                          tau=0.0)
    got = _f32(O[0, 0])
    assert lo[0, 0] == pytest.approx(l, rel=1e-15)
    assert got[0] == np.float32(_f32(orc.bf16_round(ch0)))
    assert got[1] == np.float32(_f32(orc.bf16_round(ch1)))
    assert np.all(got[2:] == np.float32(_f32(orc.bf16_round(rest))))
    # codes taken against the final max instead would give block 0 key 0 the
    # code of t = 27.65 -> 28 (0.09375), not alpha * 1.0 = 0.0884: distinguishable
    assert abs(0.09375 - a) > 1e-3
    # exp-then-convert path: block 0 as above (2^-0.6875 = 0.6209 -> 0.625; 0.5);
    # block 1: 2^-2.5 = 0.17678 -> 0.171875 (35); 2^-4.5 = 0.044194 -> 0.04296875 (19)
    r1 = 1.0 + 0.171875 + 126 * 0.04296875
    l2 = 64.625 * a + r1
    rest2 = (a * 64.625 * 0.5 + r1 * -0.25) / l2
    O2, lo2 = orc.attention(p, orc.P_EXP, softmax_scale=LN2_F32, rows=np.array([0], np.int32), return_l=True,
                            tau=0.0)
    assert lo2[0, 0] == pytest.approx(l2, rel=1e-15)
    assert np.all(_f32(O2[0, 0])[2:] == np.float32(_f32(orc.bf16_round(rest2))))


def test_lazy_rescale_worked_example(orc):
    """tau = 8 (FlashAttention-4's lazy rescale): the reference max moves only
    when a block's max exceeds it by more than 8 (log2 units)."""
    row = np.array([0], np.int32)
    p = _two_block_case(orc, third=True)
    # block 0: m = 1, codes as in the tau = 0 example, rowsum0 = 64.625
    # block 1: 4.5 <= 1 + 8, m stays 1: key128 t=83.65 -> 84 (12.0); key129
    #          t=63.65 -> 64 (2.0); zeros t=47.65 -> 48 (0.5) x126  rowsum1 = 77
    # block 2: 12 > 1 + 8: alpha = 2^-11, m = 12; key256 -> 56 (1.0); zeros
    #          t=-40.35 -> flushed                                   rowsum2 = 1
    a = 2.0 ** -11
    l = (64.625 + 77.0) * a + 1.0
    ch0 = ((0.625 * 2.0 + 64.625 * 0.5 + 77.0 * -0.25) * a + 1.0) / l
    ch1 = ((-1.0 + 64.625 * 0.5 + 2.0 * 1.0 + 77.0 * -0.25) * a + 1.0) / l
    rest = ((64.625 * 0.5 + 77.0 * -0.25) * a + 1.0) / l
    O, lo = orc.attention(p, orc.P_EXPCAST, softmax_scale=LN2_F32, rows=row, return_l=True, tau=8.0)
    got = _f32(O[0, 0])
    assert lo[0, 0] == pytest.approx(l, rel=1e-15)
    assert got[0] == np.float32(_f32(orc.bf16_round(ch0)))
    assert got[1] == np.float32(_f32(orc.bf16_round(ch1)))
    assert np.all(got[2:] == np.float32(_f32(orc.bf16_round(rest))))
    # two blocks only, exp path: block 1 against m = 1: 2^3.5 = 11.31 -> 11 (83);
    # 2^1 -> 2 (64); 2^-1 -> 0.5                                      rowsum1 = 76
    p2 = _two_block_case(orc)
    O2, lo2 = orc.attention(p2, orc.P_EXP, softmax_scale=LN2_F32, rows=row, return_l=True, tau=8.0)
    assert lo2[0, 0] == pytest.approx(64.625 + 76.0, rel=1e-15)
    rest2 = (64.625 * 0.5 + 76.0 * -0.25) / (64.625 + 76.0)
    assert np.all(_f32(O2[0, 0])[2:] == np.float32(_f32(orc.bf16_round(rest2))))
    # with tau = 0 the same two blocks rescale at block 1 (the earlier example)
    _, lo3 = orc.attention(p2, orc.P_EXP, softmax_scale=LN2_F32, rows=row, return_l=True, tau=0.0)
    assert lo3[0, 0] != pytest.approx(lo2[0, 0])


@pytest.mark.parametrize("mode", [0, 1, 2, 3])
def test_constant_v_comes_back(orc, mode):
    vmode = 1 if mode == 2 else 0
    _, p = _prepped(seed=3, N=256, BH=1, vmode=vmode)
    p = dict(p)
    p["v_res"] = np.zeros_like(p["v_res"])
    const = np.array([orc.bf16_round(x) for x in np.linspace(-3, 3, 128)], np.uint16)
    p["v_mean"] = np.broadcast_to(const, p["v_mean"].shape).copy()
    O = orc.attention(p, mode)
    assert np.all(O == const[None, None, :])


@pytest.mark.parametrize("mode,tol", [(0, 0.0364), (1, 0.0294), (2, 0.25)])
def test_quantised_p_within_tv_of_exact_p(orc, mode, tol):
    # The TV bound holds in the normal range; a small softmax scale keeps every
    # row's log2-domain scores within 6 of its max, so nothing underflows.
    vmode = 1 if mode == 2 else 0
    _, p = _prepped(seed=4, N=512, BH=1, vmode=vmode)
    scale = 0.004
    rows = np.arange(0, 512, 17, dtype=np.int32)
    qh, kh, vh = _dequant(orc, p, 0)
    s = (qh[rows] @ kh.T) * scale * math.log2(math.e)
    assert (s.max(1) - s.min(1)).max() < 6.0
    Oq = _f32(orc.attention(p, mode, softmax_scale=scale, rows=rows)).astype(np.float64)
    Oe = _f32(orc.attention(p, orc.P_EXACT, softmax_scale=scale, rows=rows)).astype(np.float64)
    # |sum (w - w') v| <= 2 TV(w, w') max|v - centre| for each channel
    spread = (vh.max(0) - vh.min(0)) / 2
    dev = np.abs(Oq - Oe)[0] / spread[None, :]
    assert dev.max() <= 2 * tol + 2 ** -7


def test_nvfp4_worked_example(orc):
    """NVFP4 P and NVFP4 V on the two-block case (scores as in _two_block_case).

    V: g = 1, every 16-token scale E4M3 1.0; residual E2M1 codes 2.0 at
    (key 1, ch 0), -1.0 at (key 0, ch 1), 1.0 at (key 129, ch 1); means 0.5 and
    -0.25.  Per 16 keys: p = 2^(s - m), sf = E4M3(amax / 6),
    P = E2M1(p / dec(sf)) * dec(sf), worked by hand:

    tau = 8 (m = 1 throughout)
      block 0, keys 0-15: amax 1 -> sf E4M3(0.16667) = 0.171875 (midpoint to
               0.15625 is 0.1640625); p/sf: key0 5.818 -> 6 (P 1.03125), key1
               2^-0.6875 / 0.171875 = 3.611 -> 4 (P 0.6875), p = 0.5 -> 2.909 -> 3
               (P 0.515625); keys 16-127: amax 0.5 -> sf 0.0859375, 5.818 -> 6
               (P 0.515625).                                   rowsum0 = 66.6875
      block 1, keys 128-143: amax 2^3.5 -> sf E4M3(1.8856) = 1.875; key128
               6.034 -> 6 (saturated, P 11.25), key129 1.0667 -> 1 (P 1.875),
               0.2667 -> 0.5 (P 0.9375); keys 144-255 as above.  rowsum1 = 84
    tau = 0 (block 1 moves m to 4.5, alpha = 2^-3.5)
      block 1, keys 128-143: amax 1 -> sf 0.171875; key128 P 1.03125, key129
               2^-2.5 / 0.171875 = 1.0285 -> 1 (P 0.171875), 2^-4.5 -> 0.2571 ->
               0.5 (P 0.0859375); keys 144-255: amax 2^-4.5 -> amax / 6 = 0.0073657
               lies below E4M3's normal range (2^-6): the subnormal 3.771 * 2^-9
               rounds to sf = 4 * 2^-9, p / sf = 5.657 -> 6 (P 0.046875).
                                                               rowsum1 = 7.65625
    """
    p = nvfp4_two_block_case(orc)
    row = np.array([0], np.int32)
    mean = 66.6875 * 0.5  # block 0's mean term
    for tau, a, r1, res1 in [(8.0, 1.0, 84.0, (0.0, 1.875)), (0.0, 2.0 ** -3.5, 7.65625, (0.0, 0.171875))]:
        l = 66.6875 * a + r1
        ch0 = (a * (0.6875 * 2.0 + mean) + res1[0] + r1 * -0.25) / l
        ch1 = (a * (1.03125 * -1.0 + mean) + res1[1] + r1 * -0.25) / l
        rest = (a * mean + r1 * -0.25) / l
        O, lo = orc.attention(p, orc.P_NVFP4, softmax_scale=LN2_F32, rows=row, return_l=True, tau=tau)
        got = _f32(O[0, 0])
        assert lo[0, 0] == pytest.approx(l, rel=1e-15), tau
        assert got[0] == np.float32(_f32(orc.bf16_round(ch0))), tau
        assert got[1] == np.float32(_f32(orc.bf16_round(ch1))), tau
        assert np.all(got[2:] == np.float32(_f32(orc.bf16_round(rest)))), tau
