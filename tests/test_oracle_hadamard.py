"""Pins for the QK Hadamard option of the oracle's prep (the Q/K prior art the
insight page discusses, section "Softmax Has to Be Designed for Low-Bit
Execution Too"; an optional prep flag here).

The transform is pinned against the Sylvester Hadamard matrix (scipy), its
algebra (H H = 128 I, rows of H as transforms of basis vectors) and, through
the prep, against what the rotation must preserve: the dequantised scores
sq sk (q8 . k8) approximate Q K^T with the key scale carrying the exact factor
1/128 (a missing or wrong factor puts them off by ~128x).  Whether the
rotation improves the FP8 scores depends on the data: E4M3 is a floating-point
format, so an outlier channel costs the others little precision, and on this
recipe the rotation does not help (the pages find QK Hadamard moves results
by only 0.1-0.3 dB); the tests check correctness, not a gain."""
import numpy as np
import pytest

from bit_attention_video_smooth_gb300 import inputs as I

pytestmark = pytest.mark.filterwarnings("ignore::DeprecationWarning")


def test_fwht_matches_the_hadamard_matrix(orc):
    scipy_linalg = pytest.importorskip("scipy.linalg")
    H = scipy_linalg.hadamard(128).astype(np.float64)
    # small integers: every butterfly is exact, so the transform is exactly H x
    xi = np.random.default_rng(1).integers(-60, 60, (8, 128)).astype(np.float32)
    assert np.array_equal(orc.fwht_f32(xi).astype(np.float64), xi.astype(np.float64) @ H.T)
    # general values: within the rounding of seven fp32 butterfly stages
    x = np.random.default_rng(2).standard_normal((16, 128)).astype(np.float32)
    ref = x.astype(np.float64) @ H.T
    assert np.abs(orc.fwht_f32(x) - ref).max() <= 8 * np.abs(x).sum(axis=1).max() * 2.0 ** -24


def test_fwht_algebra(orc):
    e = np.eye(128, dtype=np.float32)
    rows = orc.fwht_f32(e)                       # H e_j = column j of H (H is symmetric)
    assert np.array_equal(rows[0], np.ones(128, np.float32))
    assert np.array_equal(rows[1], np.tile(np.array([1, -1], np.float32), 64))
    assert np.array_equal(rows[2], np.tile(np.array([1, 1, -1, -1], np.float32), 32))
    xi = np.random.default_rng(3).integers(-30, 30, (4, 128)).astype(np.float32)
    assert np.array_equal(orc.fwht_f32(orc.fwht_f32(xi)), 128 * xi)     # H H = 128 I


def _dequant_scores(orc, ref, h, rows, N):
    q = orc.e4m3_decode(ref["q8"][h][rows]).astype(np.float64) * np.repeat(ref["sq"][h], 128)[rows][:, None]
    k = orc.e4m3_decode(ref["k8"][h]).astype(np.float64) * np.repeat(ref["sk"][h], 128)[:, None]
    return q @ k.T


def test_hadamard_prep_keeps_the_scores(orc):
    w = I.WORKLOADS["tiny"]
    Q, K, V = I.make_qkv(w, seed=21)
    perm = I.random_perm(w.BH, w.N, seed=22).numpy()
    q16, k16, v16 = (I.to_u16(t).reshape(w.BH, w.N, 128) for t in (Q, K, V))
    plain = orc.prep(q16, k16, v16, perm)
    had = orc.prep(q16, k16, v16, perm, qk_hadamard=True)
    # V is untouched by the option
    for key in ("v_res", "v_scale", "v_mean"):
        assert np.array_equal(plain[key], had[key])
    # the key scale carries exactly 1/128: amax of the rotated block / 448 / 128
    kf = (k16[0][perm[0]].astype(np.uint32) << 16).view(np.float32)
    rot = orc.fwht_f32(kf[:128])
    amax = np.float32(np.abs(rot).max())
    assert had["sk"][0][0] == np.float32(np.float32(amax / np.float32(448.0)) * np.float32(1.0 / 128.0))
    # dequantised scores approximate Q K^T (keys in permuted order) in both modes
    rows = np.arange(0, w.N, 37)
    qf = (q16[0].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    exact = qf[rows] @ kf.astype(np.float64).T
    err = {}
    for name, ref in (("plain", plain), ("hadamard", had)):
        s = _dequant_scores(orc, ref, 0, rows, w.N)
        err[name] = np.linalg.norm(s - exact) / np.linalg.norm(exact)
        assert err[name] < 0.1, (name, err[name])


def test_hadamard_prep_attention_stays_close_to_exact(orc):
    w = I.WORKLOADS["tiny"]
    Q, K, V = I.make_qkv(w, seed=23)
    perm = I.random_perm(w.BH, w.N, seed=24).numpy()
    q16, k16, v16 = (I.to_u16(t).reshape(w.BH, w.N, 128) for t in (Q, K, V))
    rows = np.arange(0, w.N, 64)
    exact = orc.attention_exact(q16, k16, v16, rows=rows)
    errs = {}
    for had in (False, True):
        ref = orc.prep(q16, k16, v16, perm, qk_hadamard=had)
        got = orc.bf16_to_f32(orc.attention(ref, orc.P_EXACT, rows=rows)).astype(np.float64)
        errs[had] = np.linalg.norm(got - exact) / np.linalg.norm(exact)
    # exact-P attention over the dequantised operands: the error is the Q/K FP8
    # quantisation alone, of the same size with or without the rotation
    assert errs[False] < 0.2 and errs[True] < 0.2, errs
    assert errs[True] < 2 * errs[False], errs
