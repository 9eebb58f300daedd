"""The oracle's K smoothing option (prep flag), pinned on the CPU.

K smoothing subtracts the keys' channel mean over the sequence of each (b,h)
before the FP8 quantisation (SageAttention's treatment of the keys' channel
bias, which the paper page's motivation and the insight page's section "Value
Is the Error Source Earlier Methods Underestimated" cite as the handling of
Q/K outliers).  Every score of a query row then moves by the same amount, so
exact softmax attention is unchanged.  The mean is fp32 with a fixed order (a
halving tree per permuted 128-token block, the block sums in block order,
divided by N), so that the device can reproduce it bit for bit.
"""
import numpy as np
import pytest
import torch

import oracle
from bit_attention_video_smooth_gb300 import inputs as I

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _u16(t):
    return I.to_u16(t).numpy() if isinstance(t, torch.Tensor) else t


def _f32(u16):
    return (u16.astype(np.uint32) << 16).view(np.float32)


def _case(BH=2, N=512, seed=3, offset=0.0):
    w = I.with_n(I.WORKLOADS["tiny"], N, H=BH)
    q, k, v = I.make_qkv(w, seed=seed)
    if offset:
        # a channel bias on a few key channels, the case smoothing is for
        k = k.float()
        k[..., :4] += offset
        k = k.to(torch.bfloat16)
    u = lambda t: I.to_u16(t).reshape(BH, N, 128)
    perm = I.random_perm(BH, N, seed=seed + 1).numpy()
    return u(q), u(k), u(v), perm


def test_mean_is_the_sequence_mean_within_the_fp32_bound():
    _, k, _, perm = _case(BH=3, N=1024)
    mu = oracle.k_channel_mean(k, perm)
    kf = _f32(k).astype(np.float64)
    exact = kf.mean(axis=1)
    # fp32 rounding of at most N additions and one division
    bound = 1024 * 2.0 ** -24 * np.abs(kf).max(axis=1) + 2.0 ** -23 * np.abs(exact)
    assert np.all(np.abs(mu - exact) <= bound)
    # and it is no other statistic: far from the first block's mean where they differ
    first = kf[:, :128].mean(axis=1)
    assert np.abs(mu - exact).max() < 0.1 * np.abs(first - exact).max()


def test_mean_is_exact_when_every_partial_sum_is():
    rng = np.random.default_rng(5)
    BH, N = 2, 1024
    # small integers times 1/4: every partial sum is exact in fp32, whatever the order
    vals = rng.integers(-64, 64, size=(BH, N, 128)).astype(np.float32) / 4
    k = (vals.view(np.uint32) >> 16).astype(np.uint16)
    assert np.array_equal(_f32(k), vals)
    perm = np.stack([rng.permutation(N) for _ in range(BH)]).astype(np.int32)
    mu = oracle.k_channel_mean(k, perm)
    total = vals.astype(np.float64).sum(axis=1)
    assert np.array_equal(mu, (total.astype(np.float32) / np.float32(N)).astype(np.float32))


def test_mean_follows_the_stated_order():
    """Values whose fp32 sum depends on the order: one block holds 2^24 at token
    0, 1.0 at tokens 64 and 96, -2^24 at token 32.  The halving tree adds token
    i + 64 to token i first (2^24 + 1 rounds to 2^24), then i + 32 (-2^24 + 1 =
    -2^24 + 1 exactly); a left-to-right sum would give another result."""
    N = 256
    col = np.zeros((1, N, 128), np.float32)
    col[0, 0, :] = 2.0 ** 24
    col[0, 64, :] = 1.0
    col[0, 32, :] = -(2.0 ** 24)
    col[0, 96, :] = 1.0
    k = (col.view(np.uint32) >> 16).astype(np.uint16)
    assert np.array_equal(_f32(k), col)
    perm = np.arange(N, dtype=np.int32)[None]
    mu = oracle.k_channel_mean(k, perm)
    # tree: y0 = fl(2^24 + 1) = 2^24 (tie to even), y32 = -2^24 + 1; y0 + y32 = 1
    assert np.all(mu == np.float32(1.0) / np.float32(N))
    seq = np.float32(0)
    for x in col[0, :, 0]:
        seq = np.float32(seq + x)
    assert seq != np.float32(1.0)        # the order matters on this input


def test_exact_attention_is_unchanged_by_the_shift():
    q, k, v, perm = _case(BH=2, N=512, offset=6.0)
    mu = oracle.k_channel_mean(k, perm)
    qd, kd, vd = (_f32(a).astype(np.float64) for a in (q, k, v))
    # the oracle's mean, subtracted exactly (fp64): the invariance is a property
    # of the shift itself, before any rounding of the shifted keys
    ks = kd - mu.astype(np.float64)[:, None, :]

    def attend(qh, keys, vh):
        s = qh @ keys.T / np.sqrt(128)
        p = np.exp(s - s.max(axis=1, keepdims=True))
        return (p / p.sum(axis=1, keepdims=True)) @ vh

    for bh in range(2):
        ref = attend(qd[bh], kd[bh], vd[bh])
        got = attend(qd[bh], ks[bh], vd[bh])
        assert np.abs(got - ref).max() <= 1e-9 * np.abs(ref).max()
    # a per-block shift (a plausible mistake) is not softmax-invariant
    kb = kd.copy()
    kb[:, :128] -= 3.0
    s0 = qd[0] @ kd[0].T
    s1 = qd[0] @ kb[0].T
    d = s1 - s0
    assert np.ptp(d, axis=1).max() > 1.0


def test_smoothed_key_bytes_rederived_with_torch():
    q, k, v, perm = _case(BH=2, N=512, offset=6.0)
    ref = oracle.prep(q, k, v, perm, k_smooth=True)
    mu = oracle.k_channel_mean(k, perm)
    for bh in range(2):
        ks = torch.from_numpy(_f32(k[bh])[perm[bh]] - mu[bh][None, :])     # permuted order, fp32
        for b in range(512 // 128):
            blk = ks[128 * b:128 * (b + 1)]
            amax = blk.abs().max()
            inv = torch.tensor(448.0, dtype=torch.float32) / amax
            codes = (blk * inv).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
            assert np.array_equal(codes, ref["k8"][bh, 128 * b:128 * (b + 1)])
            assert ref["sk"][bh, b] == np.float32(amax.item() / np.float32(448.0))


def test_only_the_keys_change():
    q, k, v, perm = _case(BH=2, N=384, offset=4.0)
    a = oracle.prep(q, k, v, perm)
    b = oracle.prep(q, k, v, perm, k_smooth=True)
    for key in ("q8", "sq", "v_res", "v_scale", "v_mean"):
        assert np.array_equal(a[key], b[key]), key
    assert not np.array_equal(a["k8"], b["k8"])


def test_smoothing_reduces_the_key_quantisation_error_under_a_channel_bias():
    q, k, v, perm = _case(BH=2, N=512, offset=24.0)
    kf = _f32(k).astype(np.float64)
    mu = oracle.k_channel_mean(k, perm)
    errs = {}
    for smooth in (False, True):
        p = oracle.prep(q, k, v, perm, k_smooth=smooth)
        deq = torch.from_numpy(p["k8"]).view(torch.float8_e4m3fn).double().numpy()
        deq = deq * np.repeat(p["sk"].astype(np.float64), 128, axis=1)[:, :, None]
        target = np.stack([kf[bh][perm[bh]] for bh in range(2)])
        if smooth:
            target = target - mu[:, None, :]
        errs[smooth] = np.linalg.norm(deq - target) / np.linalg.norm(target - target.mean(axis=1, keepdims=True))
    assert errs[True] < 0.5 * errs[False]


def test_constant_keys_smooth_to_zero():
    BH, N = 1, 256
    k = np.full((BH, N, 128), 0x3FC0, np.uint16)      # 1.5 everywhere
    q = k.copy()
    v = k.copy()
    perm = np.arange(N, dtype=np.int32)[None]
    assert np.all(oracle.k_channel_mean(k, perm) == np.float32(1.5))
    p = oracle.prep(q, k, v, perm, k_smooth=True)
    assert not p["k8"].any() and np.all(p["sk"] == 1.0)
