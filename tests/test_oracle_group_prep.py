"""Pins for the oracle's V-Smooth group (k-means + stable permutation) and the
fused prep (block means, residual quantisation, Q/K FP8 quantisation).

Group (paper page, "method"): per (batch, head), online k-means on the Value
tokens; Key and Value are permuted together by cluster label.  Prep: each
128-token block subtracts its own mean (stored as a 16-bit vector), only the
residual is quantised (per-channel E4M3, or NVFP4), Q and K go to FP8.

Pins: brute-force k-means optimum on tiny inputs, the Lloyd fixed point
re-derived with numpy, numpy's stable argsort, torch's casts for every
quantiser, and the dequantisation error bounds of each format.
"""
import itertools

import numpy as np
import pytest
import torch

from bit_attention_video_smooth_gb300 import inputs as I


def _f32(u16):
    return (np.asarray(u16, np.uint16).astype(np.uint32) << 16).view(np.float32)


def _bf16(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _sse(x, lab, k):
    s = 0.0
    for c in range(k):
        pts = x[lab == c]
        if len(pts):
            s += ((pts - pts.mean(0)) ** 2).sum()
    return s


@pytest.mark.parametrize("seed", range(6))
def test_kmeans_brute_force_tiny(orc, seed):
    rng = np.random.default_rng(seed)
    N, d, k = 8, 4, 3
    x = rng.standard_normal((N, d)).astype(np.float32)
    if seed % 2 == 0:                       # well separated: three tight groups
        centres = rng.standard_normal((k, d)) * 20
        # the strided initial tokens floor((c + 1/2) N / k) = 1, 4, 6 sit in
        # clusters 0, 1, 2: Lloyd then reaches the global optimum
        lab_true = np.array([1, 0, 2, 0, 1, 2, 2, 1])
        x = (centres[lab_true] + 0.01 * rng.standard_normal((N, d))).astype(np.float32)
    v = _bf16(x)
    xf = _f32(v).astype(np.float64)
    labels, counts, cent = orc.kmeans(v[None], k, iters=10)
    lab = labels[0]
    best = min(_sse(xf, np.array(p), k) for p in itertools.product(range(k), repeat=N))
    got = _sse(xf, lab, k)
    assert got >= best - 1e-9
    if seed % 2 == 0:
        assert abs(got - best) < 1e-9       # the global optimum on separated data
    # fixed point: re-assigning to the returned centroids changes nothing
    dist = ((xf[:, None, :] - cent[0][None].astype(np.float64)) ** 2).sum(-1)
    assert np.array_equal(np.argmin(dist, axis=1), lab)
    assert np.array_equal(counts[0], np.bincount(lab, minlength=k))


def test_kmeans_objective_hand_values(orc):
    """The k-means objective the GPU group is compared by: a hand-summed case,
    the objective at the optimal centroids of the brute-force case's labels,
    and invariance under renumbering the clusters (centroid rows permuted with
    the labels), which a wrong centroid index would break."""
    v = _bf16(np.array([[1, 2], [3, 4], [0, 0], [5, -1]], np.float32))
    lab = np.array([0, 0, 1, 1], np.int32)
    cent = np.array([[2, 3], [0, 1]], np.float32)
    # (1+1) + (1+1) + (0+1) + (25+4)
    assert orc.kmeans_sse(v, lab, cent) == 34.0
    assert orc.kmeans_sse(v, 1 - lab, cent[::-1].copy()) == 34.0
    assert orc.kmeans_sse(v, lab, np.array([[2, 3], [2.5, -0.5]], np.float32)) == 4.0 + 13.0
    rng = np.random.default_rng(3)
    x = _bf16(rng.standard_normal((40, 16)).astype(np.float32))
    xf = _f32(x).astype(np.float64)
    lab = rng.integers(0, 5, 40).astype(np.int32)
    means = np.stack([xf[lab == c].mean(0) for c in range(5)])
    got = orc.kmeans_sse(x, lab, means.astype(np.float32))
    assert abs(got - _sse(xf, lab, 5)) <= 1e-6 * got


def test_kmeans_init_and_empty_cluster(orc):
    # k = N: every token is its own strided initial centroid; duplicate rows
    # leave one cluster empty and it keeps its previous centroid
    N, d = 4, 2
    x = np.array([[0, 0], [0, 0], [5, 5], [9, 9]], np.float32)
    v = _bf16(x)[None]
    labels, counts, cent = orc.kmeans(v, 4, iters=3)
    assert labels[0].tolist() == [0, 0, 2, 3]            # ties go to the lowest index
    assert counts[0].tolist() == [2, 0, 1, 1]
    assert np.array_equal(cent[0], x)                    # centroid 1 kept its init value


def test_kmeans_one_iteration_matches_numpy_lloyd(orc):
    rng = np.random.default_rng(7)
    BH, N, d, k = 2, 640, 16, 5
    v = _bf16(rng.standard_normal((BH, N, d)))
    labels, counts, cent = orc.kmeans(v, k, iters=1)
    for bh in range(BH):
        xf = _f32(v[bh]).astype(np.float64)
        init = xf[[(2 * c + 1) * N // (2 * k) for c in range(k)]]
        lab = np.argmin(((xf[:, None] - init[None]) ** 2).sum(-1), axis=1)
        assert np.array_equal(lab, labels[bh])
        for c in range(k):
            np.testing.assert_allclose(cent[bh, c], xf[lab == c].mean(0), rtol=1e-6, atol=1e-7)


def test_separated_clusters_recovered(orc):
    BH, N, d, k = 2, 1024, 128, 8
    v = I.to_u16(I.make_separated_v(BH, N, d, k, seed=3))
    labels, counts, cent = orc.kmeans(v, k, iters=4)
    for bh in range(BH):
        xf = _f32(v[bh])
        pos = [(2 * c + 1) * N // (2 * k) for c in range(k)]
        # every token lands with the strided token of its own cluster
        near = np.argmin(((xf[:, None] - xf[pos][None]) ** 2).sum(-1), axis=1)
        assert np.array_equal(labels[bh], near)


def test_stable_sort_matches_numpy(orc):
    rng = np.random.default_rng(8)
    lab = rng.integers(0, 13, (3, 5000)).astype(np.int32)
    perm, counts = orc.stable_sort(lab, 13)
    for bh in range(3):
        assert np.array_equal(perm[bh], np.argsort(lab[bh], kind="stable"))
        assert np.array_equal(counts[bh], np.bincount(lab[bh], minlength=13))
    # k = 1: identity permutation
    perm1, _ = orc.stable_sort(np.zeros((1, 300), np.int32), 1)
    assert np.array_equal(perm1[0], np.arange(300))


def _setup(seed=0, N=512, BH=2):
    w = I.with_n(I.WORKLOADS["tiny"], N, H=BH)
    q, k, v = (I.to_u16(t).reshape(BH, N, 128) for t in I.make_qkv(w, seed=seed))
    perm = I.random_perm(BH, N, seed=seed + 1).numpy()
    return q, k, v, perm


def test_prep_block_means_match_numpy(orc):
    q, k, v, perm = _setup()
    out = orc.prep(q, k, v, perm)
    BH, N, d = v.shape
    for bh in range(BH):
        g = _f32(v[bh][perm[bh]]).astype(np.float64).reshape(N // 128, 128, d)
        mean = (g.sum(1).astype(np.float32) / np.float32(128.0))
        assert np.array_equal(out["v_mean"][bh], _bf16(mean))


def test_prep_residual_e4m3_matches_torch_cast(orc):
    q, k, v, perm = _setup(seed=1)
    out = orc.prep(q, k, v, perm)
    BH, N, d = v.shape
    nb = N // 128
    for bh in range(BH):
        g = _f32(v[bh][perm[bh]]).reshape(nb, 128, d)
        mu = _f32(out["v_mean"][bh])[:, None, :]
        R = (g - mu).astype(np.float32)                       # exact fp32 subtraction
        a = np.abs(R).reshape(N, d).max(0)
        inv = np.float32(448.0) / a
        np.testing.assert_array_equal(out["v_scale"][bh], a / np.float32(448.0))
        ref = torch.from_numpy((R * inv[None, None, :]).astype(np.float32)).to(torch.float8_e4m3fn)
        ref = ref.view(torch.uint8).numpy().transpose(0, 2, 1)    # [blk][ch][tok]
        assert np.array_equal(out["v_res"][bh], ref)
        # the per-channel amax maps to exactly 448 (code 126)
        assert np.all(np.abs(out["v_res"][bh].astype(np.int16) & 0x7F).reshape(nb, d, 128).max(axis=(0, 2)) == 126)
        # dequantised residual + mean reconstructs V within the E4M3 bound
        deq = orc.e4m3_decode(out["v_res"][bh]).transpose(0, 2, 1) * out["v_scale"][bh][None, None, :]
        err = np.abs(deq + mu - g)
        bound = np.maximum(np.abs(R) * 2.0 ** -4, 2.0 ** -10 * out["v_scale"][bh][None, None, :]) * 1.0001
        assert np.all(err <= bound + 1e-6)


def test_prep_qk_fp8_matches_torch_cast(orc):
    q, k, v, perm = _setup(seed=2)
    out = orc.prep(q, k, v, perm)
    BH, N, d = q.shape
    nb = N // 128
    for bh in range(BH):
        for name, src in (("q8", _f32(q[bh])), ("k8", _f32(k[bh])[perm[bh]])):
            blocks = src.reshape(nb, 128, d)
            amax = np.abs(blocks).max(axis=(1, 2))
            inv = (np.float32(448.0) / amax).astype(np.float32)
            ref = torch.from_numpy((blocks * inv[:, None, None]).astype(np.float32)).to(torch.float8_e4m3fn)
            assert np.array_equal(out[name][bh].reshape(nb, 128, d), ref.view(torch.uint8).numpy())
            scale = out["sq" if name == "q8" else "sk"][bh]
            np.testing.assert_array_equal(scale, amax / np.float32(448.0))


def test_prep_nvfp4_residual_grid_and_bound(orc):
    q, k, v, perm = _setup(seed=3, N=256, BH=1)
    out = orc.prep(q, k, v, perm, vmode=orc.V_NVFP4)
    N, d = v.shape[1:]
    nb = N // 128
    g = _f32(v[0][perm[0]]).reshape(nb, 128, d)
    mu = _f32(out["v_mean"][0])[:, None, :]
    R = (g - mu).astype(np.float32)
    amax = np.abs(R).max()
    gs = out["v_scale"][0]
    assert gs == np.float32(amax / np.float32(6.0 * 448.0))
    grid = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6])
    for b in range(nb):
        for ch in range(0, d, 7):
            for grp in range(8):
                r = R[b, grp * 16:(grp + 1) * 16, ch].astype(np.float64)
                sf = out["v_sf"][0, b, ch, grp]
                sfv = orc.e4m3_decode(np.array([sf]))[0]
                byts = out["v_res"][0, b, ch, grp * 8:(grp + 1) * 8]
                nib = np.stack([byts & 15, byts >> 4], axis=1).ravel()
                deq = orc.e2m1_decode(nib) * sfv * gs
                if sf == 0:
                    assert np.all(deq == 0)
                    continue
                # each value is the nearest point of its scaled grid (saturating at 6)
                step = sfv * gs
                x = np.clip(np.abs(r) / step, 0, 6)
                best = np.abs(x[:, None] - grid[None]).min(1) * step
                assert np.all(np.abs(np.abs(deq) - np.clip(np.abs(r), 0, 6 * step)) <= best * (1 + 1e-5) + 1e-12)
                # the group scale is the E4M3 rounding of amax16 / (6 g)
                assert abs(sfv - np.abs(r).max() / (6 * gs)) <= 2.0 ** -4 * np.abs(r).max() / (6 * gs) + 2.0 ** -10
