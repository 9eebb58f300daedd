"""The seeded input recipe, checked against what it promises: shapes and
dtypes, determinism per seed, the channel outliers of Q and K, the token
outliers of V on a per-head channel set, the strided tokens of the separated-V
generator, and the permutation and row-sampling helpers."""
import numpy as np
import torch

from bit_attention_video_smooth_gb300 import inputs as I


def test_shapes_dtypes_and_seeding():
    w = I.WORKLOADS["tiny"]
    a = I.make_qkv(w, seed=5)
    b = I.make_qkv(w, seed=5)
    c = I.make_qkv(w, seed=6)
    for x, y, z in zip(a, b, c):
        assert x.shape == (w.B, w.H, w.N, w.d) and x.dtype == torch.bfloat16 and x.is_contiguous()
        assert torch.equal(x, y)
        assert not torch.equal(x, z)
    assert I.with_n(w, 4096, H=3).BH == 3 and I.with_n(w, 4096).N == 4096


def test_qk_channel_outliers_per_head():
    w = I.WORKLOADS["tiny"]
    q, k, _ = I.make_qkv(w, seed=1)
    for x in (q, k):
        sd = x.float().view(w.BH, w.N, w.d).std(dim=1)            # per head, per channel
        for h in range(w.BH):
            big = torch.nonzero(sd[h] > 4.0).flatten()
            assert big.numel() == w.qk_channels, (h, big)
            assert torch.all((sd[h][big] - w.qk_mult).abs() < 1.5)
            small = torch.ones(w.d, dtype=torch.bool)
            small[big] = False
            assert torch.all((sd[h][small] - 1.0).abs() < 0.15)
    # the outlier channels are drawn per head, and separately for Q and K
    sets = [set(torch.nonzero(x.float().view(w.BH, w.N, w.d).std(dim=1)[h] > 4.0).flatten().tolist())
            for x in (q, k) for h in range(w.BH)]
    assert len({frozenset(s) for s in sets}) > 1


def test_v_token_outliers_on_a_per_head_channel_set():
    w = I.WORKLOADS["tiny"]
    _, _, v = I.make_qkv(w, seed=2)
    vf = v.float().view(w.BH, w.N, w.d).abs()
    n_out = round(w.v_frac * w.N)
    chans = []
    for h in range(w.BH):
        ch = torch.nonzero(vf[h].amax(dim=0) > 6.0).flatten()
        assert ch.numel() == w.v_channels, (h, ch)
        tok = torch.nonzero(vf[h][:, ch].amax(dim=1) > 6.0).flatten()
        assert tok.numel() == n_out, (h, tok.numel())
        chans.append(frozenset(ch.tolist()))
    assert len(set(chans)) == w.BH                          # a different channel set per head


def test_separated_v_places_the_strided_tokens_in_distinct_clusters():
    BH, N, d, k = 2, 1024, 128, 8
    v = I.make_separated_v(BH, N, d, k, seed=3).float()
    pos = [((2 * c + 1) * N) // (2 * k) for c in range(k)]
    for h in range(BH):
        x = v[h, pos]
        dist = torch.cdist(x, x)
        off = dist[~torch.eye(k, dtype=torch.bool)]
        assert off.min() > 20.0                              # centres ~ N(0, 8^2) in 128 dims
        # every token sits near one of the strided tokens' centres (noise 0.05)
        near = torch.cdist(v[h], x).min(dim=1).values
        assert near.max() < 2.0


def test_perm_and_sampled_rows():
    p = I.random_perm(3, 640, seed=4)
    assert p.dtype == torch.int32 and p.shape == (3, 640)
    for r in p:
        assert np.array_equal(np.sort(r.numpy()), np.arange(640))
    rows = I.sample_rows(70656, 48, seed=9).numpy()
    assert rows.size == 48 and np.all(np.diff(rows) > 0)
    assert {0, 127, 70656 - 128, 70656 - 1} <= set(rows.tolist())
    small = I.sample_rows(256, 256, seed=1).numpy()
    assert np.array_equal(small, np.arange(256))
    assert np.array_equal(I.sample_rows(128, 8, seed=2).numpy()[[0, -1]], [0, 127])
    for seed in range(200):                               # never fewer rows than asked for
        assert I.sample_rows(512, 40, seed=seed).numpy().size == 40
