"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle on the
same seeded inputs.

Bars: ExpCast codes, E4M3 conversions, cluster labels on well-separated inputs
and the permutation bit-exact; FP8 Q/K bytes and scales exact; E4M3 residual
bytes >= 99.99% identical, the rest one code apart; attention output within
relative L2 <= 1e-3 and max-abs <= 4e-3 * max|O| of the oracle.
"""
import numpy as np
import pytest
import torch

from bit_attention_video_smooth_gb300 import inputs as I
from cases import LN2_F32, nvfp4_two_block_case, two_block_case

pytestmark = pytest.mark.gpu

REL_L2 = 1e-3
MAX_ABS = 4e-3


def _f32(u16):
    return (np.asarray(u16, np.uint16).astype(np.uint32) << 16).view(np.float32)


def _dev(a, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.view(dtype)
    return t.cuda()


def _o_close(got_u16, ref_u16):
    g = _f32(got_u16).astype(np.float64)
    r = _f32(ref_u16).astype(np.float64)
    rel = np.linalg.norm(g - r) / max(np.linalg.norm(r), 1e-30)
    mx = np.abs(g - r).max() / max(np.abs(r).max(), 1e-30)
    return rel, mx


# ---------------------------------------------------------------------------
# formats and the ExpCast map
# ---------------------------------------------------------------------------
def test_expcast_codes_bit_exact(V, orc):
    rng = np.random.default_rng(11)
    n = 1 << 20
    s = np.concatenate([rng.standard_normal(n) * 2e4, rng.uniform(-50, 50, n)]).astype(np.float32)
    c = np.concatenate([rng.uniform(1e-5, 1e-3, n), rng.uniform(0.01, 2, n)]).astype(np.float32)
    m = (s * c).astype(np.float32) + rng.uniform(0, 12, 2 * n).astype(np.float32)   # m >= s*c mostly
    # edge cases: t exactly at .5 boundaries, at the flush threshold, above the clip
    edge_s = np.array([0.0, 0.0, 0.0, 1.0, -1.0, 20.0, np.inf, -np.inf, np.nan, 1e30], np.float32)
    edge_c = np.ones_like(edge_s)
    edge_m = np.array([0.0, 6.01875, 6.0187, -10.0, 0.0, 0.0, 0.0, 0.0, 0.0, 0.0], np.float32)
    # running maxima beyond 2^26, where the FMA's rounding can push codes past
    # 126 and the clip matters (the kernel's slow path)
    big_m = np.repeat(np.array([1e8, -3e8, 3e9], np.float32), 4096)
    big_s = (big_m.astype(np.float64) * (1 + rng.uniform(-3e-7, 3e-7, big_m.size))).astype(np.float32)
    big_c = np.ones_like(big_m)
    s, c, m = (np.concatenate([a, b, e]) for a, b, e in
               ((s, edge_s, big_s), (c, edge_c, big_c), (m, edge_m, big_m)))
    ref = orc.expcast_codes(s, c, m)
    out = torch.empty(s.size, dtype=torch.uint8, device="cuda")
    V.vca_expcast_codes(_dev(s), _dev(c), _dev(m), out)
    got = out.cpu().numpy()
    assert np.array_equal(got, ref), np.flatnonzero(got != ref)[:10]


def test_e4m3_hardware_conversion_matches_oracle_everywhere(V, orc):
    # every non-NaN fp32 bit pattern, in chunks
    step = 1 << 28
    out = torch.empty(step, dtype=torch.uint8, device="cuda")
    for start in range(0, 1 << 32, step):
        V.vca_e4m3_encode_bits(start, step, out)
        got = out.cpu().numpy()
        ref = orc.e4m3_encode_bits(start, step)
        u = np.arange(start, start + step, dtype=np.uint64).astype(np.uint32)
        nan = (u & 0x7FFFFFFF) > 0x7F800000
        assert np.array_equal(got[~nan], ref[~nan]), hex(start)
        assert np.all((got[nan] & 0x7F) == 0x7F)


# ---------------------------------------------------------------------------
# group: k-means + stable permutation
# ---------------------------------------------------------------------------
# sizes span one token tile, several assign chunks with a ragged last one,
# and the cluster counts of both kernel variants (k <= 64, k <= 128)
@pytest.mark.parametrize("BH,N,k,iters", [(2, 1024, 8, 10), (3, 2 * 4096 + 384, 16, 4), (1, 256, 1, 2),
                                          (2, 2048, 64, 8), (1, 512, 128, 3), (1, 4096 + 128, 100, 5)])
def test_group_bit_exact_on_separated_clusters(V, orc, BH, N, k, iters):
    v16 = I.make_separated_v(BH, N, 128, k, seed=BH * 7 + k)
    ref_lab, ref_perm, ref_cnt, ref_cent = orc.group(I.to_u16(v16), k, iters)
    g = V.group(v16.view(1, BH, N, 128).cuda(), k, iters)
    torch.cuda.synchronize()
    assert np.array_equal(g.labels.cpu().numpy(), ref_lab)
    assert np.array_equal(g.perm.cpu().numpy(), ref_perm)
    assert np.array_equal(g.counts.cpu().numpy(), ref_cnt)
    np.testing.assert_allclose(g.centroids.cpu().numpy(), ref_cent, rtol=1e-5, atol=1e-5)


def _degenerate_v(BH, N, case, seed=17):
    """bf16 V [BH, N, 128]: every token the same vector per head ("constant"),
    or two distinct vectors alternating in runs of 8 tokens ("two")."""
    g = torch.Generator().manual_seed(seed)
    a = torch.randn((BH, 1, 128), generator=g)
    if case == "constant":
        v = a.expand(BH, N, 128)
    else:
        b = torch.randn((BH, 1, 128), generator=g) * 4.0
        pick = ((torch.arange(N) // 8) % 2 == 1).view(1, N, 1)
        v = torch.where(pick, b, a)
    return v.to(torch.bfloat16).contiguous()


@pytest.mark.parametrize("case,k", [("constant", 8), ("two", 4), ("two", 64)])
def test_group_on_degenerate_values(V, orc, case, k):
    """Ties everywhere: with every token equal all distances tie and every
    label is 0 (ties go to the lowest index; the other clusters stay empty and
    keep their centroids); with two distinct tokens the labels follow the
    initial centroids' copies of them, the lowest index among equal ones."""
    BH, N, iters = 2, 512, 3
    v16 = _degenerate_v(BH, N, case)
    ref_lab, ref_perm, ref_cnt, ref_cent = orc.group(I.to_u16(v16), k, iters)
    g = V.group(v16.view(1, BH, N, 128).cuda(), k, iters)
    torch.cuda.synchronize()
    assert np.array_equal(g.labels.cpu().numpy(), ref_lab)
    assert np.array_equal(g.perm.cpu().numpy(), ref_perm)
    assert np.array_equal(g.counts.cpu().numpy(), ref_cnt)
    np.testing.assert_allclose(g.centroids.cpu().numpy(), ref_cent, rtol=1e-6, atol=1e-6)
    if case == "constant":
        assert not ref_lab.any() and np.array_equal(ref_perm, np.tile(np.arange(N), (BH, 1)))


def _check_perm_properties(labels, perm, counts, k):
    BH, N = labels.shape
    for bh in range(BH):
        assert np.array_equal(np.sort(perm[bh]), np.arange(N))
        assert np.array_equal(perm[bh], np.argsort(labels[bh], kind="stable"))
        assert np.array_equal(counts[bh], np.bincount(labels[bh], minlength=k))


def test_group_realistic_inputs(V, orc):
    w = I.WORKLOADS["tiny"]
    _, _, v = I.make_qkv(w, seed=5)
    g = V.group(v.cuda(), w.k, w.iters)
    torch.cuda.synchronize()
    lab, perm, cnt, cent = (t.cpu().numpy() for t in (g.labels, g.perm, g.counts, g.centroids))
    _check_perm_properties(lab, perm, cnt, w.k)
    ref_lab, _, _, ref_cent = orc.group(I.to_u16(v).reshape(w.BH, w.N, 128), w.k, w.iters)
    agree = (lab == ref_lab).mean()
    assert agree > 0.99, agree
    v16 = I.to_u16(v).reshape(w.BH, w.N, 128)
    for bh in range(w.BH):
        sse_gpu = orc.kmeans_sse(v16[bh], lab[bh], cent[bh])
        sse_ref = orc.kmeans_sse(v16[bh], ref_lab[bh], ref_cent[bh])
        assert sse_gpu <= sse_ref * 1.005


# ---------------------------------------------------------------------------
# prep
# ---------------------------------------------------------------------------
def _prep_inputs(BH, N, seed):
    w = I.with_n(I.WORKLOADS["tiny"], N, H=BH)
    q, k, v = I.make_qkv(w, seed=seed)
    perm = I.random_perm(BH, N, seed=seed + 1)
    return q, k, v, perm


@pytest.mark.parametrize("BH,N,seed", [(2, 1024, 0), (3, 384, 1), (1, 128, 2), (2, 2432, 3)])
def test_prep_e4m3_parity(V, orc, BH, N, seed):
    q, k, v, perm = _prep_inputs(BH, N, seed)
    ref = orc.prep(*(I.to_u16(t).reshape(BH, N, 128) for t in (q, k, v)), perm.numpy())
    p = V.prep_quant(q.cuda(), k.cuda(), v.cuda(), perm.cuda(), V.VCA_V_E4M3)
    torch.cuda.synchronize()
    assert np.array_equal(p.q8.cpu().numpy(), ref["q8"])
    assert np.array_equal(p.k8.cpu().numpy(), ref["k8"])
    assert np.array_equal(p.sq.cpu().numpy(), ref["sq"])
    assert np.array_equal(p.sk.cpu().numpy(), ref["sk"])
    vm = p.v_mean.view(torch.int16).cpu().numpy().view(np.uint16)
    assert (vm == ref["v_mean"]).mean() >= 0.9999
    vr = p.v_res.cpu().numpy()
    same = (vr == ref["v_res"]).mean()
    assert same >= 0.9999, same
    diff = np.abs(vr.astype(np.int16) - ref["v_res"].astype(np.int16))
    near = (diff <= 1) | ((vr & 0x7F) == (ref["v_res"] & 0x7F))     # one code, or a signed zero
    assert near.all()
    np.testing.assert_allclose(p.v_scale.cpu().numpy(), ref["v_scale"], rtol=1e-6)


@pytest.mark.parametrize("BH,N,seed", [(2, 1024, 10), (3, 384, 11), (1, 2432, 12)])
def test_prep_qk_hadamard_parity(V, orc, BH, N, seed):
    """The QK Hadamard option: the device's fp32 butterflies in the documented
    order give the oracle's rotated rows bit for bit, so q8, k8, sq and sk
    match exactly; the V outputs are those of the plain prep."""
    q, k, v, perm = _prep_inputs(BH, N, seed)
    q16, k16, v16 = (I.to_u16(t).reshape(BH, N, 128) for t in (q, k, v))
    ref = orc.prep(q16, k16, v16, perm.numpy(), qk_hadamard=True)
    p = V.prep_quant(q.cuda(), k.cuda(), v.cuda(), perm.cuda(), V.VCA_V_E4M3, qk_hadamard=True)
    torch.cuda.synchronize()
    assert np.array_equal(p.q8.cpu().numpy(), ref["q8"])
    assert np.array_equal(p.k8.cpu().numpy(), ref["k8"])
    assert np.array_equal(p.sq.cpu().numpy(), ref["sq"])
    assert np.array_equal(p.sk.cpu().numpy(), ref["sk"])
    plain = V.prep_quant(q.cuda(), k.cuda(), v.cuda(), perm.cuda(), V.VCA_V_E4M3)
    torch.cuda.synchronize()
    assert torch.equal(plain.v_res, p.v_res) and torch.equal(plain.v_mean.view(torch.int16), p.v_mean.view(torch.int16))
    # attention over the rotated operands against the oracle's, end to end
    O = V.attention(p, 1, BH, N, expcast=True)
    torch.cuda.synchronize()
    O_ref = orc.attention(ref, orc.P_EXPCAST)
    rel, mx = _o_close(O.view(torch.int16).cpu().numpy().view(np.uint16).reshape(BH, N, 128), O_ref)
    assert rel <= REL_L2 and mx <= MAX_ABS, (rel, mx)


@pytest.mark.parametrize("BH,N,seed,hadamard", [(2, 1024, 20, False), (3, 384, 21, False), (1, 2432, 22, False),
                                                 (2, 640, 23, True)])
def test_prep_k_smooth_parity(V, orc, BH, N, seed, hadamard):
    """The K smoothing option: the device's block tree sums, their sum in block
    order and the division by N give the oracle's channel mean bit for bit, so
    q8, k8, sq and sk match exactly (with and without the QK Hadamard); the V
    outputs are those of the plain prep; attention over the smoothed operands
    matches the oracle's.  The keys carry a channel bias, the case smoothing
    is for."""
    q, k, v, perm = _prep_inputs(BH, N, seed)
    k = k.float()
    k[..., :6] += 5.0
    k = k.to(torch.bfloat16)
    q16, k16, v16 = (I.to_u16(t).reshape(BH, N, 128) for t in (q, k, v))
    ref = orc.prep(q16, k16, v16, perm.numpy(), qk_hadamard=hadamard, k_smooth=True)
    p = V.prep_quant(q.cuda(), k.cuda(), v.cuda(), perm.cuda(), V.VCA_V_E4M3, qk_hadamard=hadamard, k_smooth=True)
    torch.cuda.synchronize()
    assert np.array_equal(p.q8.cpu().numpy(), ref["q8"])
    assert np.array_equal(p.k8.cpu().numpy(), ref["k8"])
    assert np.array_equal(p.sq.cpu().numpy(), ref["sq"])
    assert np.array_equal(p.sk.cpu().numpy(), ref["sk"])
    plain = V.prep_quant(q.cuda(), k.cuda(), v.cuda(), perm.cuda(), V.VCA_V_E4M3, qk_hadamard=hadamard)
    torch.cuda.synchronize()
    assert torch.equal(plain.v_res, p.v_res) and torch.equal(plain.v_mean.view(torch.int16), p.v_mean.view(torch.int16))
    assert torch.equal(plain.q8, p.q8)
    O = V.attention(p, 1, BH, N, expcast=True)
    torch.cuda.synchronize()
    O_ref = orc.attention(ref, orc.P_EXPCAST)
    rel, mx = _o_close(O.view(torch.int16).cpu().numpy().view(np.uint16).reshape(BH, N, 128), O_ref)
    assert rel <= REL_L2 and mx <= MAX_ABS, (rel, mx)


def test_prep_k_smooth_needs_its_workspace(V):
    """The smoothing prep asks for more workspace (the block sums and the mean):
    a workspace sized for the plain prep is rejected before any launch."""
    B, H, N = 1, 2, 512
    plain = V.vca_workspace_bytes(V.VCA_OP_PREP, B, H, N)
    smooth = V.vca_workspace_bytes(V.VCA_OP_PREP_KSMOOTH, B, H, N)
    assert smooth > plain
    q, k, v, perm = _prep_inputs(B * H, N, 30)
    p = V.alloc_prep(B, H, N, V.VCA_V_E4M3)
    with pytest.raises(V.VCAError) as e:
        V.vca_prep_quant_ex(q.cuda(), k.cuda(), v.cuda(), perm.cuda(), V.VCA_V_E4M3, V.VCA_PREP_K_SMOOTH, p.q8, p.sq,
                            p.k8, p.sk, p.v_res, p.v_sf, p.v_scale, p.v_mean, p.ws)
    assert e.value.status == V.VCA_ERR_WORKSPACE


def test_prep_nvfp4_parity(V, orc):
    BH, N = 2, 1024
    q, k, v, perm = _prep_inputs(BH, N, 4)
    ref = orc.prep(*(I.to_u16(t).reshape(BH, N, 128) for t in (q, k, v)), perm.numpy(), vmode=orc.V_NVFP4)
    p = V.prep_quant(q.cuda(), k.cuda(), v.cuda(), perm.cuda(), V.VCA_V_NVFP4)
    torch.cuda.synchronize()
    assert np.array_equal(p.q8.cpu().numpy(), ref["q8"])
    assert np.array_equal(p.k8.cpu().numpy(), ref["k8"])
    assert np.array_equal(p.sq.cpu().numpy(), ref["sq"])
    assert np.array_equal(p.sk.cpu().numpy(), ref["sk"])
    vm = p.v_mean.view(torch.int16).cpu().numpy().view(np.uint16)
    assert (vm == ref["v_mean"]).mean() >= 0.9999
    np.testing.assert_allclose(p.v_scale.cpu().numpy(), ref["v_scale"], rtol=1e-6)
    assert (p.v_sf.cpu().numpy() == ref["v_sf"]).mean() >= 0.9999
    assert (p.v_res.cpu().numpy() == ref["v_res"]).mean() >= 0.9999


def _degenerate_inputs(BH=2, N=384, seed=13):
    """Seeded inputs with the degenerate cases the prep has to handle: an
    all-zero Q block (scale 1, codes 0, a uniform softmax row), an all-zero
    permuted K block, a permuted V block that is one constant vector (a zero
    residual), and a V channel that is zero over a whole head (a zero
    per-channel amax)."""
    q, k, v, perm = _prep_inputs(BH, N, seed)
    q, k, v = (t.view(BH, N, 128).clone() for t in (q, k, v))
    q[0, 128:256] = 0
    k[1, perm[1, 0:128].long()] = 0
    v[0, perm[0, 256:384].long()] = v[0, 7].clone()
    v[1, :, 5] = 0
    shape = (1, BH, N, 128)
    return q.view(shape), k.view(shape), v.view(shape), perm


@pytest.mark.parametrize("vmode", [0, 1])
def test_prep_and_attention_on_degenerate_inputs(V, orc, vmode):
    BH, N = 2, 384
    q, k, v, perm = _degenerate_inputs(BH, N)
    ref = orc.prep(*(I.to_u16(t).reshape(BH, N, 128) for t in (q, k, v)), perm.numpy(), vmode=vmode)
    p = V.prep_quant(q.cuda(), k.cuda(), v.cuda(), perm.cuda(), vmode)
    torch.cuda.synchronize()
    for name in ("q8", "sq", "k8", "sk"):
        assert np.array_equal(getattr(p, name).cpu().numpy(), ref[name]), name
    assert p.sq.cpu().numpy()[0, 1] == 1.0 and p.sk.cpu().numpy()[1, 0] == 1.0     # the zero blocks
    assert not p.q8.cpu().numpy()[0, 128:256].any()
    vm = p.v_mean.view(torch.int16).cpu().numpy().view(np.uint16)
    assert (vm == ref["v_mean"]).mean() >= 0.9999
    assert (p.v_res.cpu().numpy() == ref["v_res"]).mean() >= 0.9999
    assert not p.v_res.cpu().numpy()[0, 2].any()                                  # the constant block
    if vmode == 0:
        assert p.v_scale.cpu().numpy()[1, 5] == 1.0                               # the zero channel
        np.testing.assert_allclose(p.v_scale.cpu().numpy(), ref["v_scale"], rtol=1e-6)
    else:
        assert not p.v_sf.cpu().numpy()[0, 2].any()
        assert (p.v_sf.cpu().numpy() == ref["v_sf"]).mean() >= 0.9999
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    O = V.attention(p, 1, BH, N, expcast=(vmode == 0), dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    O_ref = orc.attention(ref, orc.P_EXPCAST if vmode == 0 else orc.P_NVFP4)
    rel, mx = _o_close(O.view(torch.int16).cpu().numpy().view(np.uint16).reshape(BH, N, 128), O_ref)
    assert rel <= REL_L2 and mx <= MAX_ABS, (rel, mx)


# ---------------------------------------------------------------------------
# attention
# ---------------------------------------------------------------------------
def _prepped_both(V, orc, BH, N, seed, vmode=0):
    """Oracle prep of seeded inputs, uploaded as the device operands."""
    q, k, v, perm = _prep_inputs(BH, N, seed)
    ref = orc.prep(*(I.to_u16(t).reshape(BH, N, 128) for t in (q, k, v)), perm.numpy(), vmode=vmode)
    v_sf = None if ref["v_sf"] is None else _dev(ref["v_sf"])
    p = V.Prepared(_dev(ref["q8"]), _dev(ref["sq"]), _dev(ref["k8"]), _dev(ref["sk"]), _dev(ref["v_res"]), v_sf,
                   _dev(ref["v_scale"]), _dev(ref["v_mean"], torch.bfloat16), None, vmode)
    return ref, p


# N spans one block, two, a ragged few (odd), the longest loop without an
# in-loop mean-restore MMA (19 blocks: the epilogue adds them as two MMA groups
# from means buffers 0 and 1), the first in-loop MMA on the last block (20),
# two MMAs (32), a later MMA on the last block (36), and two-group epilogue
# tails that start in means buffer 1 (35 blocks) and 0 again (51)
@pytest.mark.parametrize("expcast", [1, 0])
@pytest.mark.parametrize("BH,N,seed", [(2, 1024, 0), (1, 128, 1), (1, 256, 5), (3, 384, 2), (2, 640, 6), (1, 2304, 3),
                                        (1, 2432, 7), (1, 2560, 8), (2, 4096, 4), (1, 4608, 9), (1, 4480, 10),
                                        (1, 6528, 11)])
def test_attention_parity_on_oracle_operands(V, orc, expcast, BH, N, seed):
    ref, p = _prepped_both(V, orc, BH, N, seed)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    O = V.attention(p, 1, BH, N, expcast=bool(expcast), dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    O_ref = orc.attention(ref, orc.P_EXPCAST if expcast else orc.P_EXP)
    rel, mx = _o_close(O.view(torch.int16).cpu().numpy().view(np.uint16).reshape(BH, N, 128), O_ref)
    assert rel <= REL_L2 and mx <= MAX_ABS, (rel, mx)


# N spans one block, a ragged few, 16 blocks, 17 (a two-group epilogue tail),
# 32 (one in-loop mean-restore MMA), and 35 (a two-group tail from means
# buffer 1)
@pytest.mark.parametrize("BH,N,seed", [(1, 128, 21), (3, 384, 22), (2, 2048, 23), (1, 2176, 24), (2, 4096, 25),
                                        (1, 4480, 26)])
def test_attention_nvfp4_parity_on_oracle_operands(V, orc, BH, N, seed):
    ref, p = _prepped_both(V, orc, BH, N, seed, vmode=V.VCA_V_NVFP4)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    O = V.attention(p, 1, BH, N, expcast=False, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    O_ref = orc.attention(ref, orc.P_NVFP4)
    rel, mx = _o_close(O.view(torch.int16).cpu().numpy().view(np.uint16).reshape(BH, N, 128), O_ref)
    assert rel <= REL_L2 and mx <= MAX_ABS, (rel, mx)


def test_attention_nvfp4_end_to_end_tiny(V, orc):
    """GPU NVFP4 prep + attention against oracle NVFP4 prep + attention."""
    w = I.WORKLOADS["tiny"]
    q, k, v = I.make_qkv(w, seed=13)
    perm = I.random_perm(w.BH, w.N, seed=14)
    ref = orc.prep(*(I.to_u16(t).reshape(w.BH, w.N, 128) for t in (q, k, v)), perm.numpy(), vmode=orc.V_NVFP4)
    O_ref = orc.attention(ref, orc.P_NVFP4)
    p = V.prep_quant(q.cuda(), k.cuda(), v.cuda(), perm.cuda(), V.VCA_V_NVFP4)
    O = V.attention(p, w.B, w.H, w.N, expcast=False)
    torch.cuda.synchronize()
    rel, mx = _o_close(O.view(torch.int16).cpu().numpy().view(np.uint16).reshape(w.BH, w.N, 128), O_ref)
    assert rel <= REL_L2 and mx <= MAX_ABS, (rel, mx)


# The hand-derived two-block examples (worked out in the oracle pins) at the
# kernels' lazy threshold tau = 8: block 1 (max 4.5) does not move the reference
# max set by block 0 (max 1).  P0, P1, P129: decoded P of keys 0, 1, 129;
# rs0, rs1: the blocks' row sums.
WORKED = {
    "expcast": dict(P0=1.0, P1=0.625, P129=2.0, rs0=64.625, rs1=77.0),   # key128 code 84 (12.0)
    "exp": dict(P0=1.0, P1=0.625, P129=2.0, rs0=64.625, rs1=76.0),       # 2^3.5 -> 11.0
    "nvfp4": dict(P0=1.03125, P1=0.6875, P129=1.875, rs0=66.6875, rs1=84.0),
}


@pytest.mark.parametrize("case", sorted(WORKED))
def test_attention_worked_example(V, orc, case):
    """Every query row of the tile is the same row, so all 256 outputs must be
    the hand-derived values (to the last bf16 place: the kernel forms them in
    fp32)."""
    hp = nvfp4_two_block_case(orc) if case == "nvfp4" else two_block_case(orc)
    vmode = V.VCA_V_NVFP4 if case == "nvfp4" else V.VCA_V_E4M3
    v_sf = None if hp["v_sf"] is None else _dev(hp["v_sf"])
    p = V.Prepared(_dev(hp["q8"]), _dev(hp["sq"]), _dev(hp["k8"]), _dev(hp["sk"]), _dev(hp["v_res"]), v_sf,
                   _dev(hp["v_scale"]), _dev(hp["v_mean"], torch.bfloat16), None, vmode)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    O = V.attention(p, 1, 1, 256, expcast=(case == "expcast"), softmax_scale=LN2_F32, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    w = WORKED[case]
    l = w["rs0"] + w["rs1"]
    mean = w["rs0"] * 0.5 + w["rs1"] * -0.25
    want = np.full(128, mean / l)
    want[0] = (w["P1"] * 2.0 + mean) / l
    want[1] = (-w["P0"] + w["P129"] + mean) / l
    got = _f32(O.view(torch.int16).cpu().numpy().view(np.uint16).reshape(256, 128)).astype(np.float64)
    ulp = 2.0 ** (np.floor(np.log2(np.abs(want))) - 7)
    assert np.all(np.abs(got - want[None, :]) <= ulp[None, :]), (got[0, :3], want[:3])


def test_attention_end_to_end_tiny(V, orc):
    """Both chains from the same Q, K, V and permutation: GPU prep + attention
    against oracle prep + attention (the tiny workload, ExpCast on)."""
    w = I.WORKLOADS["tiny"]
    q, k, v = I.make_qkv(w, seed=9)
    perm = I.random_perm(w.BH, w.N, seed=10)
    ref = orc.prep(*(I.to_u16(t).reshape(w.BH, w.N, 128) for t in (q, k, v)), perm.numpy())
    O_ref = orc.attention(ref, orc.P_EXPCAST)
    p = V.prep_quant(q.cuda(), k.cuda(), v.cuda(), perm.cuda(), V.VCA_V_E4M3)
    O = V.attention(p, w.B, w.H, w.N, expcast=True)
    torch.cuda.synchronize()
    rel, mx = _o_close(O.view(torch.int16).cpu().numpy().view(np.uint16).reshape(w.BH, w.N, 128), O_ref)
    assert rel <= REL_L2 and mx <= MAX_ABS, (rel, mx)


def test_attention_whole_path_against_exact_attention(V, orc):
    """group -> prep -> attention on the GPU, and the oracle's own group -> prep
    -> attention, both against exact fp64 attention: the GPU path is as accurate
    as the method itself (the two chains may cluster a few tokens differently)."""
    w = I.WORKLOADS["tiny"]
    q, k, v = I.make_qkv(w, seed=12)
    O, g, p = V.vc_attention(q.cuda(), k.cuda(), v.cuda(), k=w.k, iters=w.iters, expcast=True)
    torch.cuda.synchronize()
    q16, k16, v16 = (I.to_u16(t).reshape(w.BH, w.N, 128) for t in (q, k, v))
    ex = orc.attention_exact(q16, k16, v16)
    _, perm, _, _ = orc.group(v16, w.k, w.iters)
    O_orc = orc.bf16_to_f32(orc.attention(orc.prep(q16, k16, v16, perm), orc.P_EXPCAST)).astype(np.float64)
    got = O.float().cpu().numpy().reshape(w.BH, w.N, 128)
    rel_gpu = np.linalg.norm(got - ex) / np.linalg.norm(ex)
    rel_orc = np.linalg.norm(O_orc - ex) / np.linalg.norm(ex)
    assert rel_gpu <= rel_orc * 1.02 + 1e-3, (rel_gpu, rel_orc)


def test_nvfp4_with_expcast_is_rejected(V):
    p = V.alloc_prep(1, 1, 256, V.VCA_V_NVFP4)
    with pytest.raises(V.VCAError) as e:
        V.attention(p, 1, 1, 256, expcast=True)
    assert e.value.status == V.VCA_ERR_UNSUPPORTED


def test_bounded_wait_reports_timeout_and_context_survives(V, orc):
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    V.vca_selftest_timeout(status, 2_000_000)          # 2 ms on a barrier nothing completes
    torch.cuda.synchronize()
    assert int(status.item()) == V.VCA_ERR_TIMEOUT
    # the context is still usable
    ref, p = _prepped_both(V, orc, 1, 256, 5)
    O = V.attention(p, 1, 1, 256, expcast=True)
    torch.cuda.synchronize()
    rel, mx = _o_close(O.view(torch.int16).cpu().numpy().view(np.uint16).reshape(1, 256, 128),
                       orc.attention(ref, orc.P_EXPCAST))
    assert rel <= REL_L2
