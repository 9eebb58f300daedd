"""The Python binding's buffer checks, on a machine without a GPU.

The C ABI takes plain pointers and cannot see how large the buffers behind
them are, so the binding checks every tensor's byte size against the problem
size before anything is launched, then that all of them sit on one CUDA device.
Here host tensors stand in for device ones: a call whose sizes are right fails
only on the device check, one with a short or non-contiguous buffer fails on
the size check and names the buffer.  The sized cases are built the way the
GPU tests, the smoke run and bench.py build theirs (the binding's own
allocators, oracle operands, the hand-built worked examples), so a size rule
that rejected a valid call would show here first.
"""
import numpy as np
import pytest
import torch

from bit_attention_video_smooth_gb300 import inputs as I

from cases import nvfp4_two_block_case, two_block_case


@pytest.fixture(scope="module")
def V():
    from bit_attention_video_smooth_gb300 import build
    build.build()
    from bit_attention_video_smooth_gb300 import vca
    return vca


NOT_CUDA = "is not a CUDA tensor"


def _host(a, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a))
    return t.view(dtype) if dtype is not None else t


def _prepared(V, ref, vmode):
    v_sf = None if ref["v_sf"] is None else _host(ref["v_sf"])
    return V.Prepared(_host(ref["q8"]), _host(ref["sq"]), _host(ref["k8"]), _host(ref["sk"]), _host(ref["v_res"]),
                      v_sf, _host(ref["v_scale"]), _host(ref["v_mean"], torch.bfloat16), None, vmode)


@pytest.mark.parametrize("vmode", [0, 1])
def test_allocated_buffers_pass_the_size_checks(V, vmode):
    w = I.WORKLOADS["tiny"]
    q, k, v = I.make_qkv(w, seed=3)
    perm = I.random_perm(w.BH, w.N, seed=4).view(w.B, w.H, w.N)
    with pytest.raises(ValueError, match=NOT_CUDA):
        V.group(v, w.k, w.iters)
    with pytest.raises(ValueError, match=NOT_CUDA):
        V.prep_quant(q, k, v, perm, vmode)
    with pytest.raises(ValueError, match=NOT_CUDA):
        V.prep_quant(q, k, v, perm, vmode, qk_hadamard=True)
    p = V.alloc_prep(w.B, w.H, w.N, vmode, device="cpu")
    with pytest.raises(ValueError, match=NOT_CUDA):
        V.vca_prep_quant_noalloc(q, k, v, perm, vmode, p.q8, p.sq, p.k8, p.sk, p.v_res, p.v_sf, p.v_scale, p.v_mean)
    status = torch.zeros(1, dtype=torch.int32)
    with pytest.raises(ValueError, match=NOT_CUDA):
        V.attention(p, w.B, w.H, w.N, expcast=(vmode == 0), dev_status=status)


@pytest.mark.parametrize("vmode,BH,N", [(0, 2, 256), (0, 1, 2432), (1, 3, 384)])
def test_oracle_operands_pass_the_size_checks(V, orc, vmode, BH, N):
    q, k, v = I.make_qkv(I.with_n(I.WORKLOADS["tiny"], N, H=BH), seed=5)
    perm = I.random_perm(BH, N, seed=6)
    ref = orc.prep(*(I.to_u16(t).reshape(BH, N, 128) for t in (q, k, v)), perm.numpy(), vmode=vmode)
    with pytest.raises(ValueError, match=NOT_CUDA):
        V.attention(_prepared(V, ref, vmode), 1, BH, N, expcast=(vmode == 0))


@pytest.mark.parametrize("case", ["e4m3", "nvfp4"])
def test_worked_examples_pass_the_size_checks(V, orc, case):
    hp = nvfp4_two_block_case(orc) if case == "nvfp4" else two_block_case(orc)
    vmode = 1 if case == "nvfp4" else 0
    with pytest.raises(ValueError, match=NOT_CUDA):
        V.attention(_prepared(V, hp, vmode), 1, 1, 256, expcast=False)


def test_short_or_strided_buffers_are_named(V):
    B, H, N = 1, 2, 256
    p = V.alloc_prep(B, H, N, 0, device="cpu")
    short_o = torch.empty((B, H, N - 1, 128), dtype=torch.bfloat16)
    with pytest.raises(ValueError, match=r"O holds \d+ bytes, 131072 needed"):
        V.attention(p, B, H, N, out=short_o)
    # attention at twice the sequence the buffers were sized for
    with pytest.raises(ValueError, match="q8 holds"):
        V.attention(p, B, H, 2 * N)
    # a NVFP4 call with E4M3-sized scales
    p4 = V.alloc_prep(B, H, N, 1, device="cpu")
    p4.v_sf = torch.empty(10, dtype=torch.uint8)
    with pytest.raises(ValueError, match="v_sf holds 10 bytes"):
        V.attention(p4, B, H, N, expcast=False)
    strided = torch.empty((B, H, N, 256), dtype=torch.bfloat16)[..., :128]
    with pytest.raises(ValueError, match="O must be contiguous"):
        V.attention(p, B, H, N, out=strided)
    q = torch.zeros((B, H, N, 128), dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="perm holds"):
        V.prep_quant(q, q, q, torch.zeros(N, dtype=torch.int32))
    g = V.alloc_group(B, H, N, 8, device="cpu")
    with pytest.raises(ValueError, match="counts holds 64 bytes, 128 needed"):
        V.vca_group(q, 16, 4, g.labels, g.perm, g.counts, g.centroids, g.ws)   # sized for k = 8
    with pytest.raises(ValueError, match="dev_status holds 0 bytes"):
        V.vca_selftest_timeout(torch.empty(0, dtype=torch.int32), 1000)


def test_test_entry_points_check_sizes(V):
    s = torch.zeros(1000, dtype=torch.float32)
    with pytest.raises(ValueError, match=NOT_CUDA):
        V.vca_expcast_codes(s, torch.ones_like(s), s.clone(), torch.empty(1000, dtype=torch.uint8))
    with pytest.raises(ValueError, match="m holds 3996 bytes"):
        V.vca_expcast_codes(s, torch.ones_like(s), s[:999].clone(), torch.empty(1000, dtype=torch.uint8))
    with pytest.raises(ValueError, match=NOT_CUDA):
        V.vca_e4m3_encode_bits(0, 4096, torch.empty(4096, dtype=torch.uint8))
    with pytest.raises(ValueError, match="out holds 4095 bytes"):
        V.vca_e4m3_encode_bits(0, 4096, torch.empty(4095, dtype=torch.uint8))
