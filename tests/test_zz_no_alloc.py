"""vca_prep_quant_noalloc: the prep for callers that cannot give the library any
scratch device memory (a host program that owns all device memory and passes an
operator only its tensors, or a code path that must not call cudaMalloc).  It
keeps its scratch in a buffer built into the library, so its outputs must equal
vca_prep_quant's, call after call, whatever an earlier call left in that buffer.

This file is collected last so that a run stopping at the first failure has
already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

from bit_attention_video_smooth_gb300 import inputs as I

pytestmark = pytest.mark.gpu


def _outputs(p):
    outs = [p.q8, p.sq, p.k8, p.sk, p.v_res, p.v_scale, p.v_mean.view(torch.int16)]
    if p.v_sf is not None:
        outs.append(p.v_sf)
    return [t.cpu().numpy() for t in outs]


@pytest.mark.parametrize("vmode", [0, 1])
def test_noalloc_prep_matches_workspace_prep_on_consecutive_calls(V, vmode):
    for call, (BH, N, seed) in enumerate([(3, 1152, 21), (2, 640, 22)]):
        w = I.with_n(I.WORKLOADS["tiny"], N, H=BH)
        q, k, v = (t.cuda() for t in I.make_qkv(w, seed=seed))
        perm = I.random_perm(BH, N, seed=seed + 1).cuda()
        ref = V.prep_quant(q, k, v, perm, vmode)
        got = V.alloc_prep(1, BH, N, vmode)
        V.vca_prep_quant_noalloc(q, k, v, perm, vmode, got.q8, got.sq, got.k8, got.sk, got.v_res, got.v_sf,
                                 got.v_scale, got.v_mean)
        torch.cuda.synchronize()
        for a, b in zip(_outputs(got), _outputs(ref)):
            assert np.array_equal(a, b), f"call {call}: outputs differ from vca_prep_quant"


def test_noalloc_prep_rejects_problems_beyond_its_scratch(V):
    lib = ctypes.CDLL(V.LIB_PATH)
    fn = lib.vca_prep_quant_noalloc
    P = ctypes.c_void_p
    # Q, K, V, perm; B, H, N, d, vmode; q8, sq, k8, sk, v_res, v_sf, v_scale, v_mean; stream
    fn.argtypes = [P] * 4 + [ctypes.c_int] * 5 + [P] * 8 + [P]
    fake = P(0x10000)   # aligned, never dereferenced: the size check comes first
    # B=1, H=64, N=65,536: 64 * 512 blocks + 64 heads = 32,832 units of 512 bytes, above 16 MiB
    st = fn(fake, fake, fake, fake, 1, 64, 65536, 128, 0, *([fake] * 8), None)
    assert st == V.VCA_ERR_WORKSPACE
    assert V.vca_workspace_bytes(V.VCA_OP_PREP, 1, 64, 65536) > (16 << 20)


def test_noalloc_prep_at_the_size_limit(V):
    """B*H*(N/128) + B*H = 32,768 exactly: the prep workspace fills the
    built-in scratch to the last byte, and the outputs still equal
    vca_prep_quant's."""
    B, H, N = 1, 64, 511 * 128
    assert V.vca_workspace_bytes(V.VCA_OP_PREP, B, H, N) == (16 << 20)
    w = I.with_n(I.WORKLOADS["wan"], N, H=H, B=B)
    q, k, v = I.make_qkv(w, seed=31, device="cuda")
    perm = I.random_perm(B * H, N, seed=32).cuda()
    ref = V.prep_quant(q, k, v, perm, 0)
    got = V.alloc_prep(B, H, N, 0)
    V.vca_prep_quant_noalloc(q, k, v, perm, 0, got.q8, got.sq, got.k8, got.sk, got.v_res, got.v_sf,
                             got.v_scale, got.v_mean)
    torch.cuda.synchronize()
    for a, b in zip(_outputs(got), _outputs(ref)):
        assert np.array_equal(a, b), "outputs at the size limit differ from vca_prep_quant"
