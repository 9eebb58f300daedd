"""Hand-built attention inputs shared by the oracle pins and the GPU worked
examples: one (b,h) whose scores and V values are chosen so that every P value
and every output can be derived by hand (see the tests that use them)."""
import math

import numpy as np

LN2_F32 = float(np.float32(math.log(2.0)))   # softmax scale whose log2(e) multiple is 1.0 in fp32


def two_block_case(orc, third=False):
    """One (b,h), N = 256 (384 with `third`), d = 128: query row 0 is e4m3 1.0 on channel 0; key j
    carries a_j on channel 0, so S_raw = a_j; sq = sk = 1 and the softmax scale
    is fp32(ln 2), making c = 1 and s = S_raw.

    block 0: a = 1.0 (key 0), 0.3125 (key 1), 0 (keys 2..127)
    block 1: a = 4.5 (key 128), 2.0 (key 129), 0 (keys 130..255)
    V: residual scale 1; mean 0.5 in block 0, -0.25 in block 1; residual codes
    2.0 at (key 1, ch 0), -1.0 at (key 0, ch 1), 1.0 at (key 129, ch 1).
    """
    N, d = (384 if third else 256), 128
    code = {v: int(orc.e4m3_encode(np.array([v], np.float32))[0]) for v in (1.0, 0.3125, 4.5, 2.0, -1.0, 12.0)}
    q8 = np.zeros((1, N, d), np.uint8)
    q8[0, :, 0] = code[1.0]
    k8 = np.zeros((1, N, d), np.uint8)
    k8[0, 0, 0], k8[0, 1, 0], k8[0, 128, 0], k8[0, 129, 0] = code[1.0], code[0.3125], code[4.5], code[2.0]
    nb = N // 128
    v_res = np.zeros((1, nb, d, 128), np.uint8)
    v_res[0, 0, 0, 1] = code[2.0]
    v_res[0, 0, 1, 0] = code[-1.0]
    v_res[0, 1, 1, 1] = code[1.0]
    v_mean = np.zeros((1, nb, d), np.uint16)
    v_mean[0, 0, :] = orc.bf16_round(0.5)
    v_mean[0, 1, :] = orc.bf16_round(-0.25)
    if third:                      # block 2: a = 12 at key 256, mean 1.0
        k8[0, 256, 0] = code[12.0]
        v_mean[0, 2, :] = orc.bf16_round(1.0)
    return {"q8": q8, "sq": np.ones((1, nb), np.float32), "k8": k8, "sk": np.ones((1, nb), np.float32),
            "v_res": v_res, "v_sf": None, "v_scale": np.ones((1, d), np.float32), "v_mean": v_mean}


def nvfp4_two_block_case(orc):
    """two_block_case with the V residual in NVFP4: g = 1, every 16-token scale
    E4M3 1.0, E2M1 codes 2.0 at (key 1, ch 0), -1.0 at (key 0, ch 1), 1.0 at
    (key 129, ch 1); means 0.5 and -0.25."""
    p = two_block_case(orc)
    nb, d = 2, 128
    v_res = np.zeros((1, nb, d, 64), np.uint8)
    v_res[0, 0, 0, 0] = 4 << 4      # key 1 (high nibble), ch 0: E2M1 2.0
    v_res[0, 0, 1, 0] = 8 | 2       # key 0 (low nibble), ch 1: E2M1 -1.0
    v_res[0, 1, 1, 0] = 2 << 4      # key 129, ch 1: E2M1 1.0
    return dict(p, v_res=v_res, v_sf=np.full((1, nb, d, 8), 0x38, np.uint8), v_scale=np.ones(1, np.float32))
