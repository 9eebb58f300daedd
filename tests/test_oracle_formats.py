"""Pins for the oracle's number formats: E4M3, E2M1, bf16.

The oracle's encoders and decoders are checked against (a) the values the pages
fix (an E4M3 byte read as an integer is about 8 log2 v + 56: code 56 is 1.0,
code 8 is the smallest normal 2^-6, code 126 is 448), (b) PyTorch's own CPU
casts to float8_e4m3fn and bfloat16 (library routines), and (c) enumeration of
the E2M1 grid and its ties.
"""
import json
import math
import os

import numpy as np
import torch

GOLD = os.path.join(os.path.dirname(__file__), "golden", "pages_constants.json")


def test_e4m3_decode_matches_torch_and_pages(orc):
    codes = np.arange(256, dtype=np.uint8)
    ours = orc.e4m3_decode(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    fin = np.isfinite(ref)
    assert np.array_equal(np.isfinite(ours), fin)
    assert np.array_equal(ours[fin], ref[fin])
    # signs of zero
    assert math.copysign(1.0, ours[0x80]) == -1.0
    g = json.load(open(GOLD))["e4m3_code_of_value"]
    # byte ~= 8 log2 v + 56: exact at powers of two in the normal range
    for e in range(-6, 9):
        code = g["slope"] * e + g["offset"]
        assert ours[code] == 2.0 ** e
    assert ours[8] == 2.0 ** -6 and ours[126] == 448.0 and np.isnan(ours[127])


def test_e4m3_encode_roundtrip_and_torch_cast(orc):
    codes = np.arange(256, dtype=np.uint8)
    vals = orc.e4m3_decode(codes)
    fin = np.isfinite(vals)
    assert np.array_equal(orc.e4m3_encode(vals[fin].astype(np.float32)), codes[fin])
    # random fp32 values inside the finite range: identical to torch's RNE cast
    rng = np.random.default_rng(1)
    x = np.concatenate([
        rng.standard_normal(200_000) * 50,
        rng.standard_normal(200_000) * 1e-3,          # subnormal range
        (rng.random(100_000) * 2 - 1) * 447.9,
    ]).astype(np.float32)
    ours = orc.e4m3_encode(x)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)


def test_e4m3_ties_to_even_and_saturation(orc):
    vals = orc.e4m3_decode(np.arange(0, 126, dtype=np.uint8))
    mids = ((vals[:-1] + vals[1:]) / 2).astype(np.float32)   # exact in fp32
    enc = orc.e4m3_encode(mids)
    lo, hi = np.arange(0, 125), np.arange(1, 126)
    expect = np.where(lo % 2 == 0, lo, hi)                   # even mantissa wins
    assert np.array_equal(enc, expect.astype(np.uint8))
    big = np.array([448.0, 449.0, 463.9, 464.0, 500.0, 1e30, np.inf], np.float32)
    assert np.all(orc.e4m3_encode(big) == 126)
    assert np.all(orc.e4m3_encode(-big) == 0xFE)
    assert orc.e4m3_encode(np.array([np.nan], np.float32))[0] == 0x7F
    tiny = np.array([2.0 ** -11, -(2.0 ** -11), 2.0 ** -10 * 1.0001], np.float32)
    assert list(orc.e4m3_encode(tiny)) == [0x00, 0x80, 0x01]


def test_e4m3_exhaustive_against_torch(orc):
    # every non-negative fp32 bit pattern below 448 (the finite range, where
    # torch's cast does not saturate), in chunks: identical bytes
    end = int(np.array([448.0], np.float32).view(np.uint32)[0])
    step = 1 << 26
    for start in range(0, end + 1, step):
        cnt = min(step, end + 1 - start)
        ours = orc.e4m3_encode_bits(start, cnt)
        x = torch.arange(start, start + cnt, dtype=torch.int64).to(torch.int32).view(torch.float32)
        ref = x.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        assert np.array_equal(ours, ref), hex(start)
    # negative patterns on a stride: encode(-x) == encode(x) | 0x80
    u = np.arange(0, 0x7F800000, 7919, dtype=np.uint32)
    pos = orc.e4m3_encode(u.view(np.float32))
    neg = orc.e4m3_encode((u | np.uint32(0x80000000)).view(np.float32))
    assert np.array_equal(neg, pos | 0x80)


def test_e2m1_grid_and_ties(orc):
    dec = orc.e2m1_decode(np.arange(16))
    assert list(dec[:8]) == [0, 0.5, 1, 1.5, 2, 3, 4, 6]
    assert list(dec[8:]) == [-0.0, -0.5, -1, -1.5, -2, -3, -4, -6]
    ties = {0.25: 0.0, 0.75: 1.0, 1.25: 1.0, 1.75: 2.0, 2.5: 2.0, 3.5: 4.0, 5.0: 4.0}
    for x, y in ties.items():
        assert dec[orc.e2m1_encode(np.array([x], np.float32))[0]] == y
        assert dec[orc.e2m1_encode(np.array([-x], np.float32))[0]] == -y
    assert dec[orc.e2m1_encode(np.array([7.0, 100.0], np.float32))].tolist() == [6.0, 6.0]
    # brute force: the encoder picks a nearest grid value for random inputs
    rng = np.random.default_rng(2)
    x = (rng.random(20000) * 14 - 7).astype(np.float32)
    got = dec[orc.e2m1_encode(x)]
    grid = np.array([-6, -4, -3, -2, -1.5, -1, -0.5, 0, 0.5, 1, 1.5, 2, 3, 4, 6])
    best = np.abs(np.clip(x, -6, 6)[:, None] - grid[None, :]).min(axis=1)
    assert np.allclose(np.abs(np.clip(x, -6, 6) - got), best)


def test_bf16_round_matches_torch(orc):
    rng = np.random.default_rng(3)
    x = np.concatenate([rng.standard_normal(3000) * 10.0 ** rng.integers(-30, 30, 3000),
                        rng.standard_normal(1000)]).astype(np.float64)
    ours = np.array([orc.bf16_round(v) for v in x.astype(np.float32)], np.uint16)
    ref = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
