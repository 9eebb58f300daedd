"""The arithmetic behind the attention kernel's ExpCast codes, checked on the
CPU (the GPU tests compare the device codes with the oracle bit for bit on
millions of inputs; these checks cover every value the steps can see).

Fast path (every code at most 126; nine instructions per four codes): the
kernel forms the oracle's t = fma(s, 8c, 55.65 - 8m) in fp32 (packed, two at a
time), multiplies it by 2^-149, the smallest subnormal (packed): the exact
product rounds, nearest even, to a multiple of 2^-149, so the product's bit
pattern is rne(t) for 0 <= t < 2^23 and has the sign bit set for t < 0; then
`cvt.pack.sat.u8.s32.b32` (d = (c & 0xffff) << 16 | sat(a) << 8 | sat(b), each
operand clamped to [0, 255] as a signed integer; the layout measured on the
device) packs two such patterns per instruction, and the flush below zeroes
codes 1..7.

Clipped form (taken only for |m| >= 2^22): per element the kernel forms
u = sat(fma(s, 8c/256, (55.65 - 8m)/256)), which
is t/256 for the oracle's t = fma(s, 8c, 55.65 - 8m) (a power-of-two scaling
changes no rounding), clamped to [0, 1].  It then
  1. adds 1.5 * 2^15 in fp32: the sum's unit in the last place is 2^-8, so its
     bit pattern is 0x47400000 + rne(256 u) -- the code in the low byte;
  2. packs four such patterns into one word: a byte permute (PTX `prmt`,
     selector 0x1140) for codes 0 and 1, and 32-bit multiply-adds by 2^16 and
     2^24 for codes 2 and 3 (the pattern's high half vanishes modulo 2^32);
  3. zeroes the codes 1..7: w + 0x78787878 sets a byte's top bit exactly when
     its code is >= 8 (no carry crosses bytes for codes <= 126), and a byte
     permute with sign replication (selector 0xBA98) turns those bits into a
     byte mask.
The fast path has no clip at 126; that is safe when fp32(s c) <= fp32(m + 8)
and |m| < 2^22 (the lazy reference max is never more than 8 below the block
max), because t then stays below 126.5.
"""
import numpy as np

MAGIC = np.float32(49152.0)                 # 1.5 * 2^15
M32 = 0xFFFFFFFF


def prmt(a, b, sel):
    """PTX prmt.b32 (default mode): byte i of the result is byte (sel nibble i &
    7) of the 8-byte value {b, a}; nibble bit 3 replicates that byte's top bit."""
    src = (int(b) << 32) | int(a)
    out = 0
    for i in range(4):
        nib = (sel >> (4 * i)) & 0xF
        byte = (src >> (8 * (nib & 7))) & 0xFF
        if nib & 8:
            byte = 0xFF if byte & 0x80 else 0x00
        out |= byte << (8 * i)
    return out


def pattern(code):
    """Bit pattern of fp32(code / 256 + 1.5 * 2^15)."""
    return int((np.float32(code / 256.0) + MAGIC).view(np.uint32))


def pack_and_flush(codes):
    x = [pattern(c) for c in codes]
    w = prmt(x[0], x[1], 0x1140)
    w = (w + x[2] * 65536) & M32                  # mad.lo.u32 w, x2, 2^16, w
    w = (w + x[3] * 16777216) & M32               # mad.lo.u32 w, x3, 2^24, w
    t = (w * 1 + 0x78787878) & M32                # mad.lo.u32 t, w, one, 0x78787878
    return w & prmt(t, 0, 0xBA98)


def flushed_word(codes):
    return sum((c if c >= 8 else 0) << (8 * i) for i, c in enumerate(codes))


def test_magic_add_puts_the_rounded_code_in_the_low_byte():
    """Every fp32 u in [2^-10, 127/256): the sum's pattern is 0x47400000 plus
    rne(256 u); below 2^-10 the code is 0."""
    for e in range(-10, -1):
        base = (e + 127) << 23
        u = np.arange(base, base + (1 << 23), dtype=np.uint32).view(np.float32)
        u = u[u < np.float32(127.0 / 256.0)]
        bits = (u + MAGIC).view(np.uint32)
        want = np.rint(u.astype(np.float64) * 256.0).astype(np.uint32)   # half to even
        assert np.array_equal(bits, np.uint32(0x47400000) + want), e
    tiny = np.array([0.0, 2.0 ** -30, 2.0 ** -11, np.nextafter(np.float32(2.0 ** -9), np.float32(0))], np.float32)
    assert np.all((tiny + MAGIC).view(np.uint32) == 0x47400000)
    # exactly half a code rounds to even
    assert pattern(0.5) == 0x47400000 and pattern(1.5) == 0x47400002 and pattern(2.5) == 0x47400002


def test_packing_and_flush_of_every_code_in_every_lane():
    rng = np.random.default_rng(0)
    for lane in range(4):
        for code in range(127):
            codes = [int(x) for x in rng.integers(0, 127, 4)]
            codes[lane] = code
            assert pack_and_flush(codes) == flushed_word(codes), (lane, codes)
    for _ in range(20000):
        codes = [int(x) for x in rng.integers(0, 127, 4)]
        assert pack_and_flush(codes) == flushed_word(codes), codes
    # the byte-permute model itself on documented cases
    assert prmt(0x44332211, 0x88776655, 0x3210) == 0x44332211
    assert prmt(0x44332211, 0x88776655, 0x7654) == 0x88776655
    assert prmt(0x00800180, 0, 0xBA98) == 0x00FF00FF


TINY = np.float32(2.0 ** -149)


def cvt_pack_sat_u8(a, b, c):
    """cvt.pack.sat.u8.s32.b32 d, a, b, c: a and b as signed 32-bit integers
    clamped to [0, 255], d = (c & 0xffff) << 16 | sat(a) << 8 | sat(b)."""
    def sat(v):
        v = int(v) & M32
        v = v - (1 << 32) if v & 0x80000000 else v
        return min(max(v, 0), 255)
    return ((int(c) & 0xFFFF) << 16) | (sat(a) << 8) | sat(b)


def fast_codes(t4):
    """The fast path from four fp32 t values: patterns of t * 2^-149, two packs,
    the flush."""
    y = [int((np.float32(t) * TINY).view(np.uint32)) for t in t4]
    hi = cvt_pack_sat_u8(y[3], y[2], 0)
    w = cvt_pack_sat_u8(y[1], y[0], hi)
    tt = (w * 1 + 0x78787878) & M32
    return w & prmt(tt, 0, 0xBA98)


def test_subnormal_multiply_rounds_t_to_the_code():
    """Every fp32 t in [2^-10, 127): the bit pattern of fp32(t * 2^-149) is
    rne(t); every t in (-2^12, 0) gives a pattern with the sign bit set (a
    negative integer, which the pack clamps to 0); so does -0."""
    for e in range(-10, 7):
        base = (e + 127) << 23
        t = np.arange(base, base + (1 << 23), dtype=np.uint32).view(np.float32)
        t = t[t < np.float32(127.0)]
        bits = (t * TINY).view(np.uint32)
        want = np.rint(t.astype(np.float64)).astype(np.uint32)   # half to even
        assert np.array_equal(bits, want), e
    neg = -np.arange(1, 1 << 20, dtype=np.float32) / np.float32(256.0)
    assert np.all(((neg * TINY).view(np.uint32) & 0x80000000) != 0)
    assert (np.float32(-0.0) * TINY).view(np.uint32) == 0x80000000
    # far below: the product is a negative normal or subnormal, sign bit set all the same
    far = -np.float32(2.0) ** np.arange(12, 127, dtype=np.float32)
    assert np.all(((far * TINY).view(np.uint32) & 0x80000000) != 0)
    # halves go to the even neighbour
    for t, r in ((0.5, 0), (1.5, 2), (2.5, 2), (7.5, 8), (125.5, 126), (33.5, 34), (34.5, 34)):
        assert int((np.float32(t) * TINY).view(np.uint32)) == r


def test_fast_path_pack_and_flush_of_every_code_in_every_lane():
    """Four t values -> the word of their flushed codes, for every code in every
    lane, negative t (code 0) included."""
    rng = np.random.default_rng(2)
    def word(ts):
        codes = [0 if t < 0 else int(np.rint(np.float64(t))) for t in ts]
        return flushed_word(codes)
    for lane in range(4):
        for code in range(127):
            ts = [float(x) for x in rng.uniform(-40, 126.4, 4).astype(np.float32)]
            ts[lane] = float(np.float32(code + rng.uniform(-0.49, 0.49)))
            assert fast_codes(ts) == word(ts), (lane, ts)
    for _ in range(20000):
        ts = [float(x) for x in rng.uniform(-300, 126.4, 4).astype(np.float32)]
        assert fast_codes(ts) == word(ts), ts
    # the pack's measured layout and saturation
    assert cvt_pack_sat_u8(1, 2, 0) == 0x0102
    assert cvt_pack_sat_u8(300, -7, 0) == 0xFF00
    assert cvt_pack_sat_u8(7, 8, 0xAABBCCDD) == 0xCCDD0708
    assert cvt_pack_sat_u8(0xFFFFFFFF, 128, 0xABCD) == 0xABCD0080


def _fma_f32(a, b, c):
    """RN32(a * b + c) for fp32 inputs: the product is exact in fp64; the sum is
    rounded once through an exact two-sum."""
    a, b, c = (np.asarray(v, np.float32).astype(np.float64) for v in (a, b, c))
    p = a * b
    t = p + c
    bp = t - p
    err = (p - (t - bp)) + (c - bp)
    f = t.astype(np.float32)
    ff = f.astype(np.float64)
    g = np.where(t > ff, np.nextafter(f, np.float32(np.inf)), np.nextafter(f, np.float32(-np.inf)))
    gf = g.astype(np.float64)
    mid = (t != ff) & (ff + gf == 2.0 * t)
    hi = np.maximum(ff, gf).astype(np.float32)
    lo = np.minimum(ff, gf).astype(np.float32)
    return np.where(mid & (err > 0), hi, np.where(mid & (err < 0), lo, f))


def test_codes_stay_below_the_clip_on_the_fast_path():
    """Adversarial draws: m anywhere below 2^22 in magnitude, scores at or just
    under the largest value the lazy rule allows, fp32(s c) <= fp32(m + 8)."""
    rng = np.random.default_rng(1)
    n = 400000
    mag = 2.0 ** rng.uniform(-4, 22, n)
    m = (np.sign(rng.uniform(-1, 1, n)) * mag).astype(np.float32)
    m = np.clip(m, np.float32(-4194303.5), np.float32(4194303.5))
    c = (2.0 ** rng.uniform(-12, 2, n)).astype(np.float32)
    lim = (m + np.float32(8.0)).astype(np.float32)
    s = (lim.astype(np.float64) / c.astype(np.float64)).astype(np.float32)
    # the largest s with fp32(s c) <= lim: step s down while the product exceeds it
    for _ in range(4):
        over = (s * c) > lim
        s = np.where(over, np.nextafter(s, np.float32(-np.inf) * np.sign(c)), s)
    assert np.all((s * c) <= lim)
    bias = (np.float32(55.65) - np.float32(8.0) * m).astype(np.float32)
    t = _fma_f32(s, np.float32(8.0) * c, bias)
    assert np.all(t < 126.5), float(t.max())
    assert float(t.max()) <= 55.65 + 68.0         # the bound the kernel states
