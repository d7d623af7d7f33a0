"""The arithmetic behind the dequantising GEMM's weight decode, checked on the host against the
oracle's format decoders (no GPU).

The kernel turns a word of eight E2M1 codes into four BF16x2 words by placing bits: the byte
permute puts code 2i in bits 0-3 and code 2i+1 in bits 16-19 with zeros around them, a multiply
by 2^6 + 2^12 and a mask move each code's three magnitude bits to the two lowest exponent bits
and the top mantissa bit of its BF16 half and its sign to the sign bit.  The claim: each half is
the code's value times 2^-126 (E2M1's subnormal magnitude 0.5 lands on BF16's subnormal), and
one BF16 multiplication by (E4M3 scale) x 2^118, built from the scale's bits times 2^120 and
then 2^118, gives value x scale x 2^-8 exactly, for every code and every finite scale byte;
for MXFP4, x 2^126 and then x 2^(b - 127) give value x 2^(b - 127) (rounded as the exact product
would be).  Restated here in numpy from the description above, compared with
oracle.e2m1_decode / e4m3_decode / e8m0_decode."""
import math

import numpy as np

import oracle


def bf16_value(bits: int) -> float:
    return float(np.array([bits << 16], dtype=np.uint32).view(np.float32)[0])


def bf16_round(x: float) -> float:
    """x rounded to BF16 (nearest even), via FP32 for values that are FP32-exact."""
    f = np.float32(x)
    assert float(f) == x
    u = int(np.array([f], dtype=np.float32).view(np.uint32)[0])
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return bf16_value(u)


def byte_permute(a: int, b: int, sel: int) -> int:
    """The byte permute's default mode: selector nibble bits 0-2 pick a byte of {b, a}, bit 3
    replicates that byte's top bit."""
    src = [(a >> (8 * i)) & 0xFF for i in range(4)] + [(b >> (8 * i)) & 0xFF for i in range(4)]
    out = 0
    for n in range(4):
        s = (sel >> (4 * n)) & 0xF
        v = src[s & 7]
        if s & 8:
            v = 0xFF if v & 0x80 else 0x00
        out |= v << (8 * n)
    return out


def place_bits(w: int):
    ev = w & 0x0F0F0F0F
    od = (w >> 4) & 0x0F0F0F0F
    halves = []
    for i in range(4):
        r = byte_permute(ev, od, 0x8080 | i | ((4 + i) << 8))
        o = (r * 4160) & 0x81C081C0
        halves += [o & 0xFFFF, o >> 16]
    return halves


def test_bit_placement_is_value_times_2_pow_minus_126():
    rng = np.random.default_rng(0)
    words = [0x76543210, 0xFEDCBA98, 0x88888888, 0x11111111, 0]
    words += [int(x) for x in rng.integers(0, 2 ** 32, 4000, dtype=np.uint64)]
    for w in words:
        got = [bf16_value(h) * 2.0 ** 126 for h in place_bits(w)]
        for k in range(8):
            want = oracle.e2m1_decode((w >> (4 * k)) & 0xF)
            assert got[k] == want and math.copysign(1, got[k]) == math.copysign(1, want), (hex(w), k)


def test_every_code_pair_in_every_position():
    for c0 in range(16):
        for c1 in range(16):
            for pos in range(4):
                w = (c0 | (c1 << 4)) << (8 * pos)
                h = place_bits(w)
                assert bf16_value(h[2 * pos]) * 2.0 ** 126 == oracle.e2m1_decode(c0)
                assert bf16_value(h[2 * pos + 1]) * 2.0 ** 126 == oracle.e2m1_decode(c1)


def test_nvfp4_scale_multiplier_is_exact():
    pow120, pow118 = bf16_value(0x7B80), bf16_value(0x7A80)
    assert pow120 == 2.0 ** 120 and pow118 == 2.0 ** 118
    for b in range(256):
        if (b & 0x7F) == 0x7F:          # NaN encodings never appear as block scales
            continue
        h = ((b & 0x7F) << 4) | ((b & 0x80) << 8)
        s = bf16_value(h) * pow120
        assert s == oracle.e4m3_decode(b) and bf16_round(s) == s
        m = s * pow118
        assert bf16_round(m) == m and abs(m) < 2.0 ** 128
        for c in range(16):
            v = oracle.e2m1_decode(c) * 2.0 ** -126
            prod = v * m
            assert bf16_round(prod) == prod, (b, c)
            assert prod == oracle.e2m1_decode(c) * oracle.e4m3_decode(b) * 2.0 ** -8


def test_mxfp4_two_multiplications_round_as_the_exact_product():
    pow126 = bf16_value(0x7E80)
    assert pow126 == 2.0 ** 126
    for b in range(255):
        h = (b << 7) if b else 0x40
        s = bf16_value(h)
        assert s == oracle.e8m0_decode(b)
        for c in range(16):
            first = bf16_round(oracle.e2m1_decode(c) * 2.0 ** -126 * pow126)
            assert first == oracle.e2m1_decode(c)
            exact = oracle.e2m1_decode(c) * s
            if exact != 0.0 and abs(exact) < 2.0 ** -133:
                continue                 # below BF16's smallest subnormal: both flush alike
            if abs(exact) >= 2.0 ** 128:
                continue                 # beyond BF16's range on both routes
            assert bf16_round(first * s) == bf16_round(exact), (b, c)
