"""Pins for the oracle's scalar codecs (E2M1 values, E4M3 block scales, BF16 output rounding).

Each codec is checked against something other than itself: hand-worked tables from the format
definition (tests/golden), brute-force nearest-value search over every code, and PyTorch's own
float8_e4m3fn / bfloat16 casts (library routines).
"""
import math
import struct

import numpy as np
import pytest
import torch

from conftest import read_table


def _f32(v):
    return struct.unpack("<f", struct.pack("<f", v))[0]


def test_e2m1_decode_table(orc):
    rows = read_table("e2m1_table.txt")
    assert len(rows) == 16
    for code, val in rows:
        got = orc.e2m1_decode(int(code, 16))
        want = float(val)
        assert got == want and math.copysign(1, got) == math.copysign(1, want), (code, got, want)


def test_e2m1_encode_hand_points(orc):
    for inp, code in read_table("e2m1_encode_points.txt"):
        assert orc.e2m1_encode(float(inp)) == int(code, 16), inp


def _e2m1_bruteforce(q):
    """Nearest of the 8 magnitudes by distance; on a tie the even code; sign bit kept."""
    mags = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    a = abs(q)
    best = None
    for c, m in enumerate(mags):
        d = abs(a - m)
        if best is None or d < best[0] or (d == best[0] and c % 2 == 0):
            best = (d, c)
    return best[1] | (8 if math.copysign(1.0, q) < 0 else 0)


def test_e2m1_encode_bruteforce_sweep(orc):
    rng = np.random.default_rng(1)
    pts = list(np.linspace(-7.5, 7.5, 6001)) + list(rng.uniform(-8, 8, 4000))
    mids = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]
    for m in mids:
        for d in (0.0, 1e-6, -1e-6):
            pts += [m + d, -(m + d)]
    for q in pts:
        q = _f32(float(q))
        assert orc.e2m1_encode(q) == _e2m1_bruteforce(q), q


def _e4m3_closed_form(c):
    s = -1.0 if c & 0x80 else 1.0
    e, m = (c >> 3) & 15, c & 7
    if e == 15 and m == 7:
        return float("nan")
    if e == 0:
        return s * m / 8.0 * 2.0 ** -6
    return s * (1 + m / 8.0) * 2.0 ** (e - 7)


def test_e4m3_decode_hand_points(orc):
    for code, val in read_table("e4m3_points.txt"):
        got = orc.e4m3_decode(int(code, 16))
        assert got == float(val) and math.copysign(1, got) == math.copysign(1, float(val)), code


def test_e4m3_decode_all_codes_vs_torch(orc):
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float32).tolist()
    for c in range(256):
        got = orc.e4m3_decode(c)
        cf = _e4m3_closed_form(c)
        if math.isnan(ref[c]):
            assert math.isnan(got) and math.isnan(cf) and (c & 0x7F) == 0x7F
        else:
            assert got == ref[c] == cf, c


def _e4m3_bruteforce(v):
    """Nearest finite E4M3 value by distance, ties to the even code; saturate to +-448."""
    if math.isnan(v):
        return 0x7F
    s = 0x80 if math.copysign(1.0, v) < 0 else 0
    a = abs(v)
    best = None
    for c in range(0x7F):  # 0x00..0x7E are the finite non-negative codes
        d = abs(a - _e4m3_closed_form(c))
        if best is None or d < best[0] or (d == best[0] and c % 2 == 0):
            best = (d, c)
    return s | best[1]


def test_e4m3_encode_bruteforce(orc):
    pos = [_e4m3_closed_form(c) for c in range(0x7F)]
    pts = set(pos)
    for a, b in zip(pos[:-1], pos[1:]):   # every midpoint and its neighbours
        mid = (a + b) / 2
        pts.update([mid, np.nextafter(np.float32(mid), np.float32(0)).item(),
                    np.nextafter(np.float32(mid), np.float32(1e9)).item()])
    pts.update([448.0, 449.0, 463.9, 464.0, 500.0, 1e6, 1e-12, 2.0 ** -10, 2.0 ** -11, float("inf")])
    rng = np.random.default_rng(2)
    pts.update(np.exp(rng.uniform(-14, 7, 3000)).astype(np.float32).tolist())
    for v in sorted(pts):
        v = _f32(v)
        for sv in (v, -v):
            want = 0x7E | (0x80 if sv < 0 else 0) if math.isinf(sv) else _e4m3_bruteforce(sv)
            assert orc.e4m3_encode(sv) == want, sv


def test_e4m3_encode_vs_torch_in_range(orc):
    rng = np.random.default_rng(3)
    v = np.concatenate([np.exp(rng.uniform(-13, 6.0, 20000)), rng.uniform(0, 440, 5000)]).astype(np.float32)
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    for x, r in zip(v.tolist(), ref.tolist()):
        assert orc.e4m3_encode(x) == r, x


def test_bf16_round_vs_torch(orc):
    rng = np.random.default_rng(4)
    v = np.concatenate([rng.normal(0, 1, 20000), rng.normal(0, 1e-3, 2000), rng.normal(0, 1e5, 2000)])
    v = v.astype(np.float32)
    # include exact ties (the 16 low bits 0x8000)
    ties = (np.arange(1000, dtype=np.uint32) << 16 | 0x8000).view(np.float32)
    v = np.concatenate([v, ties, -ties])
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    for x, r in zip(v.tolist(), ref.tolist()):
        assert orc.f32_to_bf16_bits(x) == r
