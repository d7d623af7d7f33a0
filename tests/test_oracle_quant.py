"""Pins for the oracle's NVFP4 quantiser: a hand-worked row, round-trip error bounds that the
format fixes, exactness on inputs that already lie on the grid, and the zero-block rule."""
import numpy as np
import torch

from conftest import read_kv

E2M1_MAGS = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], np.float64)


def test_hand_worked_row(orc):
    kv = read_kv("nvfp4_row_example.txt")
    x = torch.tensor([float(v) for v in kv["x"]]).to(torch.bfloat16).reshape(1, -1)
    codes, sf, ts, st = orc.quantize_bf16(x)
    assert st == 0
    assert ts == float(kv["ts"][0])
    assert sf.tobytes().hex() == "".join(kv["sf"])
    assert codes.tobytes().hex() == "".join(kv["codes"])


def _gap(q):
    """Spacing of the E2M1 grid around |q| (0.5 below 2, 1 below 4, 2 up to 6)."""
    return np.where(q < 2, 0.5, np.where(q < 4, 1.0, 2.0))


def test_round_trip_bounds(orc):
    g = torch.Generator().manual_seed(5)
    for scale, rows, cols in ((1.0, 64, 256), (0.02, 32, 512), (300.0, 8, 2048), (1e-3, 16, 64)):
        x = (torch.randn(rows, cols, generator=g) * scale)
        x[0, :16] = 0.0                       # a zero block
        x[1, 16:32] *= 1e-4                   # a tiny block
        xb = x.to(torch.bfloat16)
        codes, sf, ts, st = orc.quantize_bf16(xb)
        assert st == 0
        xf = xb.float().numpy().astype(np.float64)
        amax = np.abs(xf).max()
        assert ts == np.float32(np.float32(amax) / np.float32(2688.0))
        xhat = orc.dequantize(codes, sf, ts).astype(np.float64)
        S = np.array([orc.e4m3_decode(int(s)) for s in sf.reshape(-1)]).reshape(sf.shape) * ts
        S = np.repeat(S, 16, axis=1)
        err = np.abs(xf - xhat)
        bam = np.repeat(np.abs(xf).reshape(rows, -1, 16).max(-1), 16, axis=1)
        q = np.abs(xf) / np.where(S > 0, S, 1)
        inside = (q <= 6.0) & (S > 0)
        # on the grid's range: half a grid step (plus FP32 slack of the scale product)
        bound = 0.5 * _gap(np.minimum(q, 6.0)) * S * (1 + 2e-6) + 1e-30
        assert np.all(err[inside] <= bound[inside])
        # saturated elements: the block maximum is off by at most half an E4M3 step (2^-4 rel.)
        sat = (q > 6.0) & (S > 0)
        assert np.all(err[sat] <= bam[sat] * (2.0 ** -4) * 1.0001)
        # zero blocks decode to exact zeros
        assert np.all(sf[0, 0] == 0) and np.all(codes[0, :8] == 0)
        # the block maximum is always reproduced within 2^-4 relative (E4M3 half-step)
        blk = np.argmax(np.abs(xf).reshape(rows, -1, 16), axis=-1)
        for r in range(rows):
            for b in range(cols // 16):
                i = b * 16 + blk[r, b]
                if bam[r, i] > 0 and S[r, i] > 0:
                    assert abs(xf[r, i] - xhat[r, i]) <= bam[r, i] * 2.0 ** -4 * 1.0001


def test_exact_on_grid(orc):
    """x = e2m1 * 2^a * ts with power-of-two block scales: the codes come back exactly."""
    rng = np.random.default_rng(6)
    rows, cols = 8, 128
    codes_in = rng.integers(0, 16, size=(rows, cols)).astype(np.uint8)
    # each block gets a power-of-two scale 2^a and contains its maximum magnitude code (6.0)
    a = rng.integers(-3, 4, size=(rows, cols // 16))
    codes_in.reshape(rows, -1, 16)[:, :, 0] = 7
    mags = np.where(codes_in & 8, -1.0, 1.0) * E2M1_MAGS[codes_in & 7]
    # a tensor scale that is a power of two: make the largest block max equal 2688 * 2^-10
    ts = 2.0 ** -10
    amax_target = 2688 * ts                       # = 2.625
    blockscale = (2.0 ** a) * ts                 # decoded E4M3 * ts, with E4M3 = 2^a
    x = mags * np.repeat(blockscale, 16, axis=1)
    x[0, 0] = amax_target                        # sets max|x| exactly (code 7 at scale 448*ts/...)
    xb = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16)
    assert np.array_equal(xb.float().numpy(), x.astype(np.float32))   # exactly representable
    codes, sf, tsq, st = orc.quantize_bf16(xb)
    assert tsq == ts
    for r in range(rows):
        for b in range(cols // 16):
            if r == 0 and b == 0:
                continue
            assert orc.e4m3_decode(int(sf[r, b])) == 2.0 ** a[r, b]
            blk = codes[r, b * 8:(b + 1) * 8]
            lo, hi = blk & 15, blk >> 4
            got = np.stack([lo, hi], 1).reshape(-1)
            want = codes_in[r, b * 16:(b + 1) * 16].copy()
            want[(want & 7) == 0] = np.where(want[(want & 7) == 0] & 8, 8, 0)
            assert np.array_equal(got, want), (r, b)


def test_fixed_scale_quantiser_matches_bf16_path(orc):
    """quantize_f32 with the tensor scale the BF16 path computed yields the same bytes."""
    g = torch.Generator().manual_seed(7)
    xb = torch.randn(16, 256, generator=g).to(torch.bfloat16)
    codes, sf, ts, _ = orc.quantize_bf16(xb)
    c2, s2 = orc.quantize_f32(xb.float().numpy(), ts)
    assert np.array_equal(codes, c2) and np.array_equal(sf, s2)


def test_nonfinite_reported(orc):
    xb = torch.zeros(2, 32, dtype=torch.bfloat16)
    xb[1, 3] = float("inf")
    _, _, _, st = orc.quantize_bf16(xb)
    assert st == -6
    xb[1, 3] = float("nan")
    _, _, _, st = orc.quantize_bf16(xb)
    assert st == -6


def test_all_zero_tensor(orc):
    xb = torch.zeros(4, 64, dtype=torch.bfloat16)
    codes, sf, ts, st = orc.quantize_bf16(xb)
    assert st == 0 and ts == 0.0 and not codes.any() and not sf.any()
