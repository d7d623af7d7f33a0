"""Oracle pins for RMSNorm + NVFP4 quantisation (the producer feeding the activation quantiser;
"nvfp4-megamoe-kernel compare pre-b1...master", sections "P4 - Fused RMSNorm + NVFP4 quantize"
and "P5"): exact special cases, scale invariance, float64 agreement, the sum of squares against
exact rational arithmetic, and the reduction to the plain quantiser of the normalised values."""
import numpy as np
import torch

import oracle


def _gamma(cols, seed=0):
    g = torch.from_numpy(np.random.default_rng(seed).normal(1.0, 0.1, cols).astype(np.float32))
    return g.to(torch.bfloat16)


def test_constant_rows_normalise_to_gamma():
    cols = 512
    g = _gamma(cols)
    x = torch.full((3, cols), 2.0).to(torch.bfloat16)       # mean square 4, rms 2 exactly
    _, _, _, st, y = oracle.rmsnorm_quantize(x, g, 0.0)
    assert st == 0
    assert np.array_equal(y, np.tile(g.float().numpy(), (3, 1)))


def test_scale_invariance_is_bit_exact():
    rng = np.random.default_rng(1)
    x = torch.from_numpy(rng.standard_normal((16, 1024)).astype(np.float32)).to(torch.bfloat16)
    g = _gamma(1024, 2)
    c1, s1, t1, _, y1 = oracle.rmsnorm_quantize(x, g, 0.0)
    c2, s2, t2, _, y2 = oracle.rmsnorm_quantize((x.float() * 2).to(torch.bfloat16), g, 0.0)
    assert np.array_equal(y1, y2) and t1 == t2
    assert np.array_equal(c1, c2) and np.array_equal(s1, s2)


def test_matches_float64_rmsnorm():
    rng = np.random.default_rng(3)
    x = torch.from_numpy((rng.standard_normal((32, 2048)) * 3).astype(np.float32)).to(torch.bfloat16)
    g = _gamma(2048, 4)
    eps = 1e-5
    _, _, ts, st, y = oracle.rmsnorm_quantize(x, g, eps)
    xd = x.float().numpy().astype(np.float64)
    ref = xd / np.sqrt((xd * xd).mean(axis=1, keepdims=True) + eps) * g.float().numpy()
    assert st == 0
    assert np.abs(y - ref).max() <= 1e-6 * np.abs(ref).max()
    assert ts == np.float32(np.abs(y).max()) / np.float32(2688.0)


def test_codes_are_the_quantiser_of_the_normalised_values():
    rng = np.random.default_rng(5)
    x = torch.from_numpy(rng.standard_normal((8, 768)).astype(np.float32)).to(torch.bfloat16)
    codes, sf, ts, st, y = oracle.rmsnorm_quantize(x, _gamma(768, 6), 1e-6)
    c2, s2 = oracle.quantize_f32(y, ts)
    assert st == 0 and np.array_equal(codes, c2) and np.array_equal(sf, s2)


def test_zero_gamma_gives_zero():
    x = torch.randn(4, 256).to(torch.bfloat16)
    codes, sf, ts, st, y = oracle.rmsnorm_quantize(x, torch.zeros(256).to(torch.bfloat16), 1e-6)
    assert st == 0 and ts == 0.0 and not y.any() and not codes.any() and not sf.any()


def _round_f32(q):
    """The FP32 value nearest to the exact rational q >= 0 (ties to even), in exact arithmetic."""
    from fractions import Fraction
    if q == 0:
        return 0.0
    e = q.numerator.bit_length() - q.denominator.bit_length()
    if Fraction(2) ** e > q:
        e -= 1
    quantum = Fraction(2) ** (e - 23)          # 24 significant bits (normal range)
    n, rem = divmod(q, quantum)
    if rem * 2 > quantum or (rem * 2 == quantum and n % 2 == 1):
        n += 1
    return float(n * quantum)


def test_sum_squares_is_the_exact_sum_rounded_once():
    from fractions import Fraction
    # a power-of-two count of equal squares sums exactly
    assert oracle.sum_squares(np.ones(128, np.float32)) == 128.0
    # squares 2^24, 1, 1, 1: the exact sum 2^24 + 3 lies halfway between two FP32 values and
    # rounds to the even one, 2^24 + 4.  A left-to-right FP32 sum stays at 2^24 and a pairwise
    # tree over chunks of 8 gives 2^24 + 2: both fail here.
    v = np.zeros(32, np.float32)
    v[0] = 4096.0
    v[8] = v[16] = v[24] = 1.0
    assert oracle.sum_squares(v) == 2.0**24 + 4
    # BF16-valued rows with a wide spread of magnitudes (tiny values included): the correctly
    # rounded FP32 of the exact rational sum, whatever the order of the elements
    rng = np.random.default_rng(8)
    for n in (7, 2048, 7168):
        r = (rng.standard_normal(n) * np.exp2(rng.integers(-20, 8, n))).astype(np.float32)
        r = torch.from_numpy(r).to(torch.bfloat16).float().numpy()
        exact = sum(Fraction(float(a)) ** 2 for a in r)
        assert oracle.sum_squares(r) == _round_f32(exact)
        assert oracle.sum_squares(rng.permutation(r)) == oracle.sum_squares(r)


def test_rms_of_each_row():
    """Each row's 1/rms follows from the rounded sum: r = 1 / sqrt(sum / cols + eps) in FP32."""
    rng = np.random.default_rng(9)
    x = torch.from_numpy(rng.standard_normal((6, 512)).astype(np.float32)).to(torch.bfloat16)
    g = _gamma(512, 10)
    *_, r = oracle.rmsnorm_quantize(x, g, 1e-5, want_r=True)
    for i in range(6):
        s = np.float32(oracle.sum_squares(x[i].float().numpy()))
        want = np.float32(1.0) / np.sqrt(s / np.float32(512) + np.float32(1e-5))
        assert r[i] == want
