"""Oracle pins for RMSNorm + NVFP4 quantisation (the producer feeding the activation quantiser;
"nvfp4-megamoe-kernel compare pre-b1...master", sections "P4 - Fused RMSNorm + NVFP4 quantize"
and "P5"): exact special cases, scale invariance, float64 agreement and the reduction to the
plain quantiser of the normalised values."""
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


def test_sum_squares_tree_exact_cases():
    # a power-of-two count of equal squares sums exactly; sixteen chunks of ones = 128
    assert oracle.sum_squares_tree(np.ones(128, np.float32)) == 128.0
    # the pairwise order is observable: chunk sums 2^24, 1, 1, 1 give (2^24 + 1) + (1 + 1)
    # = 2^24 + 2 (the first pair rounds to 2^24, the second is exact), where a left-to-right sum
    # would stay at 2^24
    v = np.zeros(32, np.float32)
    v[0] = 4096.0
    v[8] = v[16] = v[24] = 1.0
    assert oracle.sum_squares_tree(v) == np.float32(2.0**24 + 2)
    # agreement with float64 within the FP32 tree's error bound
    r = np.random.default_rng(8).standard_normal(7168).astype(np.float32)
    exact = float((r.astype(np.float64) ** 2).sum())
    assert abs(oracle.sum_squares_tree(r) - exact) <= 7168 * 2 ** -24 * exact
