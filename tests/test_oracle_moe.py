"""Pins for the oracle's whole layer.

* the permuted, expert-by-expert path equals a brute-force per-token loop bit for bit;
* the shared expert equals a routed expert reached with k = 1;
* the down projection and combine agree with a float64 evaluation from the oracle's own
  requantised intermediate, within the FP32 summation bound;
* the gate/up GEMM + SwiGLU agree with a float64 evaluation, and requantising that float64 h
  gives the oracle's codes except at rare rounding boundaries;
* on inputs whose every product and partial sum is exact in FP32, GEMM1 (with SiLU saturated to
  the identity) and GEMM2 reproduce a float64 evaluation exactly.
"""
import numpy as np
import pytest
import torch

import synth

E2M1 = np.array([0, .5, 1, 1.5, 2, 3, 4, 6, -0.0, -.5, -1, -1.5, -2, -3, -4, -6], np.float64)


def _dec(codes, sf, ts, orc):
    lo, hi = codes & 15, codes >> 4
    v = E2M1[np.stack([lo, hi], -1).reshape(codes.shape[0], -1)]
    s = np.vectorize(orc.e4m3_decode)(sf).astype(np.float64)
    return v * np.repeat(s, 16, axis=1) * ts


def _layer(cfg, T, orc, shared=True):
    x = synth.gen_x(cfg, T)
    logits = synth.gen_logits(cfg, T).numpy()
    xq, xsf, ts_a, st = orc.quantize_bf16(x)
    assert st == 0
    experts = [orc.QuantExpert.from_bf16(*synth.gen_expert(cfg, e)) for e in range(cfg.experts)]
    sh = orc.QuantExpert.from_bf16(*synth.gen_shared(cfg)) if (cfg.shared_inter and shared) else None
    return xq, xsf, ts_a, logits, experts, sh


CASES = [
    synth.CONFIGS["tiny"],
    synth.custom_config("small_shared", 5, 64, 4, 2, 64, shared_inter=32, config_id=101),
    synth.custom_config("k_eq_e", 3, 32, 3, 3, 48, config_id=102),
    synth.custom_config("k1", 6, 64, 5, 1, 32, config_id=103),
]


@pytest.mark.parametrize("cfg", CASES, ids=lambda c: c.name)
def test_permuted_equals_bruteforce(orc, cfg):
    T = cfg.tokens[0]
    xq, xsf, ts_a, logits, experts, sh = _layer(cfg, T, orc)
    y1 = orc.moe_forward(xq, xsf, ts_a, logits, experts, cfg.top_k, shared=sh)
    y2 = orc.moe_forward(xq, xsf, ts_a, logits, experts, cfg.top_k, shared=sh, bruteforce=True)
    assert np.array_equal(y1, y2)
    assert np.abs(orc.bf16_bits_to_f32(y1)).max() > 0


def test_shared_expert_equals_k1_routed(orc):
    cfg = synth.custom_config("sh_eq", 7, 64, 1, 1, 32, shared_inter=32, config_id=104)
    x = synth.gen_x(cfg, 7)
    xq, xsf, ts_a, _ = orc.quantize_bf16(x)
    logits = np.zeros((7, 1), np.float32)
    W = orc.QuantExpert.from_bf16(*synth.gen_shared(cfg))
    Z = orc.QuantExpert.from_bf16(*[torch.zeros_like(w) for w in synth.gen_shared(cfg)])
    ya, da = orc.moe_forward(xq, xsf, ts_a, logits, [W], 1, want_debug=True)
    yb, db = orc.moe_forward(xq, xsf, ts_a, logits, [Z], 1, shared=W, want_debug=True)
    assert np.array_equal(ya, yb)
    assert np.array_equal(da["hq"], db["shq"]) and np.array_equal(da["hsf"], db["shsf"])


@pytest.mark.parametrize("cfg", CASES[:2], ids=lambda c: c.name)
def test_against_float64(orc, cfg):
    T, H, I, k = cfg.tokens[0], cfg.hidden, cfg.inter, cfg.top_k
    xq, xsf, ts_a, logits, experts, sh = _layer(cfg, T, orc)
    y, dbg = orc.moe_forward(xq, xsf, ts_a, logits, experts, k, shared=sh, want_debug=True)
    xhat = _dec(xq, xsf, ts_a, orc)
    ids, w, inv = dbg["ids"], dbg["w"].astype(np.float64), dbg["inv"]
    hq, hsf = dbg["hq"], dbg["hsf"]
    n_code_diff = n_codes = 0
    acc = np.zeros((T, H))
    bound = np.zeros((T, H))
    for t in range(T):
        for j in range(k):
            ex = experts[ids[t, j]]
            Wg, Wu, Wd = (_dec(ex.codes[m], ex.sf[m], ex.ts[m], orc) for m in range(3))
            g = Wg @ xhat[t]
            u = Wu @ xhat[t]
            h = g / (1 + np.exp(-g)) * u
            p = inv[t * k + j]
            # requantising the float64 h reproduces the oracle's codes except at boundaries
            c64, s64 = orc.quantize_f32(h[None, :].astype(np.float32), 1.0)
            n_code_diff += int(np.sum(c64 != hq[p])) + int(np.sum(s64 != hsf[p]))
            n_codes += hq.shape[1] + hsf.shape[1]
            hhat = _dec(hq[p:p + 1], hsf[p:p + 1], 1.0, orc)[0]
            d = Wd @ hhat
            acc[t] += w[t, j] * d
            bound[t] += abs(w[t, j]) * (np.abs(Wd) @ np.abs(hhat)) * I * 2.0 ** -23
        if sh is not None:
            Wg, Wu, Wd = (_dec(sh.codes[m], sh.sf[m], sh.ts[m], orc) for m in range(3))
            g, u = Wg @ xhat[t], Wu @ xhat[t]
            hhat = _dec(dbg["shq"][t:t + 1], dbg["shsf"][t:t + 1], 1.0, orc)[0]
            acc[t] += Wd @ hhat
            bound[t] += (np.abs(Wd) @ np.abs(hhat)) * cfg.shared_inter * 2.0 ** -23
    yf = orc.bf16_bits_to_f32(y).astype(np.float64)
    # FP32 sequential-sum bound, plus half a BF16 ulp of the rounding to the output
    tol = bound + 2 * k * 2.0 ** -24 * np.abs(acc) + np.abs(acc) * 2.0 ** -8 + 1e-30
    assert np.all(np.abs(yf - acc) <= tol)
    assert n_code_diff <= max(2, n_codes // 1000)


def test_exact_products_against_float64(orc):
    """E=1, k=1, positive on-grid x and gate weights so that g >= 100 (SiLU(g) == g in FP32):
    every product and partial sum is exact, so h = g*u and y are exact."""
    H, I, T = 32, 16, 3
    rng = np.random.default_rng(21)
    # quantised operands built directly: power-of-two scales, small codes
    def mk(rows, cols, positive, ts, lo=1, hi=6):
        codes = rng.integers(lo, hi, size=(rows, cols)).astype(np.uint8)   # e.g. 0.5 .. 3.0
        if not positive:
            codes |= (rng.integers(0, 2, size=(rows, cols)).astype(np.uint8) << 3)
        packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
        sf = np.full((rows, cols // 16), 0x38, np.uint8)     # block scale 1.0
        return packed, sf, ts
    xq, xsf, ts_a = mk(T, H, True, 2.0, 3, 6)      # x_hat in {3, 4, 6}
    g_ = mk(I, H, True, 1.0, 3, 6)                 # 1.5 .. 3: g >= 144
    u_ = mk(I, H, False, 0.25)
    d_ = mk(H, I, False, 0.5)
    ex = orc.QuantExpert([g_[0], u_[0], d_[0]], [g_[1], u_[1], d_[1]], [g_[2], u_[2], d_[2]])
    logits = np.zeros((T, 1), np.float32)
    ts_h = 2.0 ** 8
    y, dbg = orc.moe_forward(xq, xsf, ts_a, logits, [ex], 1, ts_h=ts_h, want_debug=True)
    xhat = _dec(xq, xsf, ts_a, orc)
    Wg, Wu, Wd = (_dec(ex.codes[m], ex.sf[m], ex.ts[m], orc) for m in range(3))
    for t in range(T):
        g = Wg @ xhat[t]
        assert g.min() >= 100
        h = g * (Wu @ xhat[t])                      # SiLU(g) == g exactly in FP32 here
        c, s = orc.quantize_f32(h[None].astype(np.float32), ts_h)
        assert np.array_equal(c[0], dbg["hq"][t]) and np.array_equal(s[0], dbg["hsf"][t])
        hhat = _dec(c, s, ts_h, orc)[0]
        yt = Wd @ hhat
        want = torch.from_numpy(yt.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy()
        assert np.array_equal(y[t].view(np.int16), want)


def test_openmp_build_gives_identical_bits(orc):
    """The all-core build of the oracle (OpenMP over independent experts, rows and tokens) gives
    the single-threaded oracle's bits: outputs, routing, plan and requantised intermediates."""
    cs = synth.custom_config("omp", 24, 256, 6, 3, 256, shared_inter=256, config_id=170)
    x = synth.gen_x(cs, 24)
    lg = synth.gen_logits(cs, 24).numpy()
    ex = [orc.QuantExpert.from_bf16(*synth.gen_expert(cs, e)) for e in range(cs.experts)]
    sh = orc.QuantExpert.from_bf16(*synth.gen_shared(cs))
    outs = []
    for n in (1, 4):
        if orc.use_threads(n) != n and n != 1:
            pytest.skip("no OpenMP build of the oracle on this host")
        xq, xsf, ts, _ = orc.quantize_bf16(x)
        y, d = orc.moe_forward(xq, xsf, ts, lg, ex, cs.top_k, shared=sh, want_debug=True)
        outs.append((xq, xsf, ts, y, d))
    orc.use_threads(1)
    a, b = outs
    assert a[2] == b[2] and np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    assert np.array_equal(a[3], b[3])
    for key in a[4]:
        assert np.array_equal(a[4][key], b[4][key]), key
