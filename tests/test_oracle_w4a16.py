"""Pins for the oracle's W4A16 layer (BF16 activations enter the expert GEMMs as they are, the
NVFP4 weights are decoded at the point of use, h is rounded to BF16 before the down projection;
"b12x" README, section "What's in here", moe: W4A16).

* the permuted, expert-by-expert path equals the brute-force per-token loop bit for bit;
* on activations that are fixed points of NVFP4 quantisation (every 16-block holds a +-6 code, the
  tensor scale is a power of two), the W4A16 gate/up GEMM + SwiGLU equals the pinned NVFP4 layer's
  bit for bit - the two paths see the same activation values;
* h is the BF16 rounding of the FP32 h, which agrees with a float64 evaluation of the gate/up
  GEMM within the FP32 summation bound;
* the down projection and combine agree with a float64 evaluation from the oracle's own BF16 h,
  within the FP32 summation bound plus the final BF16 rounding.
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


def _bf16_bits(x_f32: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(x_f32, np.float32)).to(torch.bfloat16) \
        .view(torch.int16).numpy().view(np.uint16)


def _bf16_to_f64(bits) -> np.ndarray:
    return (np.asarray(bits, np.uint32) << 16).view(np.float32).astype(np.float64)


CASES = [
    synth.CONFIGS["tiny"],
    synth.custom_config("w16_shared", 5, 64, 4, 2, 64, shared_inter=32, config_id=141),
    synth.custom_config("w16_k_eq_e", 3, 32, 3, 3, 48, config_id=142),
    synth.custom_config("w16_k1", 6, 64, 5, 1, 32, config_id=143),
]


def _experts(cfg, orc):
    experts = [orc.QuantExpert.from_bf16(*synth.gen_expert(cfg, e)) for e in range(cfg.experts)]
    sh = orc.QuantExpert.from_bf16(*synth.gen_shared(cfg)) if cfg.shared_inter else None
    return experts, sh


@pytest.mark.parametrize("cfg", CASES, ids=lambda c: c.name)
def test_w4a16_permuted_equals_bruteforce(orc, cfg):
    T = cfg.tokens[0]
    x = synth.gen_x(cfg, T)
    logits = synth.gen_logits(cfg, T).numpy()
    experts, sh = _experts(cfg, orc)
    y1 = orc.moe_forward(None, None, None, logits, experts, cfg.top_k, shared=sh, act="bf16", x_bf16=x)
    y2 = orc.moe_forward(None, None, None, logits, experts, cfg.top_k, shared=sh, act="bf16",
                         x_bf16=x, bruteforce=True)
    assert np.array_equal(y1, y2)
    assert np.abs(orc.bf16_bits_to_f32(y1)).max() > 0


def _grid_activations(T, H, seed, orc):
    """x on the NVFP4 grid and a fixed point of its quantisation: random codes with a +-6 code in
    every 16-block, random E4M3 scales, tensor scale 2^-4 (one block holds 6 * 448 * 2^-4)."""
    rng = np.random.default_rng(seed)
    codes = rng.integers(0, 16, size=(T, H), dtype=np.uint8)
    six = rng.integers(0, 16, size=(T, H // 16))
    sign = rng.integers(0, 2, size=(T, H // 16)).astype(np.uint8)
    for t in range(T):
        for b in range(H // 16):
            codes[t, b * 16 + six[t, b]] = 7 | (sign[t, b] << 3)
    sf = rng.integers(0x28, 0x48, size=(T, H // 16), dtype=np.uint8)
    sf[0, 0] = 0x7E                                    # 448: the tensor max is 6 * 448 * ts
    ts = 2.0 ** -4
    packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    xhat = _dec(packed, sf, ts, orc)
    x_bits = _bf16_bits(xhat.astype(np.float32))
    assert np.array_equal(_bf16_to_f64(x_bits), xhat)  # every value is exact in BF16
    return x_bits, packed, sf, ts


def test_w4a16_gemm1_equals_nvfp4_on_grid_activations(orc):
    cfg = synth.custom_config("w16_grid", 6, 64, 4, 2, 48, shared_inter=32, config_id=144)
    T, H = 6, 64
    x_bits, packed, sf, ts = _grid_activations(T, H, 7, orc)
    xq, xsf, ts_a, st = orc.quantize_bf16(x_bits)
    assert st == 0 and ts_a == np.float32(ts)
    assert np.array_equal(xq, packed) and np.array_equal(xsf, sf)   # a fixed point
    logits = synth.gen_logits(cfg, T).numpy()
    experts, sh = _experts(cfg, orc)
    _, d4 = orc.moe_forward(xq, xsf, ts_a, logits, experts, 2, shared=sh, want_debug=True)
    _, d16 = orc.moe_forward(None, None, None, logits, experts, 2, shared=sh, want_debug=True,
                             act="bf16", x_bf16=x_bits)
    assert np.array_equal(d4["ids"], d16["ids"]) and np.array_equal(d4["inv"], d16["inv"])
    assert np.array_equal(d4["hf"].view(np.uint32), d16["hf"].view(np.uint32))
    assert np.abs(d16["hf"]).max() > 0


@pytest.mark.parametrize("cfg", CASES[:2], ids=lambda c: c.name)
def test_w4a16_h_and_output_against_float64(orc, cfg):
    T, k, H = cfg.tokens[0], cfg.top_k, cfg.hidden
    x = synth.gen_x(cfg, T)
    logits = synth.gen_logits(cfg, T).numpy()
    experts, sh = _experts(cfg, orc)
    y, d = orc.moe_forward(None, None, None, logits, experts, k, shared=sh, want_debug=True,
                           act="bf16", x_bf16=x)
    xv = _bf16_to_f64(orc.as_bf16_bits(x))
    # h: the BF16 rounding of the FP32 h
    assert np.array_equal(d["hb"], _bf16_bits(d["hf"]))
    # the FP32 h against float64 GEMM1 + SiLU, row by row in permuted order
    I = experts[0].codes[0].shape[0]
    for p in range(T * k):
        t = d["perm_src"][p]
        e = int(np.searchsorted(d["offsets"], p, side="right") - 1)
        ex = experts[e]
        wg = _dec(ex.codes[0], ex.sf[0], ex.ts[0], orc)
        wu = _dec(ex.codes[1], ex.sf[1], ex.ts[1], orc)
        g, u = wg @ xv[t], wu @ xv[t]
        h64 = g / (1 + np.exp(-g)) * u
        bg = H * 2.0 ** -24 * (np.abs(wg) @ np.abs(xv[t]))    # FP32 summation bounds
        bu = H * 2.0 ** -24 * (np.abs(wu) @ np.abs(xv[t]))
        tol = (np.abs(u) + bu) * bg * 1.1 + np.abs(g) * bu + 1e-6 * np.abs(h64) + 1e-30
        assert np.all(np.abs(d["hf"][p].astype(np.float64) - h64) <= tol), p
    # the down projection + combine from the oracle's own BF16 h
    hb = _bf16_to_f64(d["hb"])
    y64 = np.zeros((T, H))
    bound = np.zeros((T, H))
    for t in range(T):
        for j in range(k):
            p = d["inv"][t * k + j]
            ex = experts[d["ids"][t, j]]
            wd = _dec(ex.codes[2], ex.sf[2], ex.ts[2], orc)
            dd = wd @ hb[p]
            w = float(d["w"][t, j])
            y64[t] += w * dd
            bound[t] += abs(w) * (I * 2.0 ** -24 * (np.abs(wd) @ np.abs(hb[p])) + np.abs(dd) * 2.0 ** -23)
        if sh is not None:
            wd = _dec(sh.codes[2], sh.sf[2], sh.ts[2], orc)
            ws = [_dec(sh.codes[m], sh.sf[m], sh.ts[m], orc) for m in (0, 1)]
            hs = ws[0] @ xv[t]
            hsh = _bf16_to_f64(_bf16_bits((hs / (1 + np.exp(-hs)) * (ws[1] @ xv[t])).astype(np.float32)))
            # the shared row's h is re-derived in float64 and may round to another BF16 value than
            # the oracle's FP32 h; its share of the bound covers one BF16 step of every h element
            ds = wd @ hsh
            y64[t] += ds
            bound[t] += (np.abs(wd) @ (np.abs(hsh) * 2.0 ** -7)) + np.abs(ds) * 2.0 ** -20
    bound += (k + 2) * 2.0 ** -24 * np.abs(y64)
    yv = orc.bf16_bits_to_f32(y).astype(np.float64)
    assert np.all(np.abs(yv - y64) <= bound + np.abs(y64) * 2.0 ** -8 + 1e-30)
