"""Pins for the oracle's MX formats and its W4A8 layer (MXFP4 weights, MXFP8 activations and
intermediate, one E8M0 scale per 32 elements, no tensor scale; "b12x" README, section "DeepSeek V4
Flash 0731 MoE reproduction"; E8M0 = 2^(byte - 127): "vllm.cpp docs/STATUS.md", MXFP4 row).

* E8M0 decoding of every byte against 2^(b - 127) (0xFF NaN);
* the block-scale rule 2^(floor(log2 max|x|) - emax) against math.frexp, with the byte clamps;
* every quantised element against a brute-force nearest search over the element format's values
  (built here from the format's closed form), ties to the even code, saturation;
* round-trip bounds, and blocks on the grid (max in the top binade) as fixed points;
* the W4A8 layer: permuted == brute force bit for bit; h and the output against float64 within the
  FP32 summation bounds.
"""
import math

import numpy as np
import pytest

import synth


def _e4m3_values():
    """(code, value) of every finite E4M3 ("fn") code: bias 7, exponent 0 subnormal."""
    out = []
    for c in range(256):
        s, e, m = c >> 7, (c >> 3) & 15, c & 7
        if e == 15 and m == 7:
            continue                                  # NaN
        v = (m / 8.0) * 2.0 ** -6 if e == 0 else (1 + m / 8.0) * 2.0 ** (e - 7)
        out.append((c, -v if s else v))
    return out


def _e2m1_values():
    mags = [0, 0.5, 1, 1.5, 2, 3, 4, 6]
    return [(c, (-1 if c & 8 else 1) * mags[c & 7]) for c in range(16)]


def _nearest(q, table, vmax):
    """Value nearest to q among the format's values, ties to the even code; |q| > vmax -> vmax."""
    if abs(q) >= vmax:
        return math.copysign(vmax, q)
    best = None
    for c, v in table:
        d = abs(v - q)
        if best is None or d < best[0] or (d == best[0] and (c & 1) == 0 and (best[1] & 1) == 1):
            best = (d, c, v)
    return best[2]


E4M3 = _e4m3_values()
E2M1 = _e2m1_values()


def test_e8m0_decode_every_byte(orc):
    for b in range(255):
        assert orc.e8m0_decode(b) == np.float32(2.0 ** (b - 127)), b
    assert math.isnan(orc.e8m0_decode(255))


@pytest.mark.parametrize("emax", [8, 2])
def test_mx_scale_rule(orc, emax):
    rng = np.random.default_rng(emax)
    vals = [0.0, 2.0 ** -149, 2.0 ** -126, 1.0, 448.0, 6.0, 3.0e38]
    vals += [float(np.float32(2.0 ** e)) for e in range(-140, 128, 7)]
    vals += [float(np.nextafter(np.float32(2.0 ** e), np.float32(0))) for e in range(-120, 120, 9)]
    vals += [float(np.float32(v)) for v in 2.0 ** rng.uniform(-140, 127, 200)]
    for a in vals:
        if a == 0.0:
            want = 0
        else:
            _, e = math.frexp(a)                      # a = m 2^e, m in [0.5, 1)
            want = min(254, max(0, (e - 1) - emax + 127))
        assert orc.mx_scale(a, emax) == want, (a, emax)


@pytest.mark.parametrize("kind", ["e4m3", "e2m1"])
def test_mx_quantize_against_brute_force(orc, kind):
    rng = np.random.default_rng(3)
    rows = []
    for mag in (1e-3, 0.7, 1.0, 37.0, 5e4):
        rows.append(rng.standard_normal(64) * mag)
    rows.append(np.zeros(64))                         # an all-zero block pair
    z = rng.standard_normal(64)
    z[:32] = 0.0
    z[5] = 1e-30                                      # a tiny block
    rows.append(z)
    x = np.array(rows, np.float32)
    codes, sc = orc.mx_quantize(x, kind)
    deq = orc.mx_dequantize(codes, sc, kind)
    table, vmax = (E4M3, 448.0) if kind == "e4m3" else (E2M1, 6.0)
    for r in range(x.shape[0]):
        for i in range(x.shape[1]):
            X = 2.0 ** (int(sc[r, i // 32]) - 127)
            want = _nearest(float(x[r, i]) / X, table, vmax) * X
            assert float(deq[r, i]) == want, (kind, r, i, x[r, i], deq[r, i], want)


@pytest.mark.parametrize("kind", ["e4m3", "e2m1"])
def test_mx_round_trip_and_fixed_points(orc, kind):
    rng = np.random.default_rng(11)
    x = (rng.standard_normal((16, 128)) * rng.uniform(0.01, 100, (16, 1))).astype(np.float32)
    codes, sc = orc.mx_quantize(x, kind)
    deq = orc.mx_dequantize(codes, sc, kind).astype(np.float64)
    emax, vmax = (8, 448.0) if kind == "e4m3" else (2, 6.0)
    mant = 3 if kind == "e4m3" else 1
    for r in range(16):
        for b in range(4):
            blk = x[r, b * 32:(b + 1) * 32].astype(np.float64)
            X = 2.0 ** (int(sc[r, b]) - 127)
            amax = np.abs(blk).max()
            assert 2.0 ** emax <= amax / X < 2.0 ** (emax + 1)     # the max in the top binade
            for i in range(32):
                q, v = blk[i] / X, deq[r, b * 32 + i]
                if abs(q) > vmax:                                   # clipped by the format
                    assert v == math.copysign(vmax * X, q)
                    continue
                # spacing of the format's values around q: binade exponent, floored at the
                # smallest normal exponent (E4M3: -6, E2M1: 0), over 2^mantissa bits
                emin = -6 if kind == "e4m3" else 0
                e = max(math.floor(math.log2(abs(q))) if q != 0 else emin, emin)
                gap = 2.0 ** (e - mant)
                assert abs(v - blk[i]) <= 0.5 * gap * X
    # decoded values requantise to themselves: the block max stays in the top binade, so the
    # scale is unchanged and every element is on the grid
    c2, s2 = orc.mx_quantize(deq.astype(np.float32), kind)
    assert np.array_equal(s2, sc) and np.array_equal(c2, codes)


CASES = [
    synth.CONFIGS["tiny"],
    synth.custom_config("w8_shared", 5, 64, 4, 2, 64, shared_inter=32, config_id=151),
    synth.custom_config("w8_k_eq_e", 3, 32, 3, 3, 64, config_id=152),
]


def _mx_experts(cfg, orc):
    experts = [orc.QuantExpertMX.from_bf16(*synth.gen_expert(cfg, e)) for e in range(cfg.experts)]
    sh = orc.QuantExpertMX.from_bf16(*synth.gen_shared(cfg)) if cfg.shared_inter else None
    return experts, sh


@pytest.mark.parametrize("cfg", CASES, ids=lambda c: c.name)
def test_w4a8_permuted_equals_bruteforce(orc, cfg):
    T = cfg.tokens[0]
    x = synth.gen_x(cfg, T)
    logits = synth.gen_logits(cfg, T).numpy()
    experts, sh = _mx_experts(cfg, orc)
    y1 = orc.moe_forward(None, None, None, logits, experts, cfg.top_k, shared=sh, act="mxfp8",
                         x_bf16=x)
    y2 = orc.moe_forward(None, None, None, logits, experts, cfg.top_k, shared=sh, act="mxfp8",
                         x_bf16=x, bruteforce=True)
    assert np.array_equal(y1, y2)
    assert np.abs(orc.bf16_bits_to_f32(y1)).max() > 0


def _dec_e4m3(codes, sc):
    lut = np.full(256, np.nan)
    for c, v in E4M3:
        lut[c] = v
    return lut[codes] * np.repeat(2.0 ** (sc.astype(np.float64) - 127), 32, axis=1)


def _dec_e2m1(codes, sc):
    lut = np.array([v for _, v in E2M1])
    v = lut[np.stack([codes & 15, codes >> 4], -1).reshape(codes.shape[0], -1)]
    return v * np.repeat(2.0 ** (sc.astype(np.float64) - 127), 32, axis=1)


@pytest.mark.parametrize("cfg", CASES[:2], ids=lambda c: c.name)
def test_w4a8_h_and_output_against_float64(orc, cfg):
    T, k, H = cfg.tokens[0], cfg.top_k, cfg.hidden
    x = synth.gen_x(cfg, T)
    logits = synth.gen_logits(cfg, T).numpy()
    experts, sh = _mx_experts(cfg, orc)
    y, d = orc.moe_forward(None, None, None, logits, experts, k, shared=sh, want_debug=True,
                           act="mxfp8", x_bf16=x)
    xf = (np.asarray(orc.as_bf16_bits(x), np.uint32) << 16).view(np.float32)
    xc, xs = orc.mx_quantize(xf, "e4m3")                  # pinned above
    xv = _dec_e4m3(xc, xs)
    I = experts[0].codes[0].shape[0]
    W = [[_dec_e2m1(ex.codes[m], ex.sf[m]) for m in range(3)] for ex in experts]
    for p in range(T * k):
        t = d["perm_src"][p]
        e = int(np.searchsorted(d["offsets"], p, side="right") - 1)
        wg, wu = W[e][0], W[e][1]
        g, u = wg @ xv[t], wu @ xv[t]
        h64 = g / (1 + np.exp(-g)) * u
        bg = H * 2.0 ** -24 * (np.abs(wg) @ np.abs(xv[t]))
        bu = H * 2.0 ** -24 * (np.abs(wu) @ np.abs(xv[t]))
        tol = (np.abs(u) + bu) * bg * 1.1 + np.abs(g) * bu + 1e-6 * np.abs(h64) + 1e-30
        assert np.all(np.abs(d["hf"][p].astype(np.float64) - h64) <= tol), p
    # h in MXFP8 is the requantisation of the FP32 h (the quantiser is pinned above)
    hc, hs = orc.mx_quantize(d["hf"], "e4m3")
    assert np.array_equal(hc, d["hq"]) and np.array_equal(hs, d["hsf"])
    hh = _dec_e4m3(d["hq"], d["hsf"])
    y64 = np.zeros((T, H))
    bound = np.zeros((T, H))
    for t in range(T):
        for j in range(k):
            p = d["inv"][t * k + j]
            wd = W[d["ids"][t, j]][2]
            dd = wd @ hh[p]
            w = float(d["w"][t, j])
            y64[t] += w * dd
            bound[t] += abs(w) * (I * 2.0 ** -24 * (np.abs(wd) @ np.abs(hh[p])) + np.abs(dd) * 2.0 ** -23)
        if sh is not None:
            Ws = [_dec_e2m1(sh.codes[m], sh.sf[m]) for m in range(3)]
            gs, us = Ws[0] @ xv[t], Ws[1] @ xv[t]
            hsv = (gs / (1 + np.exp(-gs)) * us).astype(np.float32)[None, :]
            c8, s8 = orc.mx_quantize(hsv, "e4m3")
            hsh = _dec_e4m3(c8, s8)[0]
            # the float64 h may land on another E4M3 value than the oracle's FP32 h: one step
            # (2^-3 relative) of every element is in the bound
            ds = Ws[2] @ hsh
            y64[t] += ds
            bound[t] += (np.abs(Ws[2]) @ (np.abs(hsh) * 2.0 ** -2)) + np.abs(ds) * 2.0 ** -20
    bound += (k + 2) * 2.0 ** -24 * np.abs(y64)
    yv = orc.bf16_bits_to_f32(y).astype(np.float64)
    assert np.all(np.abs(yv - y64) <= bound + np.abs(y64) * 2.0 ** -8 + 1e-30)
