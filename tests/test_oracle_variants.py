"""Oracle pins for the router and activation variants (sqrt-softplus router with a selection-only
bias, clamped SwiGLU), against closed forms, special cases that reduce to the base layer, and
brute force.  Definitions: "vllm.cpp docs/STATUS.md", paragraph "W6 sqrtsoftplus + hash-routed
MoE"; "nvfp4-megamoe-kernel compare pre-b1...master", sections "Dense Router (L3+)" and
"Nvfp4MoE (Routed Experts)" (swiglu_limit=10.0)."""
import math

import numpy as np
import pytest

import oracle
import synth
from parity import oracle_experts_from


def test_sqrt_softplus_closed_forms():
    assert oracle.sqrt_softplus(0.0) == np.float32(math.sqrt(math.log(2.0)))
    assert oracle.sqrt_softplus(25.0) == 5.0                     # softplus(x) = x above 20
    for x in (-20.0, -5.0, -0.5, 0.5, 3.0, 19.5):
        want = math.sqrt(math.log1p(math.exp(x)))
        assert abs(oracle.sqrt_softplus(x) - want) <= 2e-7 * want
    xs = np.linspace(-30, 30, 2001, dtype=np.float32)
    v = np.array([oracle.sqrt_softplus(float(x)) for x in xs])
    assert np.all(np.diff(v) >= 0)                                # monotone


def _scores64(lg):
    lg = lg.astype(np.float64)
    return np.where(lg > 20, np.sqrt(np.maximum(lg, 0)), np.sqrt(np.log1p(np.exp(lg))))


def test_zero_bias_selects_like_softmax():
    """sqrt(softplus) is increasing, so without a bias it picks the same experts in the same
    order as the softmax router."""
    lg = np.random.default_rng(1).standard_normal((256, 64)).astype(np.float32)
    ids0, _ = oracle.router(lg, 8)
    ids1, _ = oracle.router(lg, 8, "sqrtsoftplus")
    ids2, _ = oracle.router(lg, 8, "sqrtsoftplus", np.zeros(64, np.float32))
    assert np.array_equal(ids0, ids1) and np.array_equal(ids0, ids2)


def test_weights_are_normalised_unbiased_scores():
    rng = np.random.default_rng(2)
    lg = rng.standard_normal((128, 32)).astype(np.float32)
    bias = (rng.standard_normal(32) * 0.5).astype(np.float32)
    ids, w = oracle.router(lg, 6, "sqrtsoftplus", bias)
    s = _scores64(lg)
    chosen = np.take_along_axis(s, ids, axis=1)
    np.testing.assert_allclose(w.sum(axis=1), 1.0, rtol=2e-6)
    np.testing.assert_allclose(w, chosen / chosen.sum(axis=1, keepdims=True), rtol=2e-6)


def test_bias_selects_but_does_not_weight():
    lg = np.linspace(1.0, 0.0, 16, dtype=np.float32)[None, :].copy()   # expert 15 is the worst
    bias = np.zeros(16, np.float32)
    bias[15] = 10.0
    ids, w = oracle.router(lg, 4, "sqrtsoftplus", bias)
    assert ids[0, 0] == 15 and list(ids[0, 1:]) == [0, 1, 2]
    s = _scores64(lg)[0]
    np.testing.assert_allclose(w[0], s[[15, 0, 1, 2]] / s[[15, 0, 1, 2]].sum(), rtol=2e-6)
    assert w[0, 0] < w[0, 1]          # the biased pick keeps its own, smallest score as weight


def test_selection_matches_brute_force():
    rng = np.random.default_rng(3)
    T, E, k = 512, 96, 8
    lg = (rng.standard_normal((T, E)) * 2).astype(np.float32)
    bias = (rng.standard_normal(E) * 0.3).astype(np.float32)
    ids, _ = oracle.router(lg, k, "sqrtsoftplus", bias)
    sel = _scores64(lg) + bias.astype(np.float64)
    checked = 0
    for t in range(T):
        order = sorted(range(E), key=lambda e: (-sel[t, e], e))
        if sel[t, order[k - 1]] - sel[t, order[k]] < 1e-5:     # a float32 near-tie: skip
            continue
        assert list(ids[t]) == order[:k]
        checked += 1
    assert checked > T - 5


@pytest.fixture(scope="module")
def tiny_layer():
    cs = synth.CONFIGS["tiny"]
    T = 16
    x = synth.gen_x(cs, T)
    lg = synth.gen_logits(cs, T).numpy()
    wg, wu, wd = synth.gen_all_experts(cs)
    xq, xsf, ts_a, st = oracle.quantize_bf16(x)
    assert st == 0
    experts = oracle_experts_from(wg, wu, wd, np.arange(cs.experts))
    return cs, xq, xsf, ts_a, lg, experts


def _run(layer, **kw):
    cs, xq, xsf, ts_a, lg, experts = layer
    return oracle.moe_forward(xq, xsf, ts_a, lg, experts, cs.top_k, want_debug=True, **kw)


def test_clamp_with_huge_limit_is_the_plain_layer(tiny_layer):
    y0, d0 = _run(tiny_layer)
    y1, d1 = _run(tiny_layer, swiglu_limit=1e30)
    assert np.array_equal(y0, y1) and np.array_equal(d0["hq"], d1["hq"])


def test_clamp_with_zero_limit_zeroes_the_experts(tiny_layer):
    y, d = _run(tiny_layer, swiglu_limit=0.0)
    assert not np.any(y & 0x7FFF)                 # +-0 everywhere
    assert not np.any(d["hsf"]) and not np.any(d["hq"] & 0x77)


def test_small_limit_bounds_h(tiny_layer):
    L = 0.05
    y0, _ = _run(tiny_layer)
    y, d = _run(tiny_layer, swiglu_limit=L)
    assert not np.array_equal(y0, y)
    hh = oracle.dequantize(d["hq"], d["hsf"], 1.0)
    silu_max = max(L / (1.0 + math.exp(-L)), 0.2785)            # |silu(g)| for g <= L
    assert np.abs(hh).max() <= silu_max * L * 1.07              # + the E4M3 scale rounding


@pytest.mark.parametrize("limit", [None, 0.05, 10.0])
def test_variants_permuted_equals_brute_force(tiny_layer, limit):
    cs, xq, xsf, ts_a, lg, experts = tiny_layer
    bias = (np.random.default_rng(4).standard_normal(cs.experts) * 0.2).astype(np.float32)
    kw = dict(router_mode="sqrtsoftplus", router_bias=bias, swiglu_limit=limit)
    y = oracle.moe_forward(xq, xsf, ts_a, lg, experts, cs.top_k, **kw)
    yb = oracle.moe_forward(xq, xsf, ts_a, lg, experts, cs.top_k, bruteforce=True, **kw)
    assert np.array_equal(y, yb)


def _silu64(g):
    return g / (1.0 + math.exp(-g))


@pytest.mark.parametrize("g,u,L,gate,up", [
    (-5.0, 3.0, 1.0, -5.0, 1.0),     # gate clamped from above only: -5 passes, up clipped to L
    (5.0, -3.0, 1.0, 1.0, -1.0),     # gate clipped to L, up clipped to -L
    (0.3, 0.2, 1.0, 0.3, 0.2),       # inside the limits: plain SwiGLU
    (-40.0, -40.0, 10.0, -40.0, -10.0),
    (12.0, 7.0, 10.0, 10.0, 7.0),
])
def test_swiglu_clamp_closed_forms(g, u, L, gate, up):
    want = _silu64(gate) * up
    got = oracle.swiglu(g, u, L)
    assert abs(got - want) <= 1e-6 * max(abs(want), 1e-30)
    assert oracle.swiglu(g, u) == pytest.approx(_silu64(g) * u, rel=1e-6, abs=1e-30)


def test_swiglu_zero_limit_is_zero():
    for g in (-3.0, -0.1, 0.0, 0.1, 50.0):
        for u in (-2.0, 0.0, 9.0):
            assert oracle.swiglu(g, u, 0.0) == 0.0


# ---- the other activations of the pages' MoE ("b12x" README, "What's in here", moe: "with
# SiLU/ReLU2/SwiGLU-OAI activations"): squared ReLU of a non-gated expert, gpt-oss SwiGLU

def test_relu2_closed_forms():
    for u, want in ((3.0, 9.0), (0.5, 0.25), (-2.0, 0.0), (0.0, 0.0), (-0.0, 0.0), (1e-20, 0.0)):
        for g in (-7.0, 0.0, 11.0):                              # the gate plays no part
            assert oracle.activation(g, u, "relu2") == np.float32(np.float32(u) * np.float32(u)
                                                                  if u > 0 else 0.0)
            assert oracle.activation(g, u, "relu2") == want or u == 1e-20


def _oai64(g, u, L, a):
    g = min(g, L)
    u = min(max(u, -L), L)
    return (u + 1.0) * g / (1.0 + math.exp(-a * g))


@pytest.mark.parametrize("g,u", [(0.3, 0.2), (-2.0, 1.5), (3.0, -0.5), (12.0, 3.0), (2.0, 9.0),
                                 (2.0, -9.0), (-30.0, 2.0), (6.99, 6.99)])
def test_swiglu_oai_closed_forms(g, u):
    L, a = 7.0, 1.702
    want = _oai64(g, u, L, a)
    got = oracle.activation(g, u, "swiglu_oai", L, a)
    # the rounding of alpha * g' moves exp(-alpha * g') by |alpha * g'| * 2^-24 relative
    rel = (abs(a * min(g, L)) + 8) * 2.0 ** -24
    assert abs(got - want) <= rel * max(abs(want), 1e-30) + 1e-30


def test_swiglu_oai_special_values():
    L, a = 7.0, 1.702
    for g in (-3.0, 0.5, 40.0):
        assert oracle.activation(g, -1.0, "swiglu_oai", L, a) == 0.0    # u + 1 = 0
    for u in (-5.0, 0.0, 5.0):
        assert oracle.activation(0.0, u, "swiglu_oai", L, a) == 0.0     # g = 0
    # the gate is clamped from above only, the up value on both sides
    assert oracle.activation(100.0, 2.0, "swiglu_oai", L, a) == \
        oracle.activation(L, 2.0, "swiglu_oai", L, a)
    assert oracle.activation(1.0, 100.0, "swiglu_oai", L, a) == \
        oracle.activation(1.0, L, "swiglu_oai", L, a)
    assert oracle.activation(1.0, -100.0, "swiglu_oai", L, a) == \
        oracle.activation(1.0, -L, "swiglu_oai", L, a)
    assert oracle.activation(-100.0, 2.0, "swiglu_oai", L, a) != \
        oracle.activation(-L, 2.0, "swiglu_oai", L, a)


@pytest.fixture(scope="module")
def act_layer():
    """A layer with a shared expert whose expert weights serve all three activations (the ReLU2
    experts drop their gate matrix)."""
    cs = synth.custom_config("act_variants", 12, 256, 6, 2, 256, shared_inter=256, config_id=172)
    x = synth.gen_x(cs, 12)
    lg = synth.gen_logits(cs, 12).numpy()
    ws = [synth.gen_expert(cs, e) for e in range(cs.experts)]
    sh = synth.gen_shared(cs)
    xq, xsf, ts_a, st = oracle.quantize_bf16(x)
    gated = [oracle.QuantExpert.from_bf16(*w) for w in ws]
    plain = [oracle.QuantExpert.from_bf16(None, w[1], w[2]) for w in ws]
    return dict(cs=cs, xq=xq, xsf=xsf, ts=ts_a, lg=lg, gated=gated, plain=plain,
                sh_g=oracle.QuantExpert.from_bf16(*sh), sh_p=oracle.QuantExpert.from_bf16(None, *sh[1:]))


def _act_run(L, kind, bruteforce=False, debug=False):
    ex, sh = (L["plain"], L["sh_p"]) if kind == "relu2" else (L["gated"], L["sh_g"])
    lim = 7.0 if kind == "swiglu_oai" else None
    return oracle.moe_forward(L["xq"], L["xsf"], L["ts"], L["lg"], ex, L["cs"].top_k, shared=sh,
                              activation=kind, swiglu_limit=lim, bruteforce=bruteforce,
                              want_debug=debug)


@pytest.mark.parametrize("kind", ["relu2", "swiglu_oai"])
def test_activation_variants_permuted_equals_brute_force(act_layer, kind):
    assert np.array_equal(_act_run(act_layer, kind), _act_run(act_layer, kind, bruteforce=True))


@pytest.mark.parametrize("kind", ["relu2", "swiglu_oai"])
def test_activation_variants_h_against_float64(act_layer, kind):
    """The FP32 h of every routed row equals a float64 evaluation of the activation's formula on
    the decoded operands within the FP32 summation bound of its dot products: a gated ReLU2, an
    unsquared one, or swapped gate and up values of SwiGLU-OAI all fail here."""
    L = act_layer
    cs = L["cs"]
    _, d = _act_run(L, kind, debug=True)
    xh = oracle.dequantize(L["xq"], L["xsf"], L["ts"]).astype(np.float64)
    ex = L["plain"] if kind == "relu2" else L["gated"]
    H, k = cs.hidden, cs.top_k
    for p in range(cs.tokens[0] * k):
        t = d["perm_src"][p]
        e = d["ids"].reshape(-1)[[i for i in range(len(d["inv"])) if d["inv"][i] == p][0]]
        wu = oracle.dequantize(ex[e].codes[1], ex[e].sf[1], ex[e].ts[1]).astype(np.float64)
        u = wu @ xh[t]
        bu = H * 2.0 ** -24 * (np.abs(wu) @ np.abs(xh[t]))
        if kind == "relu2":
            want = np.maximum(u, 0) ** 2
            bound = 2 * np.abs(u) * bu + bu ** 2 + 2 ** -23 * want
        else:
            wg = oracle.dequantize(ex[e].codes[0], ex[e].sf[0], ex[e].ts[0]).astype(np.float64)
            g = wg @ xh[t]
            bg = H * 2.0 ** -24 * (np.abs(wg) @ np.abs(xh[t]))
            want = np.array([_oai64(a, b, 7.0, 1.702) for a, b in zip(g, u)])
            # |d h / d g| <= (|u'| + 1) * 1.2 and |d h / d u| <= |g'| sigmoid: first-order bound
            gc = np.minimum(g, 7.0)
            uc = np.clip(u, -7.0, 7.0)
            bound = (np.abs(uc) + 1) * 1.2 * bg + np.abs(gc) * bu + 2 ** -20 * np.abs(want)
        assert np.all(np.abs(d["hf"][p] - want) <= bound + 1e-30), (kind, p)
