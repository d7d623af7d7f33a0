"""GPU parity of the router and activation variants through the C ABI against the oracle: the
sqrt-softplus router with a per-expert selection bias, and the clamped SwiGLU
silu(min(g, L)) * clamp(u, -L, L) ("vllm.cpp docs/STATUS.md", paragraph "W6 sqrtsoftplus +
hash-routed MoE"; "nvfp4-megamoe-kernel compare pre-b1...master", sections "Dense Router (L3+)"
and "Nvfp4MoE (Routed Experts)").

Bit-exact: router ids, counts, offsets, permutation, activation codes.  Weights: relative 2e-6
(the score's exp / log1p come from different math libraries on the two sides, an ulp apart).
Within the layer's bounds: the requantised h and the output."""
import numpy as np
import pytest
import torch

import oracle
import synth
from parity import assert_h_close, assert_y_close, assert_y_close_layer, oracle_experts_from

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import nvfp4_mixture_experts_softmax_gb300 as m
    m.lib()
    return m


def check_variant(moe, cs, T, router, limit, bias_scale=0.3):
    dev = "cuda"
    k = cs.top_k
    x = synth.gen_x(cs, T, device=dev)
    logits = synth.gen_logits(cs, T, device=dev)
    wg, wu, wd = synth.gen_all_experts(cs, device=dev)
    sh = synth.gen_shared(cs, device=dev) if cs.shared_inter else None
    bias = None
    if router == "sqrtsoftplus":
        bias = (np.random.default_rng(cs.config_id).standard_normal(cs.experts) * bias_scale)
        bias = bias.astype(np.float32)
    cfg = moe.make_config(cs.experts, cs.hidden, cs.inter, k, shared_inter=cs.shared_inter,
                          max_tokens=T, router=router, swiglu_limit=limit)
    wbuf = moe.quantize_weights(cfg, wg, wu, wd, shared=sh)
    if bias is not None:
        moe.set_router_bias(cfg, wbuf, torch.from_numpy(bias))
    ws = torch.empty(moe.workspace_size(cfg, T), dtype=torch.uint8, device=dev)
    y, dbg = moe.run(cfg, wbuf, x, logits, workspace=ws, debug=True)
    assert moe.last_device_status(ws) == 0

    lg = logits.cpu().numpy()
    xq, xsf, ts_a, st = oracle.quantize_bf16(x.cpu())
    ids_o, _ = oracle.router(lg, k, router, bias)
    experts = oracle_experts_from(wg, wu, wd, ids_o)
    sho = oracle.QuantExpert.from_bf16(*[s.cpu() for s in sh]) if sh is not None else None
    y_ref, od = oracle.moe_forward(xq, xsf, ts_a, lg, experts, k, shared=sho, want_debug=True,
                                   router_mode=router, router_bias=bias, swiglu_limit=limit)
    g = {n: t.cpu().numpy() for n, t in dbg.items()}
    assert np.array_equal(g["xq"], xq) and np.array_equal(g["xsf"], xsf)
    assert np.array_equal(g["topk_ids"], od["ids"])
    np.testing.assert_allclose(g["topk_w"], od["w"], rtol=2e-6, atol=1e-9)
    assert np.array_equal(g["counts"], od["counts"])
    assert np.array_equal(g["offsets"], od["offsets"])
    assert np.array_equal(g["perm_src"], od["perm_src"])
    R = T * k
    assert_h_close(g["hq"][:R], g["hsf"][:R], od["hq"], od["hsf"])
    if sh is not None:
        assert_h_close(g["hq"][R:], g["hsf"][R:], od["shq"], od["shsf"])
    assert_y_close(y.float().cpu().numpy(), oracle.bf16_bits_to_f32(y_ref))
    return g, od


VARIANTS = [("sqrtsoftplus", None), ("softmax", "small"), ("sqrtsoftplus", 10.0),
            ("sqrtsoftplus", "small")]


def _limit(limit, cs):
    # a limit that clamps often: g and u are about N(0, 0.02 * sqrt(H)) for these inputs
    return 0.25 * 0.02 * np.sqrt(cs.hidden) if limit == "small" else limit


@pytest.mark.parametrize("router,limit", VARIANTS)
@pytest.mark.parametrize("T", [8, 64])
def test_decode_variants(moe, router, limit, T):
    cs = synth.CONFIGS["decode"]
    check_variant(moe, cs, T, router, _limit(limit, cs))


@pytest.mark.parametrize("router,limit", VARIANTS)
def test_tiny_variants(moe, router, limit):
    cs = synth.CONFIGS["tiny"]
    check_variant(moe, cs, 16, router, _limit(limit, cs))


@pytest.mark.parametrize("router,limit", VARIANTS)
def test_general_path_variants(moe, router, limit):
    cs = synth.custom_config("general_path_v", 640, 1024, 16, 4, 256, shared_inter=256,
                             config_id=130)
    check_variant(moe, cs, 640, router, _limit(limit, cs))


def test_bias_changes_the_selection(moe):
    """A large bias on one expert makes every token pick it (the selection sees the bias),
    while its weight stays its own unbiased score share."""
    cs = synth.CONFIGS["decode"]
    T = 8
    dev = "cuda"
    x = synth.gen_x(cs, T, device=dev)
    logits = synth.gen_logits(cs, T, device=dev)
    wg, wu, wd = synth.gen_all_experts(cs, device=dev)
    cfg = moe.make_config(cs.experts, cs.hidden, cs.inter, cs.top_k, max_tokens=T,
                          router="sqrtsoftplus")
    wbuf = moe.quantize_weights(cfg, wg, wu, wd)
    bias = torch.zeros(cs.experts)
    bias[77] = 50.0
    moe.set_router_bias(cfg, wbuf, bias)
    ws = torch.empty(moe.workspace_size(cfg, T), dtype=torch.uint8, device=dev)
    _, dbg = moe.run(cfg, wbuf, x, logits, workspace=ws, debug=True)
    ids = dbg["topk_ids"].cpu().numpy()
    w = dbg["topk_w"].cpu().numpy()
    assert np.all(ids[:, 0] == 77)
    ids_o, w_o = oracle.router(logits.cpu().numpy(), cs.top_k, "sqrtsoftplus", bias.numpy())
    assert np.array_equal(ids, ids_o)
    np.testing.assert_allclose(w, w_o, rtol=2e-6)
    assert np.all(w[:, 0] < 0.5)


# ---- ReLU2 (non-gated experts) and SwiGLU-OAI ("b12x" README, "What's in here", moe: "with
# SiLU/ReLU2/SwiGLU-OAI activations")

def check_activation(moe, cs, T, activation, limit=None, alpha=1.702):
    dev = "cuda"
    k = cs.top_k
    x = synth.gen_x(cs, T, device=dev)
    logits = synth.gen_logits(cs, T, device=dev)
    wg, wu, wd = synth.gen_all_experts(cs, device=dev)
    sh = synth.gen_shared(cs, device=dev) if cs.shared_inter else None
    gated = activation != "relu2"
    cfg = moe.make_config(cs.experts, cs.hidden, cs.inter, k, shared_inter=cs.shared_inter,
                          max_tokens=T, activation=activation, swiglu_limit=limit,
                          swiglu_alpha=alpha)
    # a non-gated layer never reads its gate matrices: pass none
    wbuf = moe.quantize_weights(cfg, wg if gated else None, wu, wd,
                                shared=None if sh is None else (sh[0] if gated else None, sh[1], sh[2]))
    ws = torch.empty(moe.workspace_size(cfg, T), dtype=torch.uint8, device=dev)
    y, dbg = moe.run(cfg, wbuf, x, logits, workspace=ws, debug=True)
    assert moe.last_device_status(ws) == 0
    lg = logits.cpu().numpy()
    xq, xsf, ts_a, _ = oracle.quantize_bf16(x.cpu())
    ids_o, _ = oracle.router(lg, k)
    experts = [None] * cs.experts
    for e in np.unique(ids_o):
        experts[e] = oracle.QuantExpert.from_bf16(wg[e].cpu() if gated else None, wu[e].cpu(),
                                                  wd[e].cpu())
    sho = None
    if sh is not None:
        sho = oracle.QuantExpert.from_bf16(sh[0].cpu() if gated else None, sh[1].cpu(), sh[2].cpu())
    y_ref, od = oracle.moe_forward(xq, xsf, ts_a, lg, experts, k, shared=sho, want_debug=True,
                                   activation=activation, swiglu_limit=limit, swiglu_alpha=alpha)
    g = {n: t.cpu().numpy() for n, t in dbg.items()}
    assert np.array_equal(g["topk_ids"], od["ids"]) and np.array_equal(g["inv"], od["inv"])
    R = T * k
    assert_h_close(g["hq"][:R], g["hsf"][:R], od["hq"], od["hsf"])
    if sh is not None:
        assert_h_close(g["hq"][R:], g["hsf"][R:], od["shq"], od["shsf"])
    assert_y_close_layer(y.float().cpu().numpy(), oracle.bf16_bits_to_f32(y_ref), g, od,
                         np.arange(T), T, k, experts, sho)
    if not gated:     # the packed up matrix of an expert, bit for bit; the gate is refused
        e = int(ids_o[0, 0])
        c, s, t = moe.weights_export(cfg, wbuf, e, 1)
        assert np.array_equal(c.cpu().numpy(), experts[e].codes[1])
        assert np.array_equal(s.cpu().numpy(), experts[e].sf[1]) and t.item() == experts[e].ts[1]
        with pytest.raises(RuntimeError, match="INVALID_ARG"):
            moe.weights_export(cfg, wbuf, e, 0)


ACTS = [("relu2", None), ("swiglu_oai", 7.0), ("swiglu_oai", "small")]


@pytest.mark.parametrize("activation,limit", ACTS)
@pytest.mark.parametrize("T", [1, 8, 64])
def test_decode_activations(moe, activation, limit, T):
    cs = synth.CONFIGS["decode"]
    check_activation(moe, cs, T, activation, _limit(limit, cs))


@pytest.mark.parametrize("activation,limit", ACTS)
def test_tiny_activations_with_shared_expert(moe, activation, limit):
    cs = synth.custom_config("tiny_act_sh", 16, 256, 8, 2, 512, shared_inter=512, config_id=131)
    check_activation(moe, cs, 16, activation, _limit(limit, cs))


@pytest.mark.parametrize("activation,limit", ACTS)
@pytest.mark.parametrize("T", [200, 640])
def test_general_and_small_path_activations(moe, activation, limit, T):
    cs = synth.custom_config("general_path_act", T, 1024, 16, 4, 256, shared_inter=256,
                             config_id=132)
    check_activation(moe, cs, T, activation, _limit(limit, cs))


def test_activation_config_errors(moe):
    cs = synth.CONFIGS["tiny"]
    bad = moe.make_config(cs.experts, cs.hidden, cs.inter, cs.top_k, activation="relu2")
    bad.flags |= moe.FLAG_SWIGLU_CLAMP                          # two activations at once
    assert moe.config_check(bad) == -1
    oai = moe.make_config(cs.experts, cs.hidden, cs.inter, cs.top_k, activation="swiglu_oai",
                          swiglu_limit=7.0)
    oai.swiglu_alpha = float("inf")
    assert moe.config_check(oai) == -1
