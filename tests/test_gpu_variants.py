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
from parity import assert_h_close, assert_y_close, oracle_experts_from

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
