"""The producer feeding the layer: already-quantised activations through moe_run_quantized.

* moe_quantize_act's output fed to moe_run_quantized gives moe_run's output on the same BF16 x:
  the same bits on the decode and small-batch paths (slot-order combine), at most one BF16 step
  apart on the general path (FP32 reductions in arbitrary order);
* RMSNorm + NVFP4 (moe_rmsnorm_quantize_act) -> moe_run_quantized matches the oracle's
  orc_rmsnorm_quantize -> moe_forward within the layer's output bounds, with routing and plan
  bit-exact ("nvfp4-megamoe-kernel compare pre-b1...master", sections "P4 - Fused RMSNorm + NVFP4
  quantize" and "P5": the norm's quantised output feeds the MoE without a BF16 round trip)."""
import numpy as np
import pytest
import torch

import oracle
import synth
from parity import assert_h_close, assert_y_close_layer, oracle_experts_from

pytestmark = pytest.mark.gpu

CASES = [("decode", 1), ("decode", 8), ("decode", 64), ("tiny", 16),
         ("small_general", 200), ("general", 3000)]


@pytest.fixture(scope="module")
def moe():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import nvfp4_mixture_experts_softmax_gb300 as m
    m.lib()
    return m


def _config(name):
    if name == "small_general":       # above the decode size, inside the one-block prologue
        return synth.custom_config("small_general", 200, 512, 16, 4, 256, shared_inter=256,
                                   config_id=180)
    if name == "general":
        return synth.custom_config("general_q", 3000, 1024, 32, 4, 512, config_id=181)
    return synth.CONFIGS[name]


def _layer(moe, cs, T):
    cfg = moe.make_config(cs.experts, cs.hidden, cs.inter, cs.top_k, shared_inter=cs.shared_inter,
                          max_tokens=T)
    wg, wu, wd = synth.gen_all_experts(cs, device="cuda")
    sh = synth.gen_shared(cs, device="cuda") if cs.shared_inter else None
    return cfg, moe.quantize_weights(cfg, wg, wu, wd, shared=sh), (wg, wu, wd, sh)


@pytest.mark.parametrize("name,T", CASES)
def test_quantized_input_gives_the_bf16_layer(moe, name, T):
    cs = _config(name)
    cfg, wbuf, _ = _layer(moe, cs, T)
    x = synth.gen_x(cs, T, device="cuda")
    lg = synth.gen_logits(cs, T, device="cuda")
    y = moe.run(cfg, wbuf, x, lg)
    xq, xsf, ts = moe.quantize_act(x)
    ws = torch.empty(moe.workspace_size(cfg, T), dtype=torch.uint8, device="cuda")
    yq = moe.run(cfg, wbuf, None, lg, workspace=ws, quantized=(xq, xsf, ts))
    assert moe.last_device_status(ws) == 0
    if moe.run_kernel_count(cfg, T) <= 5:            # decode and small-batch paths
        assert torch.equal(y, yq)
    else:
        # FP32 reductions in arbitrary order: the sum of k + 1 terms may differ by its rounding
        d = (y.float() - yq.float()).abs()
        mag = torch.maximum(y.float().abs(), yq.float().abs())
        ulp = torch.pow(2.0, torch.floor(torch.log2(torch.clamp(mag, min=1e-30))) - 7)
        bound = ulp + (cs.top_k + 1) * 2.0 ** -24 * 4 * float(y.float().abs().max())
        assert bool((d <= bound).all())


@pytest.mark.parametrize("name,T", CASES)
def test_rmsnorm_producer_into_layer_matches_oracle(moe, name, T):
    cs = _config(name)
    cfg, wbuf, (wg, wu, wd, sh) = _layer(moe, cs, T)
    x = synth.gen_x(cs, T, device="cuda")
    gamma = torch.from_numpy(np.random.default_rng(T).normal(1.0, 0.1, cs.hidden)
                             .astype(np.float32)).to(torch.bfloat16)
    lg = synth.gen_logits(cs, T, device="cuda")
    codes, sf, ts = moe.rmsnorm_quantize_act(x, gamma.cuda(), 1e-6)
    y, dbg = moe.run(cfg, wbuf, None, lg, quantized=(codes, sf, ts), debug=True)
    torch.cuda.synchronize()
    rc, rs, rts, st, _ = oracle.rmsnorm_quantize(x.cpu(), gamma, 1e-6)
    assert st == 0
    lgn = lg.cpu().numpy()
    ids, _ = oracle.router(lgn, cs.top_k)
    experts = oracle_experts_from(wg, wu, wd, ids)
    sho = oracle.QuantExpert.from_bf16(*[s.cpu() for s in sh]) if sh is not None else None
    y_ref, od = oracle.moe_forward(rc, rs, rts, lgn, experts, cs.top_k, shared=sho,
                                   want_debug=True)
    g = {n: t.cpu().numpy() for n, t in dbg.items()}
    assert np.array_equal(g["topk_ids"], od["ids"])
    assert np.array_equal(g["offsets"], od["offsets"]) and np.array_equal(g["inv"], od["inv"])
    assert np.array_equal(g["xq"], codes.cpu().numpy())       # the input, passed through
    assert g["ts_a"][0] == ts.item()
    assert_h_close(g["hq"][:T * cs.top_k], g["hsf"][:T * cs.top_k], od["hq"], od["hsf"])
    assert_y_close_layer(y.float().cpu().numpy(), oracle.bf16_bits_to_f32(y_ref), g, od,
                         np.arange(T), T, cs.top_k, experts, sho)


def test_quantized_input_argument_errors(moe):
    cs = synth.CONFIGS["tiny"]
    cfg, wbuf, _ = _layer(moe, cs, 16)
    lg = synth.gen_logits(cs, 16, device="cuda")
    xq, xsf, ts = moe.quantize_act(synth.gen_x(cs, 16, device="cuda"))
    with pytest.raises(RuntimeError, match="INVALID_ARG"):
        moe.run(cfg, wbuf, None, lg, quantized=(xq, xsf, None))
    bad_ts = torch.tensor([float("nan")], device="cuda")
    ws = torch.empty(moe.workspace_size(cfg, 16), dtype=torch.uint8, device="cuda")
    moe.run(cfg, wbuf, None, lg, workspace=ws, quantized=(xq, xsf, bad_ts))
    assert moe.last_device_status(ws) == -6
