"""GPU parity of the W4A16 layer (BF16 activations as they are, NVFP4 weights decoded to BF16 in
the GEMMs, h rounded to BF16; "b12x" README, section "What's in here", moe: "W4A16 (BF16
activations, inline FP4 weight dequant - no activation-scale math)") through the C ABI against
the oracle's act_mode 1.

Bit-exact: router ids, counts, offsets, permutation.  The BF16 h: the tensor core sums the
products in its own order, so the FP32 g and u differ from the oracle's sequential sums by
rounding (relative ~sqrt(K) * 2^-24), and a value within that distance of a BF16 rounding
boundary rounds the other way: about one value in 10^3.  Asserted: at most 1% of the values
differ, each by at most one BF16 step of the oracle's value plus 2^-12 of the row's largest
|h| (values near zero, where g * sigmoid(g) * u or u^2 cancel to far below the row's scale,
move by more steps than one).  The output: relative L2 <= 5e-3 and max |err| <= 3e-2 * RMS."""
import numpy as np
import pytest
import torch

import oracle
import synth
from parity import assert_y_close, bf16_to_np_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import nvfp4_mixture_experts_softmax_gb300 as m
    m.lib()
    return m


def assert_hb_close(gpu_bits, ref_bits):
    g = (gpu_bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    r = (ref_bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    d = np.abs(g - r)
    mag = np.abs(r)
    ulp = np.exp2(np.floor(np.log2(np.maximum(mag, 1e-38))) - 7)
    row_max = np.abs(r).max(axis=1, keepdims=True)
    bound = ulp + 2.0 ** -12 * row_max
    frac = float(np.mean(d > 0)) if d.size else 0.0
    assert frac <= 1e-2, f"h (BF16): {frac:.2e} of the values differ"
    assert (d <= bound).all(), f"h (BF16): max |diff| / bound = {(d / bound).max():.2f}"
    return frac


def check_w4a16(moe, cs, T, activation="swiglu", limit=None, sample=None, logits=None):
    dev = "cuda"
    k = cs.top_k
    x = synth.gen_x(cs, T, device=dev)
    if logits is None:
        logits = synth.gen_logits(cs, T, device=dev)
    wg, wu, wd = synth.gen_all_experts(cs, device=dev)
    sh = synth.gen_shared(cs, device=dev) if cs.shared_inter else None
    gated = activation != "relu2"
    cfg = moe.make_config(cs.experts, cs.hidden, cs.inter, k, shared_inter=cs.shared_inter,
                          max_tokens=T, activation=activation, swiglu_limit=limit,
                          precision="w4a16")
    wbuf = moe.quantize_weights(cfg, wg if gated else None, wu, wd,
                                shared=None if sh is None else (sh[0] if gated else None, sh[1], sh[2]))
    ws = torch.empty(moe.workspace_size(cfg, T), dtype=torch.uint8, device=dev)
    y, dbg = moe.run(cfg, wbuf, x, logits, workspace=ws, debug=True)
    assert moe.last_device_status(ws) == 0
    g = {n: t.cpu() for n, t in dbg.items()}
    lg = logits.cpu().numpy()
    ids, w = oracle.router(lg, k)
    counts, offsets, perm_src, inv = oracle.plan(ids, cs.experts)
    assert np.array_equal(g["topk_ids"].numpy(), ids)
    assert np.array_equal(g["offsets"].numpy(), offsets)
    assert np.array_equal(g["perm_src"].numpy(), perm_src) and np.array_equal(g["inv"].numpy(), inv)
    toks = np.arange(T) if sample is None else sample
    experts = [None] * cs.experts
    for e in np.unique(ids[toks]):
        experts[e] = oracle.QuantExpert.from_bf16(wg[e].cpu() if gated else None, wu[e].cpu(),
                                                  wd[e].cpu())
    sho = None
    if sh is not None:
        sho = oracle.QuantExpert.from_bf16(sh[0].cpu() if gated else None, sh[1].cpu(), sh[2].cpu())
    xc = x.cpu()[toks]
    y_ref, od = oracle.moe_forward(None, None, None, lg[toks], experts, k, shared=sho,
                                   want_debug=True, act="bf16", x_bf16=xc, activation=activation,
                                   swiglu_limit=limit)
    hb = bf16_to_np_bits(g["hb"])
    rows_gpu = np.array([inv[t * k + j] for t in toks for j in range(k)])
    rows_ref = np.array([od["inv"][i * k + j] for i in range(len(toks)) for j in range(k)])
    assert_hb_close(hb[rows_gpu], od["hb"][rows_ref])
    if sh is not None:
        assert_hb_close(hb[T * k + toks], od["shb"])
    assert_y_close(y.float().cpu().numpy()[toks], oracle.bf16_bits_to_f32(y_ref))


@pytest.mark.parametrize("T", [1, 8, 64])
def test_w4a16_decode(moe, T):
    check_w4a16(moe, synth.CONFIGS["decode"], T)


def test_w4a16_tiny(moe):
    check_w4a16(moe, synth.CONFIGS["tiny"], 16)


@pytest.mark.parametrize("activation,limit", [("swiglu", None), ("relu2", None),
                                              ("swiglu_oai", 7.0), ("swiglu", 0.5)])
def test_w4a16_shared_expert_and_activations(moe, activation, limit):
    cs = synth.custom_config("w4a16_sh", 300, 512, 16, 4, 256, shared_inter=256, config_id=160)
    check_w4a16(moe, cs, 300, activation, limit)


def test_w4a16_one_expert_many_tiles(moe):
    """Every token on one expert (k = 1 of E = 2 with a planted logit): five 128-row tiles, the
    last one ragged."""
    cs = synth.custom_config("w4a16_pop", 600, 256, 2, 1, 256, config_id=161)
    check_w4a16(moe, cs, 600)



def test_w4a16_swapped_popular_expert(moe):
    """Batches of at most 64 tokens take the swapped-operand GEMMs (16-row token tiles): one
    expert holds all 64 tokens (four full tiles), the others a few rows each."""
    cs = synth.custom_config("w4a16_dpop", 64, 512, 8, 2, 256, config_id=170)
    lg = synth.gen_logits(cs, 64)
    lg[:, 5] += 50.0
    check_w4a16(moe, cs, 64, logits=lg.cuda())


@pytest.mark.parametrize("activation,limit", [("swiglu", None), ("relu2", None),
                                              ("swiglu_oai", 7.0)])
def test_w4a16_swapped_every_expert_ragged(moe, activation, limit):
    """k = E with 50 tokens: every expert and the shared one own four 16-row tiles, the last
    one of two rows."""
    cs = synth.custom_config("w4a16_dkes", 50, 512, 4, 4, 256, shared_inter=256,
                             config_id=171)
    check_w4a16(moe, cs, 50, activation, limit)

def test_w4a16_prefill_size_sampled(moe):
    cs = synth.CONFIGS["prefill"]
    T = cs.tokens[0]
    rng = np.random.default_rng(5)
    sample = np.sort(np.concatenate([[0, T - 1], rng.choice(np.arange(1, T - 1), 30, replace=False)]))
    check_w4a16(moe, cs, T, sample=sample)


def test_w4a16_refuses_quantised_input(moe):
    cs = synth.CONFIGS["tiny"]
    cfg = moe.make_config(cs.experts, cs.hidden, cs.inter, cs.top_k, precision="w4a16")
    wg, wu, wd = synth.gen_all_experts(cs, device="cuda")
    wbuf = moe.quantize_weights(cfg, wg, wu, wd)
    x = synth.gen_x(cs, 16, device="cuda")
    xq, xsf, ts = moe.quantize_act(x)
    with pytest.raises(RuntimeError, match="INVALID_ARG"):
        moe.run(cfg, wbuf, None, synth.gen_logits(cs, 16, device="cuda"), quantized=(xq, xsf, ts))
