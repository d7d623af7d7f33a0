"""GPU parity of layers whose widths H and I are multiples of 32 but not of 256, through the C
ABI, against the oracle at the caller's widths.

The library runs such a layer at the next multiples of 256: zero rows and columns in the packed
weights, zero-padded copies of x (or of its codes and scales) and of the output rows in the
workspace.  Every padded term is an exact zero (a padded column of x meets zero weights; a
padded h feature is activation(0, 0) = 0, a zero block), so the bounds of the unpadded layer
apply unchanged: bit-exact router, permutation, activation codes and weight export; the layer's
bounds for h and y.  Widths of the pages that need it: the intermediate width 576 of DeepSeek
V4.1 and 1408 ("b12x" README, sections "DeepSeek V4.1 Flash MoE benchmark" and "What's in
here").  A shared expert of its own intermediate size runs the same way, at the larger of the two
widths."""
import numpy as np
import pytest
import torch

import oracle
import synth
from parity import assert_h_close, assert_y_close_layer
from test_gpu_producer_layer import _layer
from test_gpu_variants import check_activation, check_variant
from test_gpu_w4a8 import check_w4a8
from test_gpu_w4a16 import check_w4a16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import nvfp4_mixture_experts_softmax_gb300 as m
    m.lib()
    return m


def _cs(H, I, T, E=16, k=4, shared=True, cid=190):
    return synth.custom_config(f"pad_{H}_{I}", T, H, E, k, I, shared_inter=I if shared else 0,
                               config_id=cid)


SHAPES = [(288, 160), (544, 96), (2048, 576), (2080, 1408)]


@pytest.mark.parametrize("H,I", SHAPES)
@pytest.mark.parametrize("T", [3, 48, 300])
def test_padded_widths_decode_and_small_paths(moe, H, I, T):
    check_variant(moe, _cs(H, I, T), T, "softmax", None)


@pytest.mark.parametrize("H,I", [(288, 160), (2048, 576)])
def test_padded_widths_general_path(moe, H, I):
    # T * k above the one-block plan: the large-batch path.  Many tokens: the output is held to
    # the h-aware bound (a block of h that legitimately requantises one step apart moves its
    # token's output by more than the plain bound allows)
    T = 1500
    check_activation(moe, _cs(H, I, T, shared=False, cid=191), T, "swiglu")


@pytest.mark.parametrize("T", [40, 300])
def test_padded_widths_non_gated_experts_and_export(moe, T):
    check_activation(moe, _cs(544, 96, T, cid=192), T, "relu2")


@pytest.mark.parametrize("T", [40, 300])
def test_padded_widths_clamped_oai_activation(moe, T):
    check_activation(moe, _cs(288, 160, T, cid=193), T, "swiglu_oai", 1.5)


@pytest.mark.parametrize("T", [8, 300])
def test_padded_widths_w4a16(moe, T):
    check_w4a16(moe, _cs(288, 160, T, cid=194), T)


@pytest.mark.parametrize("H,I,T", [(288, 160, 8), (2048, 576, 300)])
def test_padded_widths_w4a8(moe, H, I, T):
    check_w4a8(moe, _cs(H, I, T, cid=195), T)


@pytest.mark.parametrize("T", [40, 1500])
def test_padded_widths_quantized_input(moe, T):
    """The quantised-input entry pads the caller's codes and scales as the BF16 entry pads x:
    both give the same output (bit for bit where the combine is deterministic)."""
    cs = _cs(544, 96, T, shared=False, cid=196)
    cfg, wbuf, _ = _layer(moe, cs, T)
    x = synth.gen_x(cs, T, device="cuda")
    lg = synth.gen_logits(cs, T, device="cuda")
    y = moe.run(cfg, wbuf, x, lg)
    xq, xsf, ts = moe.quantize_act(x)
    ws = torch.empty(moe.workspace_size(cfg, T), dtype=torch.uint8, device="cuda")
    yq = moe.run(cfg, wbuf, None, lg, workspace=ws, quantized=(xq, xsf, ts))
    assert moe.last_device_status(ws) == 0
    assert yq.shape == (T, 544)
    if moe.run_kernel_count(cfg, T) <= 5:
        assert torch.equal(y, yq)
    else:
        d = (y.float() - yq.float()).abs()
        mag = torch.maximum(y.float().abs(), yq.float().abs())
        ulp = torch.pow(2.0, torch.floor(torch.log2(torch.clamp(mag, min=1e-30))) - 7)
        bound = ulp + (cs.top_k + 1) * 2.0 ** -24 * 4 * float(y.float().abs().max())
        assert bool((d <= bound).all())


def test_padded_widths_weight_export_bit_exact(moe):
    """Every matrix of a routed and of the shared expert comes back from the padded packing as
    the oracle quantises it at the caller's widths."""
    cs = _cs(2080, 1408, 4, E=4, k=2, cid=197)
    cfg, wbuf, (wg, wu, wd, sh) = _layer(moe, cs, 4)
    for e, mats in ((3, (wg[3], wu[3], wd[3])), (-1, sh)):
        ref = oracle.QuantExpert.from_bf16(*[m.cpu() for m in mats])
        for m in range(3):
            c, s, t = moe.weights_export(cfg, wbuf, e, m)
            assert np.array_equal(c.cpu().numpy(), ref.codes[m])
            assert np.array_equal(s.cpu().numpy(), ref.sf[m])
            assert t.item() == ref.ts[m]


# ---- a shared expert of its own intermediate size (the routed and the shared intermediates both
# run at the larger one rounded up to a multiple of 256; debug rows of h are that wide)

def check_shared_width(moe, H, I, Is, T, cid, activation="swiglu"):
    cs = synth.custom_config(f"shw_{H}_{I}_{Is}", T, H, 16, 4, I, shared_inter=Is,
                             config_id=cid)
    dev, k = "cuda", cs.top_k
    gated = activation != "relu2"
    x = synth.gen_x(cs, T, device=dev)
    logits = synth.gen_logits(cs, T, device=dev)
    wg, wu, wd = synth.gen_all_experts(cs, device=dev)
    sh = synth.gen_shared(cs, device=dev)
    cfg = moe.make_config(cs.experts, H, I, k, shared_inter=Is, max_tokens=T,
                          activation=activation)
    wbuf = moe.quantize_weights(cfg, wg if gated else None, wu, wd,
                                shared=(sh[0] if gated else None, sh[1], sh[2]))
    y, dbg = moe.run(cfg, wbuf, x, logits, debug=True)
    torch.cuda.synchronize()
    lg = logits.cpu().numpy()
    xq, xsf, ts_a, _ = oracle.quantize_bf16(x.cpu())
    ids_o, _ = oracle.router(lg, k)
    experts = [None] * cs.experts
    for e in np.unique(ids_o):
        experts[e] = oracle.QuantExpert.from_bf16(wg[e].cpu() if gated else None, wu[e].cpu(),
                                                  wd[e].cpu())
    sho = oracle.QuantExpert.from_bf16(sh[0].cpu() if gated else None, sh[1].cpu(), sh[2].cpu())
    y_ref, od = oracle.moe_forward(xq, xsf, ts_a, lg, experts, k, shared=sho, want_debug=True,
                                   activation=activation)
    g = {n: t.cpu().numpy() for n, t in dbg.items()}
    R, Ih = T * k, max(I, Is)
    assert g["hq"].shape[1] == Ih // 2
    # each expert's rows at its own width, then zero codes and zero scales
    assert not g["hq"][:R, I // 2:].any() and not g["hsf"][:R, I // 16:].any()
    assert not g["hq"][R:, Is // 2:].any() and not g["hsf"][R:, Is // 16:].any()
    assert np.array_equal(g["topk_ids"], od["ids"]) and np.array_equal(g["inv"], od["inv"])
    assert_h_close(g["hq"][:R, :I // 2], g["hsf"][:R, :I // 16], od["hq"], od["hsf"])
    assert_h_close(g["hq"][R:, :Is // 2], g["hsf"][R:, :Is // 16], od["shq"], od["shsf"])
    gv = dict(g)
    gv["hq"] = [g["hq"][r, :(I if r < R else Is) // 2] for r in range(g["hq"].shape[0])]
    gv["hsf"] = [g["hsf"][r, :(I if r < R else Is) // 16] for r in range(g["hsf"].shape[0])]
    assert_y_close_layer(y.float().cpu().numpy(), oracle.bf16_bits_to_f32(y_ref), gv, od,
                         np.arange(T), T, k, experts, sho)
    for m in range(3):             # the shared expert's matrices come back at its own width
        if m == 0 and not gated:
            continue
        c, s, t = moe.weights_export(cfg, wbuf, -1, m)
        assert np.array_equal(c.cpu().numpy(), sho.codes[m])
        assert np.array_equal(s.cpu().numpy(), sho.sf[m]) and t.item() == sho.ts[m]


@pytest.mark.parametrize("H,I,Is", [(2048, 512, 1024), (288, 160, 96), (512, 256, 640)])
@pytest.mark.parametrize("T", [5, 300, 1500])
def test_shared_expert_of_its_own_width(moe, H, I, Is, T):
    check_shared_width(moe, H, I, Is, T, cid=198)


@pytest.mark.parametrize("T", [5, 300])
def test_shared_expert_of_its_own_width_non_gated(moe, T):
    check_shared_width(moe, 544, 96, 224, T, cid=199, activation="relu2")
