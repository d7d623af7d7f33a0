"""GPU parity of the W4A8 layer (MXFP4 weights, MXFP8 activations and intermediate, one E8M0
scale per 32, no tensor scales; "b12x" README, section "DeepSeek V4 Flash 0731 MoE
reproduction") through the C ABI against the oracle's act_mode 2.

Bit-exact: the MXFP4 weight codes and E8M0 scales (export), the MXFP8 codes and scales of x,
router ids, counts, offsets, permutation.  The MXFP8 codes of h: at most 0.1% differ, each by one
E4M3 step (scales likewise, one E8M0 step): the tensor core's FP32 accumulation order differs
from the oracle's, so a value within rounding noise of a boundary has two correct codes.  The
output: relative L2 <= 5e-3, and max |err| <= 3e-2 * RMS plus, for a token whose h blocks
differ, the change such a block can make (a quarter of the block's largest decoded value per
element, times the down projection's column magnitudes and the router weight)."""
import numpy as np
import pytest
import torch

import oracle
import synth
from parity import H_CODE_FRAC, Y_REL_L2, y_max_abs_bound

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import nvfp4_mixture_experts_softmax_gb300 as m
    m.lib()
    return m


def e4m3_rank(c):
    c = c.astype(np.int32)
    return np.where(c & 0x80, -(c & 0x7F), c & 0x7F)


def assert_mx8_close(gc, gs, rc, rs):
    d = np.abs(e4m3_rank(gc) - e4m3_rank(rc))
    ds = np.abs(gs.astype(np.int32) - rs.astype(np.int32))
    fc, fs = float(np.mean(d > 0)), float(np.mean(ds > 0))
    assert fc <= H_CODE_FRAC and d.max() <= 1, f"h codes: {fc:.2e} differ, max step {d.max()}"
    assert fs <= H_CODE_FRAC and ds.max() <= 1, f"h scales: {fs:.2e} differ, max step {ds.max()}"


def check_w4a8(moe, cs, T, activation="swiglu", limit=None, sample=None, logits=None):
    dev = "cuda"
    k, E = cs.top_k, cs.experts
    x = synth.gen_x(cs, T, device=dev)
    if logits is None:
        logits = synth.gen_logits(cs, T, device=dev)
    wg, wu, wd = synth.gen_all_experts(cs, device=dev)
    sh = synth.gen_shared(cs, device=dev) if cs.shared_inter else None
    gated = activation != "relu2"
    cfg = moe.make_config(E, cs.hidden, cs.inter, k, shared_inter=cs.shared_inter, max_tokens=T,
                          activation=activation, swiglu_limit=limit, precision="w4a8")
    wbuf = moe.quantize_weights(cfg, wg if gated else None, wu, wd,
                                shared=None if sh is None else (sh[0] if gated else None, sh[1], sh[2]))
    ws = torch.empty(moe.workspace_size(cfg, T), dtype=torch.uint8, device=dev)
    y, dbg = moe.run(cfg, wbuf, x, logits, workspace=ws, debug=True)
    assert moe.last_device_status(ws) == 0
    g = {n: t.cpu() for n, t in dbg.items()}
    lg = logits.cpu().numpy()
    # the activation quantiser and the routing, bit for bit
    xf = x.float().cpu().numpy()
    xc, xs = oracle.mx_quantize(xf, "e4m3")
    assert np.array_equal(g["xq"].numpy(), xc) and np.array_equal(g["xsf"].numpy(), xs)
    ids, w = oracle.router(lg, k)
    counts, offsets, perm_src, inv = oracle.plan(ids, E)
    assert np.array_equal(g["topk_ids"].numpy(), ids) and np.array_equal(g["inv"].numpy(), inv)
    toks = np.arange(T) if sample is None else sample
    experts = [None] * E
    for e in np.unique(ids[toks]):
        experts[e] = oracle.QuantExpertMX.from_bf16(wg[e].cpu() if gated else None, wu[e].cpu(),
                                                    wd[e].cpu())
    for e in np.unique(ids[toks])[:2]:          # the packed MXFP4 weights, bit for bit
        for m in (range(3) if gated else (1, 2)):
            c, s, t = moe.weights_export(cfg, wbuf, int(e), m)
            assert np.array_equal(c.cpu().numpy(), experts[e].codes[m])
            assert np.array_equal(s.cpu().numpy(), experts[e].sf[m]) and t.item() == 1.0
    sho = None
    if sh is not None:
        sho = oracle.QuantExpertMX.from_bf16(sh[0].cpu() if gated else None, sh[1].cpu(),
                                             sh[2].cpu())
    y_ref, od = oracle.moe_forward(None, None, None, lg[toks], experts, k, shared=sho,
                                   want_debug=True, act="mxfp8", x_bf16=x.cpu()[toks],
                                   activation=activation, swiglu_limit=limit)
    hq, hsf = g["hq"].numpy(), g["hsf"].numpy()
    rows_gpu = np.array([inv[t * k + j] for t in toks for j in range(k)])
    rows_ref = np.array([od["inv"][i * k + j] for i in range(len(toks)) for j in range(k)])
    assert_mx8_close(hq[rows_gpu], hsf[rows_gpu], od["hq"][rows_ref], od["hsf"][rows_ref])
    if sh is not None:
        assert_mx8_close(hq[T * k + toks], hsf[T * k + toks], od["shq"], od["shsf"])
    # the output, with the allowance for h blocks that differ
    yg = y.float().cpu().numpy()[toks].astype(np.float64)
    yr = oracle.bf16_bits_to_f32(y_ref).astype(np.float64)
    rel = np.linalg.norm(yg - yr) / np.linalg.norm(yr)
    assert rel <= Y_REL_L2, rel
    rms = np.sqrt(np.mean(yr ** 2))
    bound = y_max_abs_bound(yg, yr, rms)
    wd_cache = {}
    for i, t in enumerate(toks):
        slots = [(od["w"][i, j], inv[t * k + j], od["inv"][i * k + j], od["hq"], od["hsf"],
                  int(ids[t, j])) for j in range(k)]
        if sh is not None:
            slots.append((1.0, T * k + t, i, od["shq"], od["shsf"], -1))
        for wr, pg, pr, rq, rsf, e in slots:
            diff = (hq[pg] != rq[pr]).reshape(-1, 32).any(axis=1) | (hsf[pg] != rsf[pr])
            for b in np.nonzero(diff)[0]:
                if e not in wd_cache:
                    ex = sho if e < 0 else experts[e]
                    wd_cache[e] = oracle.mx_dequantize(ex.codes[2], ex.sf[2], "e2m1")
                vals = oracle.mx_dequantize(rq[pr][None, 32 * b:32 * b + 32],
                                            rsf[pr][None, b:b + 1], "e4m3")
                bound[i] += abs(wr) * 0.25 * np.abs(vals).max() * \
                    np.abs(wd_cache[e][:, 32 * b:32 * b + 32]).sum(axis=1)
    err = np.abs(yg - yr)
    assert (err <= bound).all(), f"y: max/rms {err.max() / rms:.3e}"


@pytest.mark.parametrize("T", [1, 8, 64])
def test_w4a8_decode(moe, T):
    check_w4a8(moe, synth.CONFIGS["decode"], T)


def test_w4a8_tiny(moe):
    check_w4a8(moe, synth.CONFIGS["tiny"], 16)


@pytest.mark.parametrize("activation,limit", [("swiglu", None), ("relu2", None),
                                              ("swiglu_oai", 7.0), ("swiglu", 0.5)])
def test_w4a8_shared_expert_and_activations(moe, activation, limit):
    cs = synth.custom_config("w4a8_sh", 300, 512, 16, 4, 256, shared_inter=256, config_id=162)
    check_w4a8(moe, cs, 300, activation, limit)



def test_w4a8_swapped_popular_expert(moe):
    """Batches of at most 64 tokens take the swapped-operand GEMMs (16-row token tiles): one
    expert holds all 64 tokens (four full tiles), the others a few rows each."""
    cs = synth.custom_config("w4a8_dpop", 64, 512, 8, 2, 256, config_id=172)
    lg = synth.gen_logits(cs, 64)
    lg[:, 5] += 50.0
    check_w4a8(moe, cs, 64, logits=lg.cuda())


@pytest.mark.parametrize("activation,limit", [("swiglu", None), ("relu2", None),
                                              ("swiglu_oai", 7.0)])
def test_w4a8_swapped_every_expert_ragged(moe, activation, limit):
    """k = E with 50 tokens: every expert and the shared one own four 16-row tiles, the last
    one of two rows."""
    cs = synth.custom_config("w4a8_dkes", 50, 512, 4, 4, 256, shared_inter=256,
                             config_id=173)
    check_w4a8(moe, cs, 50, activation, limit)

def test_w4a8_prefill_size_sampled(moe):
    cs = synth.CONFIGS["prefill"]
    T = cs.tokens[0]
    rng = np.random.default_rng(6)
    sample = np.sort(np.concatenate([[0, T - 1], rng.choice(np.arange(1, T - 1), 30, replace=False)]))
    check_w4a8(moe, cs, T, sample=sample)


def test_w4a8_config_errors(moe):
    bad = moe.make_config(8, 256, 512, 2, precision="w4a8")
    bad.flags |= moe.FLAG_ACT_BF16
    assert moe.config_check(bad) == -1
