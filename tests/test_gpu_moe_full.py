"""GPU parity at the full sizes of the prefill, large (+ shared expert) and Zipf-skewed
workloads, in the launch configuration the benchmark times.  Whole-tensor bit-exact checks where
the oracle is cheap (activation quantiser, router, permutation, sampled experts' weights) and
per-token checks of the layer output and the requantised intermediate on sampled tokens."""
import numpy as np
import pytest
import torch

import oracle
import synth
from parity import assert_h_close, assert_y_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import nvfp4_mixture_experts_softmax_gb300 as m
    m.lib()
    return m


@pytest.mark.parametrize("name,nsample", [("prefill", 12), ("skewed", 8), ("large", 3)])
def test_full_size_sampled(moe, name, nsample):
    cs = synth.CONFIGS[name]
    T, k, E = cs.tokens[0], cs.top_k, cs.experts
    dev = "cuda"
    x = synth.gen_x(cs, T, device=dev)
    logits = synth.gen_logits(cs, T, device=dev)
    wg, wu, wd = synth.gen_all_experts(cs, device=dev)
    sh = synth.gen_shared(cs, device=dev) if cs.shared_inter else None
    cfg = moe.make_config(E, cs.hidden, cs.inter, k, shared_inter=cs.shared_inter, max_tokens=T)
    wbuf = moe.quantize_weights(cfg, wg, wu, wd, shared=sh)
    ws = torch.empty(moe.workspace_size(cfg, T), dtype=torch.uint8, device=dev)
    y, dbg = moe.run(cfg, wbuf, x, logits, workspace=ws, debug=True)
    assert moe.last_device_status(ws) == 0
    g = {n: t.cpu().numpy() for n, t in dbg.items()}

    # whole-tensor bit-exact stages
    xq, xsf, ts_a, st = oracle.quantize_bf16(x.cpu())
    assert st == 0 and g["ts_a"][0] == ts_a
    assert np.array_equal(g["xq"], xq) and np.array_equal(g["xsf"], xsf)
    lg = logits.cpu().numpy()
    ids, w = oracle.router(lg, k)
    counts, offsets, perm_src, inv = oracle.plan(ids, E)
    assert np.array_equal(g["topk_ids"], ids)
    assert np.allclose(g["topk_w"], w, rtol=4e-7, atol=1e-9)
    assert np.array_equal(g["counts"], counts) and np.array_equal(g["offsets"], offsets)
    assert np.array_equal(g["perm_src"], perm_src) and np.array_equal(g["inv"], inv)

    # sampled tokens: first, last, the busiest expert's first token, and seeded random ones
    rng = np.random.default_rng(cs.config_id)
    busiest = int(np.argmax(counts))
    first_busy = int(perm_src[offsets[busiest]])
    toks = sorted(set([0, T - 1, first_busy] + rng.choice(T, nsample, replace=False).tolist()))
    toks = np.array(toks[:nsample + 3])
    used = np.unique(ids[toks])
    experts = [None] * E
    for e in used:
        experts[e] = oracle.QuantExpert.from_bf16(wg[e].cpu(), wu[e].cpu(), wd[e].cpu())
        if e in (used[0], used[-1]):   # the packed weights of a few experts, bit-exact
            for m, W in enumerate((wg[e], wu[e], wd[e])):
                c, s, t = moe.weights_export(cfg, wbuf, int(e), m)
                assert t.item() == experts[e].ts[m]
                assert np.array_equal(c.cpu().numpy(), experts[e].codes[m])
                assert np.array_equal(s.cpu().numpy(), experts[e].sf[m])
    sho = oracle.QuantExpert.from_bf16(*[s.cpu() for s in sh]) if sh is not None else None
    y_ref, od = oracle.moe_forward(xq[toks], xsf[toks], ts_a, lg[toks], experts, k, shared=sho,
                                   want_debug=True)
    yg = y.float().cpu().numpy()[toks]
    assert_y_close(yg, oracle.bf16_bits_to_f32(y_ref))
    # intermediate rows of the sampled assignments
    rows_gpu = np.array([inv[t * k + j] for t in toks for j in range(k)])
    rows_ref = np.array([od["inv"][i * k + j] for i in range(len(toks)) for j in range(k)])
    assert_h_close(g["hq"][rows_gpu], g["hsf"][rows_gpu], od["hq"][rows_ref], od["hsf"][rows_ref])
    if sh is not None:
        R = T * k
        assert_h_close(g["hq"][R + toks], g["hsf"][R + toks], od["shq"], od["shsf"])
