"""GPU parity of the whole layer (moe_run through the C ABI) against the oracle.

Bit-exact: activation codes / scales / tensor scale, router ids, counts, offsets, permutation.
Within the layer's bounds: the requantised intermediate (<= 0.1% codes off by one step) and the
output (relative L2 <= 5e-3, max |err| <= 3e-2 * RMS).
"""
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


def run_and_check(moe, cs, T, logits=None):
    dev = "cuda"
    k = cs.top_k
    x = synth.gen_x(cs, T, device=dev)
    if logits is None:
        logits = synth.gen_logits(cs, T, device=dev)
    wg, wu, wd = synth.gen_all_experts(cs, device=dev)
    sh = synth.gen_shared(cs, device=dev) if cs.shared_inter else None
    cfg = moe.make_config(cs.experts, cs.hidden, cs.inter, k, shared_inter=cs.shared_inter,
                          max_tokens=T)
    wbuf = moe.quantize_weights(cfg, wg, wu, wd, shared=sh)
    ws = torch.empty(moe.workspace_size(cfg, T), dtype=torch.uint8, device=dev)
    y, dbg = moe.run(cfg, wbuf, x, logits, workspace=ws, debug=True)
    assert moe.last_device_status(ws) == 0

    lg = logits.cpu().numpy()
    xq, xsf, ts_a, st = oracle.quantize_bf16(x.cpu())
    assert st == 0
    ids_o, _ = oracle.router(lg, k)
    experts = oracle_experts_from(wg, wu, wd, ids_o)
    sho = oracle.QuantExpert.from_bf16(*[s.cpu() for s in sh]) if sh is not None else None
    y_ref, od = oracle.moe_forward(xq, xsf, ts_a, lg, experts, k, shared=sho, want_debug=True)

    g = {n: t.cpu().numpy() for n, t in dbg.items()}
    assert g["ts_a"][0] == ts_a
    assert np.array_equal(g["xq"], xq) and np.array_equal(g["xsf"], xsf)
    assert np.array_equal(g["topk_ids"], od["ids"])
    assert np.allclose(g["topk_w"], od["w"], rtol=4e-7, atol=1e-9)
    assert np.array_equal(g["counts"], od["counts"])
    assert np.array_equal(g["offsets"], od["offsets"])
    assert np.array_equal(g["perm_src"], od["perm_src"])
    assert np.array_equal(g["inv"], od["inv"])
    R = T * k
    assert_h_close(g["hq"][:R], g["hsf"][:R], od["hq"], od["hsf"])
    if sh is not None:
        assert_h_close(g["hq"][R:], g["hsf"][R:], od["shq"], od["shsf"])
    rel, mx = assert_y_close(y.float().cpu().numpy(), oracle.bf16_bits_to_f32(y_ref))
    return y, rel, mx


@pytest.mark.parametrize("T", [16])
def test_tiny(moe, T):
    run_and_check(moe, synth.CONFIGS["tiny"], T)


@pytest.mark.parametrize("T", [1, 8, 32, 64])
def test_decode(moe, T):
    run_and_check(moe, synth.CONFIGS["decode"], T)


SMALL = [
    # several 128-row tiles per expert with a ragged last tile
    synth.custom_config("two_experts_many_rows", 300, 256, 2, 1, 256, config_id=120),
    # more experts than tokens: several experts stay empty
    synth.custom_config("empty_experts", 5, 256, 12, 1, 256, config_id=121),
    # k = E
    synth.custom_config("k_eq_e", 9, 256, 4, 4, 512, config_id=122),
    # shared expert
    synth.custom_config("shared", 20, 512, 6, 2, 256, shared_inter=256, config_id=123),
    # a single expert, a single token
    synth.custom_config("single", 1, 256, 1, 1, 256, config_id=124),
    # wider K and N than the tiny layer, ragged rows
    synth.custom_config("ragged_wide", 37, 1024, 16, 3, 768, config_id=125),
    # large enough for the multi-kernel path (chunked plan, reduction combine), with a shared expert
    synth.custom_config("general_path", 640, 1024, 16, 4, 256, shared_inter=256, config_id=127),
]


@pytest.mark.parametrize("cs", SMALL, ids=lambda c: c.name)
def test_small_shapes(moe, cs):
    run_and_check(moe, cs, cs.tokens[0])


def test_popular_expert_many_tiles(moe):
    cs = synth.custom_config("popular", 700, 512, 8, 2, 256, config_id=126)
    lg = synth.gen_logits(cs, 700)
    lg[:, 3] += 50.0      # expert 3 gets every token: 6 tiles of 128 rows
    run_and_check(moe, cs, 700, logits=lg.cuda())


def test_decode_popular_expert_multi_tile(moe):
    """Decode path with one expert taking all 64 tokens: four 16-row tiles of that expert."""
    cs = synth.custom_config("decode_popular", 64, 512, 8, 2, 256, config_id=128)
    lg = synth.gen_logits(cs, 64)
    lg[:, 5] += 50.0
    run_and_check(moe, cs, 64, logits=lg.cuda())


def test_decode_every_expert_multi_tile_with_shared(moe):
    """Decode path with k = E (every expert gets all 48 tokens: three tiles each) and a shared
    expert (three more tiles)."""
    cs = synth.custom_config("decode_k_eq_e_shared", 48, 512, 4, 4, 256, shared_inter=256,
                             config_id=129)
    run_and_check(moe, cs, 48)


def test_repeat_calls_bit_identical_on_decode_path(moe):
    """Decode-sized batches combine each token's stored rows in slot order: two calls give the
    same bits (a stale plan or a race between the GEMMs would show here)."""
    for name, T in (("tiny", 16), ("decode", 64), ("decode", 1)):
        cs = synth.CONFIGS[name]
        y1, _, _ = run_and_check(moe, cs, T)
        y2, _, _ = run_and_check(moe, cs, T)
        assert torch.equal(y1, y2), (name, T)


def test_repeat_calls_general_path_within_rounding(moe):
    """Large batches add the k routed contributions (and the shared one) into the token row with
    FP32 reductions in arbitrary order, so two calls may differ by the FP32 rounding of a sum of
    k + 1 terms, at most (k + 1) * 2^-24 times the sum of their magnitudes (taken here as 4x the
    output's maximum), plus one BF16 step of the result; and only for few values."""
    cs = synth.custom_config("general_repeat", 3000, 512, 16, 4, 256, shared_inter=256,
                             config_id=171)
    cfg = moe.make_config(cs.experts, cs.hidden, cs.inter, cs.top_k, shared_inter=256,
                          max_tokens=3000)
    assert moe.run_kernel_count(cfg, 3000) >= 6          # the general path
    wg, wu, wd = synth.gen_all_experts(cs, device="cuda")
    wbuf = moe.quantize_weights(cfg, wg, wu, wd, shared=synth.gen_shared(cs, device="cuda"))
    x = synth.gen_x(cs, 3000, device="cuda")
    lg = synth.gen_logits(cs, 3000, device="cuda")
    ys = [moe.run(cfg, wbuf, x, lg).float() for _ in range(3)]
    scale = float(ys[0].abs().max())
    for y in ys[1:]:
        d = (y - ys[0]).abs()
        mag = torch.maximum(y.abs(), ys[0].abs())
        ulp = torch.pow(2.0, torch.floor(torch.log2(torch.clamp(mag, min=1e-30))) - 7)
        bound = ulp + (cs.top_k + 1) * 2.0 ** -24 * 4 * scale
        assert bool((d <= bound).all()), float((d / bound).max())
        assert float((d > 0).float().mean()) <= 1e-2


def test_zero_tokens_and_errors(moe):
    cs = synth.CONFIGS["tiny"]
    cfg = moe.make_config(cs.experts, cs.hidden, cs.inter, cs.top_k)
    wg, wu, wd = synth.gen_all_experts(cs, device="cuda")
    wbuf = moe.quantize_weights(cfg, wg, wu, wd)
    x = torch.zeros(0, cs.hidden, dtype=torch.bfloat16, device="cuda")
    lg = torch.zeros(0, cs.experts, device="cuda")
    y = moe.run(cfg, wbuf, x, lg)
    assert y.shape == (0, cs.hidden)
    x = synth.gen_x(cs, 4, device="cuda")
    lg = synth.gen_logits(cs, 4, device="cuda")
    with pytest.raises(RuntimeError, match="INVALID_ARG"):
        moe.run(cfg, wbuf, x, lg, k=cs.top_k + 1)
    small_ws = torch.empty(1024, dtype=torch.uint8, device="cuda")
    with pytest.raises(RuntimeError, match="WORKSPACE_TOO_SMALL"):
        moe.run(cfg, wbuf, x, lg, workspace=small_ws)
    bad = moe.make_config(cs.experts, 200, cs.inter, cs.top_k)      # H not a multiple of 256
    with pytest.raises(RuntimeError, match="UNSUPPORTED_SHAPE"):
        moe.quantize_weights(bad, wg, wu, wd)


def test_cuda_graph_replay_matches_eager(moe):
    """The layer is recorded into a CUDA graph (no allocation, no host read inside moe_run) and
    the replays agree with an eager call; the pages check graph replay against eager the same
    way ("b12x" README, DeepSeek V4.1 Flash MoE benchmark)."""
    cs = synth.CONFIGS["decode"]
    T = 8
    x = synth.gen_x(cs, T, device="cuda")
    lg = synth.gen_logits(cs, T, device="cuda")
    wg, wu, wd = synth.gen_all_experts(cs, device="cuda")
    cfg = moe.make_config(cs.experts, cs.hidden, cs.inter, cs.top_k, max_tokens=T)
    wbuf = moe.quantize_weights(cfg, wg, wu, wd)
    ws = torch.empty(moe.workspace_size(cfg, T), dtype=torch.uint8, device="cuda")
    y_eager = moe.run(cfg, wbuf, x, lg, workspace=ws).clone()
    y = torch.empty_like(y_eager)
    timer = moe.StageTimer()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        moe.run(cfg, wbuf, x, lg, y=y, workspace=ws, timer=timer)
    for _ in range(3):
        y.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert moe.last_device_status(ws) == 0
        assert torch.equal(y, y_eager)      # the decode path is deterministic
        ms = timer.stage_ms()
        assert all(v >= 0 for v in ms.values()) and sum(ms.values()) > 0


def test_forced_timeout_is_reported_and_the_next_call_is_clean(moe):
    """A wait that runs out ends the call with MOE_ERR_DEVICE_TIMEOUT in the device status and
    leaves the context usable.  The hook keeps the decode prologue from raising its plan-ready
    flag, so the grouped-GEMM launch's bounded wait for it (about 2 s) expires before any copy is
    issued; the next call without the hook must be green and give the same bits as before."""
    cs = synth.CONFIGS["decode"]
    T = 8
    cfg = moe.make_config(cs.experts, cs.hidden, cs.inter, cs.top_k, max_tokens=T)
    wg, wu, wd = synth.gen_all_experts(cs, device="cuda")
    wbuf = moe.quantize_weights(cfg, wg, wu, wd)
    x = synth.gen_x(cs, T, device="cuda")
    lg = synth.gen_logits(cs, T, device="cuda")
    ws = torch.empty(moe.workspace_size(cfg, T), dtype=torch.uint8, device="cuda")
    y0 = moe.run(cfg, wbuf, x, lg, workspace=ws).clone()
    assert moe.last_device_status(ws) == 0
    moe.run(cfg, wbuf, x, lg, workspace=ws, inject=moe.MOE_INJECT_NO_PLAN_FLAG)
    assert moe.last_device_status(ws) == -5           # MOE_ERR_DEVICE_TIMEOUT
    y1 = moe.run(cfg, wbuf, x, lg, workspace=ws)
    assert moe.last_device_status(ws) == 0
    assert torch.equal(y0, y1)
