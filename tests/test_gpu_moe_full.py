"""GPU parity at the full sizes of the prefill, large (+ shared expert) and Zipf-skewed
workloads, in the launch configuration the benchmark times.

Whole-tensor bit-exact checks where the oracle is cheap (activation quantiser, router,
permutation) and per-token checks of the layer output and the requantised intermediate on tokens
chosen from the plan: at least one compared token in every 128-row tile of expert-ordered rows
(the GEMMs' M tiles, the shared expert's included), plus the token of the last row of the last,
ragged tile of each of the five busiest experts.  Every expert that any compared token uses is
quantised by the oracle and its packed weights are compared bit for bit.  The oracle runs on
all host cores (its OpenMP build, whose bits equal the single-threaded build's)."""
import concurrent.futures as cf

import numpy as np
import pytest
import torch

import oracle
import synth
from parity import assert_h_close, assert_y_close_h_aware

pytestmark = pytest.mark.gpu

TILE = 128


@pytest.fixture(scope="module")
def moe():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import nvfp4_mixture_experts_softmax_gb300 as m
    m.lib()
    oracle.use_threads(None)
    yield m
    oracle.use_threads(1)


def covering_tokens(counts, offsets, perm_src, inv, T, k, shared):
    """Tokens such that every TILE-row tile of every segment (expert, then the shared expert's T
    rows) holds a row of one of them, plus the last row of the five busiest experts."""
    E = len(counts)
    tiles = []                       # (first row, end row) in the permuted row space
    for e in range(E):
        for r0 in range(int(offsets[e]), int(offsets[e + 1]), TILE):
            tiles.append((r0, min(r0 + TILE, int(offsets[e + 1]))))
    R = T * k
    tile_of = np.empty(R, np.int64)
    for i, (a, b) in enumerate(tiles):
        tile_of[a:b] = i
    covered = np.zeros(len(tiles), bool)
    chosen = []
    for i, (a, b) in enumerate(tiles):
        if covered[i]:
            continue
        t = int(perm_src[b - 1])      # the tile's last row (the ragged end for a last tile)
        chosen.append(t)
        covered[tile_of[inv[t * k:(t + 1) * k]]] = True
    for e in np.argsort(-counts, kind="stable")[:5]:
        chosen.append(int(perm_src[offsets[e + 1] - 1]))
    toks = set(chosen)
    if shared:                       # the shared expert's rows are the tokens in order
        toks.update(range(0, T, TILE))
        toks.add(T - 1)
    return np.array(sorted(toks)), len(tiles) + (-(-T // TILE) if shared else 0)


@pytest.mark.parametrize("name", ["prefill", "skewed", "large"])
def test_full_size_every_tile(moe, name):
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

    toks, ntiles = covering_tokens(counts, offsets, perm_src, inv, T, k, sh is not None)
    used = np.unique(ids[toks])
    # oracle quantisation of every expert the compared tokens use (threads: the C calls release
    # the interpreter lock), and the packed weights of each of them bit for bit
    def quant(e):
        return oracle.QuantExpert.from_bf16(wg[e].cpu(), wu[e].cpu(), wd[e].cpu())

    with cf.ThreadPoolExecutor(4) as ex:
        qs = dict(zip(used.tolist(), ex.map(quant, used.tolist())))
    experts = [qs.get(e) for e in range(E)]
    for e in used:
        for m in range(3):
            c, s, t = moe.weights_export(cfg, wbuf, int(e), m)
            assert t.item() == experts[e].ts[m]
            assert np.array_equal(c.cpu().numpy(), experts[e].codes[m])
            assert np.array_equal(s.cpu().numpy(), experts[e].sf[m])
    sho = oracle.QuantExpert.from_bf16(*[s.cpu() for s in sh]) if sh is not None else None
    y_ref, od = oracle.moe_forward(xq[toks], xsf[toks], ts_a, lg[toks], experts, k, shared=sho,
                                   want_debug=True)
    # intermediate rows of the compared tokens' assignments (and shared-expert rows)
    rows_gpu = np.array([inv[t * k + j] for t in toks for j in range(k)])
    rows_ref = np.array([od["inv"][i * k + j] for i in range(len(toks)) for j in range(k)])
    assert_h_close(g["hq"][rows_gpu], g["hsf"][rows_gpu], od["hq"][rows_ref], od["hsf"][rows_ref])
    R = T * k
    if sh is not None:
        assert_h_close(g["hq"][R + toks], g["hsf"][R + toks], od["shq"], od["shsf"])
    # the output, allowing for the h codes that differ by one step
    wd_cache = {}

    def down(e):
        def get():
            if e not in wd_cache:
                ex = sho if e < 0 else experts[e]
                wd_cache[e] = oracle.dequantize(ex.codes[2], ex.sf[2], ex.ts[2])
            return wd_cache[e]
        return get

    rows = []
    for i, t in enumerate(toks):
        slots = []
        for j in range(k):
            pg, pr = inv[t * k + j], od["inv"][i * k + j]
            slots.append((od["w"][i, j], g["hq"][pg], g["hsf"][pg], od["hq"][pr], od["hsf"][pr],
                          down(int(ids[t, j]))))
        if sh is not None:
            slots.append((1.0, g["hq"][R + t], g["hsf"][R + t], od["shq"][i], od["shsf"][i],
                          down(-1)))
        rows.append(slots)
    yg = y.float().cpu().numpy()[toks]
    rel, mx, nflip = assert_y_close_h_aware(yg, oracle.bf16_bits_to_f32(y_ref), rows)
    print(f"{name}: {len(toks)} tokens cover {ntiles} tiles, {len(used)} experts; "
          f"rel_l2 {rel:.2e}, max/rms {mx:.2e}, {nflip} tokens with a differing h block")
