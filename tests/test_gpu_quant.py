"""GPU parity of the NVFP4 quantisers (activations and weights): bit-exact against the oracle."""
import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import nvfp4_mixture_experts_softmax_gb300 as m
    m.lib()
    return m


def _check_act(moe, x):
    codes, sf, ts = moe.quantize_act(x.cuda())
    torch.cuda.synchronize()
    rc, rs, rts, st = oracle.quantize_bf16(x.cpu())
    assert st == 0
    assert ts.item() == rts
    assert np.array_equal(sf.cpu().numpy(), rs)
    assert np.array_equal(codes.cpu().numpy(), rc)


@pytest.mark.parametrize("name,T", [("tiny", 16), ("decode", 1), ("decode", 8), ("decode", 64),
                                    ("prefill", 8192), ("large", 4096), ("skewed", 16384)])
def test_act_quant_configs(moe, name, T):
    cfg = synth.CONFIGS[name]
    x = synth.gen_x(cfg, T, device="cuda")
    _check_act(moe, x)


def test_act_quant_edge_cases(moe):
    g = torch.Generator().manual_seed(0)
    # ragged (one row, a few blocks), magnitudes over many binades, ties and tiny values
    x = (torch.randn(3, 48, generator=g) * torch.exp(torch.randn(3, 48, generator=g) * 4))
    _check_act(moe, x.to(torch.bfloat16))
    # negative values that round to zero, exact zeros, a zero block, subnormal-ish block scales
    x = torch.randn(5, 64, generator=g)
    x[0] = 0.0
    x[1, :16] = -1e-3
    x[2, 0] = 1000.0
    x[3, 16:32] = torch.tensor([-0.0] * 16)
    _check_act(moe, x.to(torch.bfloat16))
    # all-zero tensor: ts 0, every scale and code 0
    _check_act(moe, torch.zeros(4, 32, dtype=torch.bfloat16))
    # a hand-worked row (tests/golden/nvfp4_row_example.txt)
    from conftest import read_kv
    kv = read_kv("nvfp4_row_example.txt")
    row = torch.tensor([float(v) for v in kv["x"]]).to(torch.bfloat16).reshape(1, -1)
    codes, sf, ts = moe.quantize_act(row.cuda())
    assert ts.item() == float(kv["ts"][0])
    assert sf.cpu().numpy().tobytes().hex() == "".join(kv["sf"])
    assert codes.cpu().numpy().tobytes().hex() == "".join(kv["codes"])


def test_act_quant_nonfinite_status(moe):
    x = torch.randn(4, 64).to(torch.bfloat16).cuda()
    x[2, 5] = float("nan")
    ws = torch.empty(moe.lib().moe_act_workspace_size(4, 64), dtype=torch.uint8, device="cuda")
    moe.quantize_act(x, workspace=ws)
    assert moe.last_device_status(ws) == -6
    x[2, 5] = 1.0
    moe.quantize_act(x, workspace=ws)
    assert moe.last_device_status(ws) == 0


def test_act_quant_host_errors(moe):
    x = torch.randn(4, 40).to(torch.bfloat16).cuda()   # cols not a multiple of 16
    with pytest.raises(RuntimeError, match="INVALID_ARG"):
        moe.quantize_act(x)


@pytest.mark.parametrize("cfg_name,shared", [("tiny", False), ("tiny_shared", True)])
def test_weight_quant_bit_exact(moe, cfg_name, shared):
    if cfg_name == "tiny":
        cs = synth.CONFIGS["tiny"]
    else:
        cs = synth.custom_config("tiny_shared", 4, 256, 6, 2, 256, shared_inter=256, config_id=110)
    wg, wu, wd = synth.gen_all_experts(cs, device="cuda")
    sh = synth.gen_shared(cs, device="cuda") if shared else None
    cfg = moe.make_config(cs.experts, cs.hidden, cs.inter, cs.top_k, shared_inter=cs.shared_inter)
    wbuf = moe.quantize_weights(cfg, wg, wu, wd, shared=sh)
    experts = list(range(cs.experts)) + ([-1] if shared else [])
    for e in experts:
        mats = (sh if e == -1 else (wg[e], wu[e], wd[e]))
        for m in range(3):
            codes, sf, ts = moe.weights_export(cfg, wbuf, e, m)
            rc, rs, rts, st = oracle.quantize_bf16(mats[m].cpu())
            assert st == 0
            assert ts.item() == rts, (e, m)
            assert np.array_equal(sf.cpu().numpy(), rs), (e, m)
            assert np.array_equal(codes.cpu().numpy(), rc), (e, m)


def test_weight_quant_decode_sampled(moe):
    cs = synth.CONFIGS["decode"]
    wg, wu, wd = synth.gen_all_experts(cs, device="cuda")
    cfg = moe.make_config(cs.experts, cs.hidden, cs.inter, cs.top_k)
    wbuf = moe.quantize_weights(cfg, wg, wu, wd)
    for e in (0, 1, 63, 127):
        for m, W in enumerate((wg[e], wu[e], wd[e])):
            codes, sf, ts = moe.weights_export(cfg, wbuf, e, m)
            rc, rs, rts, _ = oracle.quantize_bf16(W.cpu())
            assert ts.item() == rts
            assert np.array_equal(sf.cpu().numpy(), rs) and np.array_equal(codes.cpu().numpy(), rc)


def test_act_quant_every_bf16_every_scale(moe):
    """Every finite BF16 value against every E4M3 block scale, bit-exact against the oracle.

    The tensor's max is 2688, so the tensor scale is exactly 1 and a block whose max is
    6*decode(sf) gets scale sf exactly (both divisions exact); the block's other 15 elements run
    over every BF16 value v with |v| <= 6*decode(sf).  This covers every quotient the encoder can
    meet at each scale, including those within an ulp of an E2M1 rounding boundary, so any
    difference between the GPU's quotient and the IEEE division shows up as a code mismatch."""
    bits = np.arange(1 << 16, dtype=np.uint32)
    allv = (bits << 16).view(np.float32)
    allv = allv[np.isfinite(allv)]
    dec = torch.arange(1, 127, dtype=torch.uint8).view(torch.float8_e4m3fn).float().numpy()
    blocks = [np.array([2688.0] + [0.0] * 15, dtype=np.float32)]   # fixes the tensor scale at 1
    for d in dec:
        bamax = np.float32(6.0) * np.float32(d)
        vals = allv[np.abs(allv) <= bamax]
        pad = (-len(vals)) % 15
        vals = np.concatenate([vals, np.zeros(pad, dtype=np.float32)]).reshape(-1, 15)
        blk = np.concatenate([np.full((len(vals), 1), bamax, dtype=np.float32), vals], axis=1)
        blocks.append(blk.reshape(-1))
    flat = np.concatenate(blocks)
    cols = 4096
    flat = np.concatenate([flat, np.zeros((-len(flat)) % cols, dtype=np.float32)])
    x = torch.from_numpy(flat.reshape(-1, cols)).to(torch.bfloat16)
    assert torch.equal(x.float(), torch.from_numpy(flat.reshape(-1, cols)))   # all exact in BF16
    codes, sf, ts = moe.quantize_act(x.cuda())
    torch.cuda.synchronize()
    rc, rs, rts, st = oracle.quantize_bf16(x)
    assert st == 0 and rts == 1.0 and ts.item() == 1.0
    assert np.array_equal(sf.cpu().numpy(), rs)
    assert np.array_equal(codes.cpu().numpy(), rc)


def boundary_blocks(A: float, nblk: int, seed: int):
    """BF16 rows [nblk, 16] whose tensor maximum is A (a non-power-of-two value) and whose
    elements sit on and around b * S for every E2M1 rounding boundary b, S being the block's
    decoded scale times the tensor scale: the quotients x / S that the encoder divides fall on,
    just below and just above the boundaries (at BF16 resolution), a small share of them within
    one FP32 step of a boundary.  Also returns the host-side quotients, for counting those."""
    rng = np.random.default_rng(seed)
    bounds = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])
    ts = np.float32(A) / np.float32(2688.0)
    # block maxima M in (A/64, A]: BF16 values with random significands
    M = torch.from_numpy((A * np.exp2(-rng.uniform(0, 6, nblk))).astype(np.float32))
    M = M.to(torch.bfloat16).float().numpy()
    M[0] = A
    t = (M / np.float32(6.0)).astype(np.float32) / ts
    sf = torch.from_numpy(t.astype(np.float32)).to(torch.float8_e4m3fn).float().numpy()
    S = (sf * ts).astype(np.float32)
    x = np.zeros((nblk, 16), np.float32)
    x[:, 0] = M
    b = bounds[rng.integers(0, 7, (nblk, 15))]
    c = torch.from_numpy((b * S[:, None]).astype(np.float32)).to(torch.bfloat16)
    step = torch.from_numpy(rng.integers(-1, 2, (nblk, 15)).astype(np.int16))
    bits = c.view(torch.int16) + step                 # BF16 neighbours (all values positive)
    v = bits.view(torch.bfloat16).float().numpy()
    sign = np.where(rng.random((nblk, 15)) < 0.5, -1.0, 1.0).astype(np.float32)
    x[:, 1:] = v * sign
    q = np.abs(x[:, 1:].astype(np.float64)) / S[:, None].astype(np.float64)
    return torch.from_numpy(x).to(torch.bfloat16), q, b


def test_act_quant_quotients_at_e2m1_boundaries_non_power_of_two_scale(moe):
    """The encoder's quotient x / S comes from a reciprocal, a product and one correction step;
    on inputs built so that x / S falls on and next to every E2M1 rounding boundary, with tensor
    scales whose significands are not powers of two (so S has a full 24-bit significand), the
    codes must equal the oracle's IEEE-division codes bit for bit."""
    near = 0
    ties = 0
    for i, A in enumerate((3.140625, 0.0107421875, 77.5, 1234.0, 5.96875e-3, 0.83984375)):
        A = float(torch.tensor(A).to(torch.bfloat16).float())
        x, q, b = boundary_blocks(A, 1 << 16, seed=40 + i)
        _check_act(moe, x)
        d = np.abs(q - b)
        ties += int((d == 0).sum())
        near += int(((d > 0) & (d <= np.spacing(b.astype(np.float32)).astype(np.float64))).sum())
    # the inputs reach the cases the correction step exists for
    assert ties > 0 and near > 0, (ties, near)
