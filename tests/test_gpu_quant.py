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
