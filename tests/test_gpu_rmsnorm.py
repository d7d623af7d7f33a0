"""GPU parity of RMSNorm + NVFP4 quantisation (moe_rmsnorm_quantize_act) against the oracle:
codes, block scales and the tensor scale bit-exact."""
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


def _gamma(cols, seed):
    g = np.random.default_rng(seed).normal(1.0, 0.1, cols).astype(np.float32)
    return torch.from_numpy(g).to(torch.bfloat16)


@pytest.mark.parametrize("rows,cols,eps", [(1, 2048, 1e-6), (64, 2048, 1e-6), (37, 1024, 1e-5),
                                           (8192, 2048, 1e-6), (4096, 7168, 1e-6)])
def test_rmsnorm_quant_bit_exact(moe, rows, cols, eps):
    cs = synth.custom_config("rms", rows, cols, 8, 1, 256, config_id=150)
    x = synth.gen_x(cs, rows, device="cuda")
    g = _gamma(cols, rows)
    codes, sf, ts = moe.rmsnorm_quantize_act(x, g.cuda(), eps)
    torch.cuda.synchronize()
    rc, rs, rts, st, _ = oracle.rmsnorm_quantize(x.cpu(), g, eps)
    assert st == 0
    assert ts.item() == rts
    assert np.array_equal(sf.cpu().numpy(), rs)
    assert np.array_equal(codes.cpu().numpy(), rc)


def test_rmsnorm_quant_zero_rows_and_nonfinite(moe):
    x = torch.zeros(4, 256, dtype=torch.bfloat16, device="cuda")
    x[1] = 1.0
    g = _gamma(256, 7).cuda()
    codes, sf, ts = moe.rmsnorm_quantize_act(x, g, 1e-6)
    rc, rs, rts, _, _ = oracle.rmsnorm_quantize(x.cpu(), g.cpu(), 1e-6)
    assert ts.item() == rts and np.array_equal(codes.cpu().numpy(), rc)
    assert np.array_equal(sf.cpu().numpy(), rs)
    x[2, 5] = float("inf")
    ws = torch.empty(moe.lib().moe_rmsnorm_workspace_size(4), dtype=torch.uint8, device="cuda")
    moe.rmsnorm_quantize_act(x, g, 1e-6, workspace=ws)
    assert moe.last_device_status(ws) == -6
