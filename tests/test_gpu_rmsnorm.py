"""GPU parity of RMSNorm + NVFP4 quantisation (moe_rmsnorm_quantize_act) against the oracle.

The oracle's mean square is the exact sum of squares rounded once to FP32; the kernel sums in
FP32 in its own order (8-element chunks, then a tree), whose relative error is at most
(7 + 5 + log2 J) * 2^-24 <= 18 * 2^-24 (J = 64 lanes' chunks at 16384 columns; every term is
non-negative).  Through ms = sum / cols, sqrt and the division, each row's r = 1/rms then differs
by at most about half that plus four roundings on each side: <= 2^-19 relative is asserted.  The
tensor scale max|y| / 2688 adds three roundings per side: <= 2^-18.  Codes and block scales
follow from r and ts, so only values within that distance of a rounding boundary can move: at
most 0.1% of them, each by one step (the criterion used for the requantised intermediate)."""
import numpy as np
import pytest
import torch

import oracle
import synth
from parity import assert_h_close

pytestmark = pytest.mark.gpu

R_REL = 2.0 ** -19
TS_REL = 2.0 ** -18


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


def check_against_oracle(moe, x, g, eps):
    codes, sf, ts, rr = moe.rmsnorm_quantize_act(x, g.cuda(), eps, want_rrms=True)
    torch.cuda.synchronize()
    rc, rs, rts, st, _, r_ref = oracle.rmsnorm_quantize(x.cpu(), g, eps, want_r=True)
    assert st == 0
    r_gpu = rr.cpu().numpy()
    rel = np.abs(r_gpu.astype(np.float64) - r_ref) / np.maximum(np.abs(r_ref), 1e-30)
    assert rel.max() <= R_REL, f"1/rms: max relative difference {rel.max():.3e}"
    assert abs(ts.item() - rts) <= TS_REL * rts, (ts.item(), rts)
    assert_h_close(codes.cpu().numpy(), sf.cpu().numpy(), rc, rs)
    return float(np.mean(r_gpu == r_ref)), ts.item() == rts


@pytest.mark.parametrize("rows,cols,eps", [(1, 2048, 1e-6), (64, 2048, 1e-6), (37, 1024, 1e-5),
                                           (5, 16384, 1e-6), (8192, 2048, 1e-6),
                                           (4096, 7168, 1e-6)])
def test_rmsnorm_quant_matches_oracle(moe, rows, cols, eps):
    cs = synth.custom_config("rms", rows, cols, 8, 1, 256, config_id=150)
    x = synth.gen_x(cs, rows, device="cuda")
    check_against_oracle(moe, x, _gamma(cols, rows), eps)


def test_rmsnorm_quant_wide_dynamic_range(moe):
    """Rows whose elements span 2^-20 .. 2^7 (where the order of an FP32 sum matters most)."""
    rng = np.random.default_rng(11)
    v = rng.standard_normal((256, 4096)) * np.exp2(rng.integers(-20, 8, (256, 4096)))
    x = torch.from_numpy(v.astype(np.float32)).to(torch.bfloat16).cuda()
    check_against_oracle(moe, x, _gamma(4096, 12), 1e-6)


def test_rmsnorm_quant_zero_rows_and_nonfinite(moe):
    x = torch.zeros(4, 256, dtype=torch.bfloat16, device="cuda")
    x[1] = 1.0
    g = _gamma(256, 7).cuda()
    codes, sf, ts = moe.rmsnorm_quantize_act(x, g, 1e-6)
    rc, rs, rts, _, _ = oracle.rmsnorm_quantize(x.cpu(), g.cpu(), 1e-6)
    # constant rows: every sum is exact on both sides, so everything is bit-exact
    assert ts.item() == rts and np.array_equal(codes.cpu().numpy(), rc)
    assert np.array_equal(sf.cpu().numpy(), rs)
    x[2, 5] = float("inf")
    ws = torch.empty(moe.lib().moe_rmsnorm_workspace_size(4), dtype=torch.uint8, device="cuda")
    moe.rmsnorm_quantize_act(x, g, 1e-6, workspace=ws)
    assert moe.last_device_status(ws) == -6
