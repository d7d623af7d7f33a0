"""GPU parity of the router + plan: ids, counts, offsets and the permutation bit-exact against
the oracle; router weights within FP32 rounding of exp (device and host exp may differ by an
ulp)."""
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


def _check_plan(moe, logits, k):
    T, E = logits.shape
    out = moe.plan(logits.cuda(), k)
    torch.cuda.synchronize()
    lg = logits.cpu().numpy()
    ids, w = oracle.router(lg, k)
    counts, offsets, perm_src, inv = oracle.plan(ids, E)
    assert np.array_equal(out["topk_ids"].cpu().numpy(), ids)
    assert np.allclose(out["topk_w"].cpu().numpy(), w, rtol=4e-7, atol=1e-9)
    assert np.array_equal(out["counts"].cpu().numpy(), counts)
    assert np.array_equal(out["offsets"].cpu().numpy(), offsets)
    assert np.array_equal(out["perm_src"].cpu().numpy(), perm_src)
    assert np.array_equal(out["inv"].cpu().numpy(), inv)
    return counts


@pytest.mark.parametrize("name,T", [("tiny", 16), ("decode", 1), ("decode", 8), ("decode", 32),
                                    ("decode", 64), ("prefill", 8192), ("large", 4096),
                                    ("skewed", 16384)])
def test_plan_configs(moe, name, T):
    cfg = synth.CONFIGS[name]
    counts = _check_plan(moe, synth.gen_logits(cfg, T), cfg.top_k)
    if name == "skewed":
        assert 3500 <= counts.max() <= 4500 and counts.max() >= 5 * counts.min()  # Zipf skew


@pytest.mark.parametrize("T,E,k", [(1, 1, 1), (3, 5, 5), (65, 7, 3), (100, 300, 2), (130, 1024, 32),
                                   (77, 33, 16), (5000, 64, 1)])
def test_plan_ragged_shapes(moe, T, E, k):
    g = torch.Generator().manual_seed(T * 7 + E)
    _check_plan(moe, torch.randn(T, E, generator=g), k)


def test_plan_ties_and_popular_expert(moe):
    T, E = 200, 64
    g = torch.Generator().manual_seed(3)
    logits = torch.randn(T, E, generator=g)
    logits[:50] = torch.round(logits[:50])          # many exact ties
    logits[50:100] = 0.0                            # all equal: experts 0..k-1
    logits[100:150, 17] += 100.0                    # one expert takes every token
    logits[150:, ::2] = -0.0                        # signed zeros tie with +0
    logits[150:, 1::2] = 0.0
    _check_plan(moe, logits, 6)


def test_plan_empty(moe):
    out = moe.plan(torch.zeros(0, 8, device="cuda"), 2)
    torch.cuda.synchronize()
    assert out["counts"].sum().item() == 0 and out["offsets"].sum().item() == 0


def test_plan_bad_args(moe):
    with pytest.raises(RuntimeError, match="INVALID_ARG"):
        moe.plan(torch.randn(4, 8, device="cuda"), 9)     # k > E
