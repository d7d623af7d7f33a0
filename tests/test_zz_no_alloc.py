"""moe_plan_static: the plan for callers that cannot allocate device memory.

Callers such as a plugin inside a host framework that owns all device allocations, or code
running while a memory pool is frozen, cannot hand the library a workspace.  moe_plan_static uses
a static per-device scratch array instead.  This file runs last (pytest collects it last) and
checks, through the C ABI, that two consecutive calls give what the workspace-taking moe_plan
gives, with the same tolerances as the other plan tests, and that an oversized problem is
rejected.  It passes alone in a fresh process and after the rest of the suite.
"""
import numpy as np
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import nvfp4_mixture_experts_softmax_gb300 as m
    m.lib()
    return m


def _same(a, b):
    for n in ("topk_ids", "counts", "offsets", "perm_src", "inv"):
        assert np.array_equal(a[n].cpu().numpy(), b[n].cpu().numpy()), n
    assert np.allclose(a["topk_w"].cpu().numpy(), b["topk_w"].cpu().numpy(), rtol=4e-7, atol=1e-9)


def test_static_plan_matches_workspace_plan_twice(moe):
    cases = [(synth.CONFIGS["decode"], 64), (synth.CONFIGS["prefill"], 8192),
             (synth.CONFIGS["skewed"], 16384)]
    for cs, T in cases:
        first = synth.gen_logits(cs, T, device="cuda")
        second = synth.gen_logits(cs, T, device="cuda", row0=T)
        for logits in (first, second):          # two calls in a row, different inputs
            want = moe.plan(logits, cs.top_k)
            got = moe.plan_static(logits, cs.top_k)
            torch.cuda.synchronize()
            _same(got, want)


def test_static_plan_rejects_oversized(moe):
    lg = torch.zeros(1, 1024, device="cuda")
    L = moe.lib()
    # 2^24 tokens at E = 1024 needs far more than the static scratch holds
    assert L.moe_plan_static(lg.data_ptr(), 1 << 24, 1024, 8, None, None, None, None, None, None,
                             None) == -3
