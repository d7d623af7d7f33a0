"""The expert-sharing decode workloads (shared_0 ... shared_100): the planted routing has the
unique-expert counts the pages print for six tokens at top-6, no expert twice within a token, and
the oracle's router recovers it exactly from the generated logits."""
import os

import numpy as np
import pytest

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "expert_sharing_counts.txt")


def _golden():
    rows = []
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                a, b = line.split()
                rows.append((int(a), int(b)))
    return rows


@pytest.mark.parametrize("share,unique", _golden())
def test_six_token_counts_match_the_pages(share, unique):
    cs = synth.custom_config("share6", 6, 256, 64, 6, 256, config_id=140)
    assert synth.sharing_unique_experts(6, 6, share, 64) == unique
    ids = synth.sharing_routing(cs, 6, share).numpy()
    assert len(np.unique(ids)) == unique
    for row in ids:
        assert len(set(row.tolist())) == 6


@pytest.mark.parametrize("T", [4, 5, 6, 8])
@pytest.mark.parametrize("share", [0, 20, 40, 60, 80, 100])
def test_router_recovers_the_planted_routing(T, share):
    cs = synth.CONFIGS["decode"]
    lg = synth.gen_sharing_logits(cs, T, share).numpy()
    ids, w = oracle.router(lg, cs.top_k)
    assert np.array_equal(ids, synth.sharing_routing(cs, T, share).numpy())
    assert len(np.unique(ids)) == synth.sharing_unique_experts(T, cs.top_k, share, cs.experts)
    assert np.all(np.diff(w, axis=1) < 0)         # planted slot order: strictly decreasing
