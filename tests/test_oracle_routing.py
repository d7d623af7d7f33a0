"""Pins for the oracle's router (softmax -> top-k -> renormalise) and its stable permutation."""
import numpy as np
import pytest


def _brute_topk(row, k):
    order = sorted(range(len(row)), key=lambda e: (-float(row[e]), e))   # value desc, index asc
    return order[:k]


@pytest.mark.parametrize("T,E,k", [(16, 8, 2), (7, 128, 8), (33, 256, 8), (5, 64, 4), (3, 5, 5), (9, 6, 1)])
def test_router_matches_sorted_selection(orc, T, E, k):
    rng = np.random.default_rng(T * 1000 + E)
    logits = rng.normal(size=(T, E)).astype(np.float32)
    logits[0, :3] = logits[0, 3]           # a run of equal logits
    ids, w = orc.router(logits, k)
    for t in range(T):
        assert list(ids[t]) == _brute_topk(logits[t], k)
        # weights: softmax over all E restricted to the chosen k and renormalised (float64)
        p = np.exp(logits[t].astype(np.float64) - logits[t].max())
        p /= p.sum()
        sel = p[ids[t]] / p[ids[t]].sum()
        assert np.allclose(w[t], sel, rtol=2e-6, atol=1e-7)
        assert abs(float(w[t].astype(np.float64).sum()) - 1.0) < 1e-5
        assert all(w[t][j] >= w[t][j + 1] for j in range(k - 1))


def test_router_k1_weight_is_one(orc):
    rng = np.random.default_rng(11)
    logits = rng.normal(size=(50, 32)).astype(np.float32)
    ids, w = orc.router(logits, 1)
    assert np.all(w == 1.0)
    assert np.array_equal(ids[:, 0], np.argmax(logits, 1))


def test_router_k_equals_e_is_full_softmax(orc):
    rng = np.random.default_rng(12)
    logits = rng.normal(size=(20, 16)).astype(np.float32)
    ids, w = orc.router(logits, 16)
    for t in range(20):
        p = np.exp(logits[t].astype(np.float64) - logits[t].max())
        p /= p.sum()
        assert np.allclose(w[t], p[ids[t]], rtol=2e-6)
        assert sorted(ids[t]) == list(range(16))


def test_router_ties_lowest_index(orc):
    logits = np.zeros((3, 8), np.float32)
    logits[1] = [1, 3, 3, 0, 3, -1, 2, 2]
    logits[2] = [-0.0, 0.0, -0.0, 0.0, 5, 5, 5, 5]
    ids, w = orc.router(logits, 4)
    assert list(ids[0]) == [0, 1, 2, 3]
    assert np.all(w[0] == np.float32(0.25))
    assert list(ids[1]) == [1, 2, 4, 6]
    assert list(ids[2]) == [4, 5, 6, 7]


@pytest.mark.parametrize("T,E,k", [(16, 8, 2), (64, 128, 8), (40, 300, 3), (1, 4, 4), (0, 4, 2)])
def test_plan_invariants_and_bruteforce(orc, T, E, k):
    rng = np.random.default_rng(T + E + k)
    logits = rng.normal(size=(T, E)).astype(np.float32)
    logits[:, 1] += 3.0                      # one popular expert, several empty ones
    ids, _ = orc.router(logits, k) if T else (np.zeros((0, k), np.int32), None)
    counts, offsets, perm_src, inv = orc.plan(ids, E)
    R = T * k
    assert counts.sum() == R and offsets[0] == 0 and offsets[-1] == R
    assert np.array_equal(np.diff(offsets), counts)
    assert np.array_equal(counts, np.bincount(ids.reshape(-1), minlength=E))
    assert sorted(inv.tolist()) == list(range(R))            # a bijection
    flat = ids.reshape(-1)
    for a in range(R):
        p = inv[a]
        assert perm_src[p] == a // k
        assert offsets[flat[a]] <= p < offsets[flat[a] + 1]
    # brute force: stable sort of assignment indices by expert
    order = sorted(range(R), key=lambda a: (int(flat[a]), a))
    assert [perm_src[p] for p in range(R)] == [a // k for a in order]
