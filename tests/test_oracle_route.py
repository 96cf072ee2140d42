"""Pins for the oracle's gating: softmax(TopK(logits, k)), ties toward the
lower expert index, optional group-limited routing.

Gating definition: MoE system-optimisation survey (crad.ict.ac.cn), section
1.1, eq. (2); constrained vs free routing: "不规则与流水化 AllToAll", section
"EP 不规则 a2a 的来源".
"""
import itertools
import math

import numpy as np
import pytest
import torch


def _key(l, e):
    # larger is better: higher logit, then lower index (Python's -0.0 == 0.0)
    return (float(l[e]), -e)


def brute_topk(l, k, allowed=None):
    """The k-subset whose keys, sorted best-first, are lexicographically
    largest; returned best-first."""
    E = len(l)
    cand = [e for e in range(E) if allowed is None or allowed[e]]
    best = None
    for sub in itertools.combinations(cand, k):
        keys = sorted((_key(l, e) for e in sub), reverse=True)
        if best is None or keys > best[0]:
            best = (keys, sub)
    return [-kk[1] for kk in best[0]]


def brute_group_topk(l, k, n_groups, topk_groups, group_topn):
    E = len(l)
    gsz = E // n_groups
    scores = []
    for g in range(n_groups):
        top = brute_topk(l[g * gsz:(g + 1) * gsz], group_topn)
        s = np.float32(l[g * gsz + top[0]])
        for e in top[1:]:
            s = np.float32(s + np.float32(l[g * gsz + e]))
        scores.append(s)
    best = None
    for sub in itertools.combinations(range(n_groups), topk_groups):
        keys = sorted(((float(scores[g]), -g) for g in sub), reverse=True)
        if best is None or keys > best[0]:
            best = (keys, sub)
    kept = set(best[1])
    allowed = [(e // gsz) in kept for e in range(E)]
    return brute_topk(l, k, allowed)


@pytest.mark.parametrize("E,k", [(4, 1), (5, 2), (6, 3), (8, 2), (8, 4), (7, 7)])
def test_topk_matches_brute_force_with_many_ties(orc, E, k):
    rng = np.random.default_rng(E * 10 + k)
    T = 300
    lg = rng.integers(-2, 3, size=(T, E)).astype(np.float32)  # heavy ties
    lg[rng.random((T, E)) < 0.2] = -0.0
    idx, _ = orc.route_topk(lg, k)
    for t in range(T):
        assert list(idx[t]) == brute_topk(lg[t], k), (t, lg[t])


def test_topk_matches_stable_library_sort(orc):
    rng = np.random.default_rng(7)
    lg = rng.standard_normal((512, 64)).astype(np.float32)
    lg[:, 10] = lg[:, 20]  # exact duplicates
    lg[:, 33] = lg[:, 3]
    k = 8
    idx, _ = orc.route_topk(lg, k)
    ref = torch.sort(torch.from_numpy(lg), dim=1, descending=True, stable=True).indices[:, :k]
    assert np.array_equal(idx, ref.numpy().astype(np.int32))


def test_all_equal_and_signed_zero_ties(orc):
    E, k = 16, 5
    idx, w = orc.route_topk(np.zeros((3, E), np.float32), k)
    assert (idx == np.arange(k)).all()
    assert np.allclose(w, 1.0 / k, atol=1e-7)
    lg = np.array([[-0.0, 0.0, -0.0, 0.0]], np.float32)
    idx, _ = orc.route_topk(lg, 3)
    assert list(idx[0]) == [0, 1, 2]
    lg = np.array([[1.0, -0.0, 2.0, 0.0, 2.0]], np.float32)
    idx, _ = orc.route_topk(lg, 4)
    assert list(idx[0]) == [2, 4, 0, 1]


@pytest.mark.parametrize("E,G,keep,topn,k", [(8, 4, 2, 2, 3), (12, 4, 2, 2, 3), (12, 3, 2, 1, 4),
                                            (16, 8, 3, 2, 4), (9, 3, 1, 3, 3)])
def test_group_limited_matches_brute_force(orc, E, G, keep, topn, k):
    rng = np.random.default_rng(E + G * 100 + keep)
    T = 200
    lg = rng.integers(-3, 4, size=(T, E)).astype(np.float32) * np.float32(0.5)
    lg[rng.random((T, E)) < 0.1] = -0.0
    idx, _ = orc.route_topk(lg, k, G, keep, topn)
    for t in range(T):
        assert list(idx[t]) == brute_group_topk(lg[t], k, G, keep, topn), (t, lg[t])


def test_group_limited_with_equal_groups_is_topk_over_first_groups(orc):
    rng = np.random.default_rng(3)
    E, G, keep, k = 32, 8, 3, 5
    gsz = E // G
    pat = rng.standard_normal((64, gsz)).astype(np.float32)
    lg = np.tile(pat, (1, G))  # every group scores the same
    idx, _ = orc.route_topk(lg, k, G, keep, 2)
    masked = lg.copy()
    masked[:, keep * gsz:] = -1e30
    ref, _ = orc.route_topk(masked, k)
    assert np.array_equal(idx, ref)


def test_group_score_is_an_fp32_sum(orc):
    big = np.float32(2.0 ** 23)  # fp32 spacing is 1 here and 2 above 2^24
    one = np.float32(1.0)
    # group 0 = {2^23, 2^23} scores 2^24 exactly; group 1 = {2^23+1, 2^23}
    # scores 2^24+1, which fp32 rounds (tie to even) to 2^24: the groups tie
    # and the lower one is kept.  A wider sum would keep group 1.
    lg = np.array([[big, big, big + one, big]], np.float32)
    idx, _ = orc.route_topk(lg, 1, 2, 1, 2)
    assert idx[0, 0] == 0
    # group 1 = {2^23+2, 2^23} scores 2^24+2 exactly and wins
    lg = np.array([[big, big, big + np.float32(2.0), big]], np.float32)
    idx, _ = orc.route_topk(lg, 2, 2, 1, 2)
    assert list(idx[0]) == [2, 3]


def test_weights_are_the_renormalised_softmax(orc):
    rng = np.random.default_rng(11)
    lg = (rng.standard_normal((400, 32)) * 3).astype(np.float32)
    for k in (1, 2, 6, 8, 16):
        idx, w = orc.route_topk(lg, k)
        assert np.all(np.abs(w.astype(np.float64).sum(1) - 1.0) <= 1e-6)
        assert np.all(np.diff(w, axis=1) <= 0)  # selection order = descending weight
        if k == 1:
            assert (w == 1.0).all()
    # k = 2 reduces to the logistic function of the logit gap
    idx, w = orc.route_topk(lg, 2)
    a = lg[np.arange(400), idx[:, 0]].astype(np.float64)
    b = lg[np.arange(400), idx[:, 1]].astype(np.float64)
    logistic = np.array([1.0 / (1.0 + math.exp(bb - aa)) for aa, bb in zip(a, b)])
    assert np.allclose(w[:, 0], logistic, atol=6e-8, rtol=0)


def test_rejects_non_finite_logits(orc):
    lg = np.zeros((2, 4), np.float32)
    lg[1, 2] = np.nan
    with pytest.raises(ValueError):
        orc.route_topk(lg, 2)
