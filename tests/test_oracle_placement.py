"""Pins of the oracle's placement and concentration summaries.

Greedy placement: MoE survey (crad.ict.ac.cn), section 4.2.2 "设备负载均衡" --
experts in descending order of load, each to the least-loaded device, every
device holding the same number of experts.  Ties (not on the pages): the lower
expert index first, the lower rank among equally loaded ranks.

Fitted symmetric-Dirichlet alpha: the third summary of the send-count matrix in
the DODOCO summary (section "方法论"); the pages give no fit.  Reading: method
of moments for a Dirichlet-multinomial of the N slots over E experts."""
import math

import numpy as np
import pytest

import oracle


@pytest.mark.parametrize("c,R,placement,relabel", [
    # worked by hand: order e0(5) e2(4) e3(2) e1(1); e3 joins rank 1 (4 < 5),
    # e1 must join rank 0 (rank 1 is full)
    ([5, 1, 4, 2], 2, [0, 0, 1, 1], [0, 1, 2, 3]),
    # order e1(9) e3(8) e5(7) e2(3) e4(2) e0(1): loads end 10, 10, 10
    ([1, 9, 3, 8, 2, 7], 3, [0, 0, 2, 1, 1, 2], [1, 0, 5, 2, 3, 4]),
    # all equal: index order, the lower rank on equal loads
    ([3, 3, 3, 3], 2, [0, 1, 0, 1], [0, 2, 1, 3]),
])
def test_hand_worked_placements(c, R, placement, relabel):
    got = oracle.place_greedy(np.array(c), R)
    assert got["placement"].tolist() == placement
    assert got["relabel"].tolist() == relabel


def test_placement_invariants():
    rng = np.random.default_rng(1)
    for E, R in ((16, 4), (64, 8), (128, 16), (256, 32), (128, 64)):
        c = rng.integers(0, 5000, E)
        got = oracle.place_greedy(c, R)
        per = E // R
        assert np.bincount(got["placement"], minlength=R).tolist() == [per] * R
        assert sorted(got["relabel"].tolist()) == list(range(E))
        assert np.array_equal(got["relabel"] // per, got["placement"])


def test_greedy_balances_a_perfectly_balanceable_case():
    """Loads that the greedy pairs exactly: the largest with the smallest."""
    c = np.array([10, 9, 8, 7, 3, 2, 1, 0])
    got = oracle.place_greedy(c, 4)
    loads = np.bincount(got["placement"], weights=c, minlength=4)
    assert loads.tolist() == [10.0, 10.0, 10.0, 10.0]
    assert oracle.placement_gini(c, got["placement"], 4)["gini"] == 0.0


def test_contiguous_placement_gini_matches_the_statistics():
    rng = np.random.default_rng(2)
    for E, R in ((16, 4), (64, 8), (256, 32)):
        c = rng.integers(0, 3000, E).astype(np.int32)
        ref = oracle.imbalance_stats(c, R, 1, R)  # T and k only enter max/mean
        g = oracle.placement_gini(c, np.arange(E) // (E // R), R)
        assert (g["gini_num"], g["gini_den"]) == (ref["gini_num"], ref["gini_den"])
        assert g["gini"] == ref["gini"]


def test_alpha_limits():
    assert oracle.dirichlet_alpha(np.array([12, 0, 0, 0])) == 0.0
    assert oracle.dirichlet_alpha(np.array([7, 7, 7, 7])) == math.inf
    assert oracle.dirichlet_alpha(np.zeros(8, np.int32)) == math.inf


def test_alpha_solves_the_moment_equation():
    """The share variance of a Dirichlet-multinomial,
    (1/E)(1-1/E)(N + E a)/(N (1 + E a)), equated to the observed one and
    solved in floating point from the shares, gives the oracle's alpha."""
    rng = np.random.default_rng(3)
    for E in (16, 64, 256):
        p = rng.dirichlet(np.full(E, 0.7))
        c = rng.multinomial(200000, p).astype(np.int32)
        N = c.sum()
        q = c / N
        v = np.mean((q - 1.0 / E) ** 2)
        u = (1.0 / E) * (1.0 - 1.0 / E)
        A = N * (u - v) / (v * N - u)
        assert oracle.dirichlet_alpha(c) == pytest.approx(A / E, rel=1e-9)


@pytest.mark.parametrize("alpha", [0.1, 1.0, 10.0])
def test_alpha_recovers_the_generating_concentration(alpha):
    rng = np.random.default_rng(int(alpha * 100))
    E, N = 256, 1_000_000
    est = []
    for _ in range(40):
        p = rng.dirichlet(np.full(E, alpha))
        est.append(oracle.dirichlet_alpha(rng.multinomial(N, p).astype(np.int32)))
    assert np.exp(np.mean(np.log(est))) == pytest.approx(alpha, rel=0.1)
