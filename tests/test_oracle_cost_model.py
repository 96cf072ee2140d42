"""Pins for the closed-form models of "不规则与流水化 AllToAll": the wave-time
model T(W) and its optimum W* (section "最优 wave 数") and the p95 link-load
approximation (section "长尾延迟问题")."""
import json
import math
import os

import numpy as np
import pytest

from combine_moe_route_17_b300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def test_printed_wave_optimum(orc):
    g = _load("wave_optimum.json")
    for M in g["M_bytes_readings"]:
        w_star = orc.optimal_waves(M, g["alpha_s"], g["beta_bytes_per_s"])
        assert round(w_star) == g["W_star_printed"]
        assert orc.optimal_waves_integer(M, g["alpha_s"], g["beta_bytes_per_s"]) == \
            g["W_star_printed"]
        lo, hi = g["measured_range_printed"]
        assert w_star > hi >= lo  # measured a little lower (expert compute not modelled)


def test_wave_time_minimum_by_calculus(orc):
    rng = np.random.default_rng(0)
    for _ in range(200):
        M = 10 ** rng.uniform(5, 10)
        alpha = 10 ** rng.uniform(-7, -4)
        beta = 10 ** rng.uniform(9, 12)
        ws = orc.optimal_waves(M, alpha, beta)
        # T(W*) = M/beta + 2 sqrt(M alpha / beta), by AM-GM on W alpha + M/(W beta)
        assert orc.wave_time(ws, M, alpha, beta) == pytest.approx(
            M / beta + 2 * math.sqrt(M * alpha / beta), rel=1e-12)
        h = ws * 1e-4
        left = orc.wave_time(ws - h, M, alpha, beta)
        right = orc.wave_time(ws + h, M, alpha, beta)
        mid = orc.wave_time(ws, M, alpha, beta)
        assert left >= mid and right >= mid
        wi = orc.optimal_waves_integer(M, alpha, beta, w_max=int(ws) + 50)
        assert wi in (math.floor(ws), math.ceil(ws), max(1, math.floor(ws)))


def test_wave_time_terms():
    import oracle
    # W=1: alpha + 2 M / beta (the last wave is the whole message)
    assert oracle.wave_time(1, 8.0, 1.0, 2.0) == 1.0 + 4.0 + 4.0
    assert oracle.wave_time(4, 8.0, 1.0, 2.0) == 4.0 + 4.0 + 1.0


def test_p95_page_formula_against_uniform_routing(orc):
    """Config-1 shape with i.i.d. N(0,1) logits: the send-count entries S[s][d]
    over 200 seeds.  The page's normal approximation (variance B p_bar) must
    over-predict the empirical p95 excess only mildly, and the exact variance
    of top-k routing without replacement must match it within 10%."""
    g = _load("p95_link_load.json")
    cfg = wl.CONFIGS["c1"]
    T, E, k, R = cfg.T, cfg.E, cfg.k, cfg.R
    B = (T // R) * k  # expert slots a source sends
    p_bar = 1.0 / R
    assert B * p_bar >= g["validity_floor_B_pbar"]
    m_avg = B * p_bar
    entries = []
    for seed in range(200):
        idx, _ = orc.route_topk(wl.make_logits(cfg, seed), k)
        entries.append(orc.send_counts(idx, E, R)["S"].ravel())
    S = np.concatenate(entries).astype(np.float64)
    assert S.mean() == pytest.approx(m_avg, rel=1e-12)  # rows sum to B exactly
    excess = np.percentile(S, 95) - S.mean()
    page = orc.p95_link_load_page(m_avg, B, p_bar) - m_avg
    assert page == pytest.approx(g["z95"] * math.sqrt(m_avg))
    exact = orc.p95_link_load_exact_excess(T // R, E, k, R)
    assert 0.75 <= excess / page <= 1.0
    assert abs(excess / exact - 1.0) <= 0.10
