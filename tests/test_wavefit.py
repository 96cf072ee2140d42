"""The fit of the wave-pipeline cost model T(W) = W*alpha + M/beta + M/(W*beta)
("不规则与流水化 AllToAll", section "最优 wave 数") used by the wave-scan
measurement: it recovers alpha and beta from model times, its optimum agrees
with the oracle's (itself pinned to the page's worked example), and it
reports a failed fit instead of a meaningless optimum."""
import math

import numpy as np
import pytest

from combine_moe_route_17_b300 import wavefit
from oracle import cost_model as cm


@pytest.mark.parametrize("alpha,beta,M", [(1e-6, 50e9, 16e6), (3e-6, 5e12, 4.0e8),
                                          (8e-6, 6.4e12, 4.3e9)])
def test_recovers_alpha_beta_from_model_times(alpha, beta, M):
    ws = [1, 2, 4, 8, 16, 32, 64]
    ts = [cm.wave_time(w, M, alpha, beta) for w in ws]
    f = wavefit.fit(ws, ts, M)
    assert f["alpha_s"] == pytest.approx(alpha, rel=1e-9)
    assert f["beta_Bps"] == pytest.approx(beta, rel=1e-9)
    assert f["r2"] == pytest.approx(1.0, abs=1e-12)
    assert f["w_star"] == pytest.approx(cm.optimal_waves(M, alpha, beta), rel=1e-9)
    # the measured best among the sampled W is the sampled W nearest the
    # integer optimum in model time
    best = min(ws, key=lambda w: cm.wave_time(w, M, alpha, beta))
    assert f["w_best_measured"] == best


def test_page_example_optimum():
    """alpha = 1 us, beta = 50 GB/s, M = 16 MB gives W* ~ 18 (the page's
    example); the fit of the model's own times reproduces it."""
    ws = list(range(1, 65))
    M = 16e6
    f = wavefit.fit(ws, [wavefit.model_time(w, 1e-6, 50e9, M) for w in ws], M)
    assert round(f["w_star"]) == 18
    assert f["w_best_measured"] == cm.optimal_waves_integer(M, 1e-6, 50e9)


def test_noisy_times_stay_close():
    rng = np.random.default_rng(7)
    alpha, beta, M = 4e-6, 6e12, 1e9
    ws = [1, 2, 4, 8, 16, 32, 64]
    ts = [cm.wave_time(w, M, alpha, beta) * (1 + 0.005 * rng.standard_normal()) for w in ws]
    f = wavefit.fit(ws, ts, M)
    assert f["alpha_s"] == pytest.approx(alpha, rel=0.15)
    assert f["beta_Bps"] == pytest.approx(beta, rel=0.02)
    assert f["r2"] > 0.99


def test_times_that_fall_with_w_give_no_optimum():
    """Times that fall as W grows fit a negative alpha: no W* is reported."""
    ws = [1, 2, 4, 8]
    f = wavefit.fit(ws, [10.0, 8.0, 6.0, 4.0], 1.0)
    assert f["alpha_s"] < 0
    assert f["w_star"] is None
    assert f["w_best_measured"] == 8


def test_bad_inputs_raise():
    with pytest.raises(ValueError):
        wavefit.fit([1], [1.0], 1.0)
    with pytest.raises(ValueError):
        wavefit.fit([0, 1], [1.0, 2.0], 1.0)
    with pytest.raises(ValueError):
        wavefit.fit([1, 2], [1.0, 2.0], 0.0)


def test_divisor_waves():
    assert wavefit.divisor_waves(64) == [1, 2, 4, 8, 16, 32, 64]
    assert wavefit.divisor_waves(12) == [1, 2, 4]
    assert wavefit.divisor_waves(256)[-1] == 256
    assert math.isclose(wavefit.model_time(2, 1.0, 2.0, 4.0), 2 + 2 + 1)


def test_linear_fit_recovers_a_line():
    ws = [1, 2, 4, 8, 16]
    f = wavefit.fit_linear(ws, [0.3e-3 + 11e-6 * w for w in ws])
    assert f["t0_s"] == pytest.approx(0.3e-3, rel=1e-9)
    assert f["alpha_s"] == pytest.approx(11e-6, rel=1e-9)
    assert f["r2"] == pytest.approx(1.0, abs=1e-12)
    with pytest.raises(ValueError):
        wavefit.fit_linear([1], [1.0])
