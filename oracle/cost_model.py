"""Closed-form models of the irregular-AllToAll page -- TEST INFRASTRUCTURE.

"不规则与流水化 AllToAll" (t6page.pages.dev), sections "长尾延迟问题" and
"最优 wave 数":

* p95 link load under the normal approximation to Multinomial(B, p_bar):
  m_p95 ~= m_avg * (1 + 1.645 * sqrt(1 / (B * p_bar))), with the cell variance
  B p_bar (1 - p_bar) approximated by B p_bar (eq. cc-sparse-a2a-p95).
* End-to-end time of a W-wave exchange: T(W) ~= W alpha + M/beta + M/(W beta)
  (eq. cc-a2a-window-time): W start-up latencies, the bandwidth floor, and the
  last wave's unoverlapped tail.
* Its minimiser W* ~= sqrt(M / (alpha beta)) (eq. cc-sparse-a2a-optimal-w).
"""
from __future__ import annotations

import math

Z95 = 1.645  # one-sided 95% quantile of the standard normal


def wave_time(W: float, M: float, alpha: float, beta: float) -> float:
    """T(W) = W*alpha + M/beta + M/(W*beta)  (seconds, bytes, bytes/s)."""
    return W * alpha + M / beta + M / (W * beta)


def optimal_waves(M: float, alpha: float, beta: float) -> float:
    """Stationary point of T(W): dT/dW = alpha - M/(W^2 beta) = 0."""
    return math.sqrt(M / (alpha * beta))


def optimal_waves_integer(M: float, alpha: float, beta: float, w_max: int = 4096) -> int:
    """Integer W >= 1 with the smallest T(W) (first one on ties)."""
    best, best_t = 1, wave_time(1, M, alpha, beta)
    for W in range(2, w_max + 1):
        t = wave_time(W, M, alpha, beta)
        if t < best_t:
            best, best_t = W, t
    return best


def p95_link_load_page(m_avg: float, B: float, p_bar: float) -> float:
    """The page's approximation m_avg * (1 + 1.645 / sqrt(B * p_bar))."""
    return m_avg * (1.0 + Z95 * math.sqrt(1.0 / (B * p_bar)))


def p95_link_load_exact_excess(tokens: int, E: int, k: int, R: int) -> float:
    """1.645 * sigma of one send-count entry under uniform top-k routing.

    Each of ``tokens`` tokens picks a uniformly random k-subset of E experts;
    the number landing on one rank (E/R experts) is hypergeometric with
    variance k p (1-p) (E-k)/(E-1), p = 1/R.  A link load sums ``tokens``
    independent such counts."""
    p = 1.0 / R
    var = tokens * k * p * (1.0 - p) * (E - k) / (E - 1) if E > 1 else 0.0
    return Z95 * math.sqrt(var)
