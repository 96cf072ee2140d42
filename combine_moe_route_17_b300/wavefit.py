"""Fit of the wave-pipeline cost model to measured step times.

"不规则与流水化 AllToAll", section "最优 wave 数", models a layer whose
exchange of M bytes is cut into W waves, each wave paying a fixed cost alpha,
with link bandwidth beta and the compute of a wave overlapped with the next
wave's exchange:

    T(W) = W * alpha + M / beta + M / (W * beta)

T is linear in (alpha, 1/beta), so measured (W, T) pairs give both by
ordinary least squares; the model's optimum is dT/dW = 0, i.e.
W* = sqrt(M / (alpha * beta)).  This module is host-side analysis for the
wave-pipeline measurement; it shares nothing with the oracle.
"""
from __future__ import annotations

import math
from typing import Iterable, Sequence

import numpy as np


def model_time(W: float, alpha: float, beta: float, M: float) -> float:
    """T(W) of the model (seconds, bytes, bytes/second)."""
    return W * alpha + M / beta + M / (W * beta)


def optimal_waves(alpha: float, beta: float, M: float) -> float:
    """W* = sqrt(M / (alpha * beta)), the real-valued minimiser of T(W)."""
    return math.sqrt(M / (alpha * beta))


def fit(ws: Sequence[float], ts: Sequence[float], M: float) -> dict:
    """Least-squares fit of alpha and beta to step times ts (seconds) at wave
    counts ws, for an exchange of M bytes.

    Returns alpha (s), beta (bytes/s; inf if the fitted 1/beta is not
    positive), W* (None unless both are positive), the measured best W, the
    fitted times and the coefficient of determination r2."""
    W = np.asarray(ws, dtype=np.float64)
    T = np.asarray(ts, dtype=np.float64)
    if W.shape != T.shape or W.size < 2:
        raise ValueError("need at least two (W, T) pairs of equal length")
    if np.any(W <= 0) or M <= 0:
        raise ValueError("wave counts and M must be positive")
    A = np.stack([W, M * (1.0 + 1.0 / W)], axis=1)
    (alpha, inv_beta), *_ = np.linalg.lstsq(A, T, rcond=None)
    pred = A @ np.array([alpha, inv_beta])
    ss_res = float(np.sum((T - pred) ** 2))
    ss_tot = float(np.sum((T - T.mean()) ** 2))
    r2 = 1.0 - ss_res / ss_tot if ss_tot > 0 else 1.0
    beta = 1.0 / inv_beta if inv_beta > 0 else math.inf
    w_star = optimal_waves(alpha, beta, M) if (alpha > 0 and 0 < beta < math.inf) else None
    best = int(W[int(np.argmin(T))])
    return {"alpha_s": float(alpha), "beta_Bps": float(beta), "w_star": w_star,
            "w_best_measured": best, "r2": r2, "fitted_s": pred.tolist()}


def fit_linear(ws: Sequence[float], ts: Sequence[float]) -> dict:
    """Least-squares line T(W) = t0 + alpha * W: the per-wave cost alpha when
    the waves' exchange and compute share one resource and no overlap term
    appears."""
    W = np.asarray(ws, dtype=np.float64)
    T = np.asarray(ts, dtype=np.float64)
    if W.shape != T.shape or W.size < 2:
        raise ValueError("need at least two (W, T) pairs of equal length")
    A = np.stack([np.ones_like(W), W], axis=1)
    (t0, alpha), *_ = np.linalg.lstsq(A, T, rcond=None)
    pred = A @ np.array([t0, alpha])
    ss_res = float(np.sum((T - pred) ** 2))
    ss_tot = float(np.sum((T - T.mean()) ** 2))
    return {"t0_s": float(t0), "alpha_s": float(alpha),
            "r2": 1.0 - ss_res / ss_tot if ss_tot > 0 else 1.0}


def divisor_waves(E: int, candidates: Iterable[int] = (1, 2, 4, 8, 16, 32, 64, 128, 256)):
    """Wave counts that divide E (a wave is E/W whole experts)."""
    return [w for w in candidates if w <= E and E % w == 0]
