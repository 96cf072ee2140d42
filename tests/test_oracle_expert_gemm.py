"""Pins of the oracle's linear expert on expert-major rows (MoE survey,
section 1.1, step 3): hand-computed products, identity weights, and experts
owning consecutive runs of rows (empty experts included)."""
import numpy as np

import oracle


def _bf(v):
    return oracle.bf16_round(np.asarray(v, dtype=np.float64))


def test_hand_computed_products():
    rows = _bf([[1, 2], [3, 4], [5, 6]])
    W = _bf([[[1, 0], [1, 1]], [[2, 0], [0, 2]]])  # [E][N][H]
    out = oracle.expert_gemm(rows, [2, 1], W)
    assert oracle.bf16_to_f64(out).tolist() == [[1, 3], [3, 7], [10, 12]]


def test_identity_weights_return_the_rows():
    rng = np.random.default_rng(1)
    H = 16
    rows = _bf(rng.standard_normal((40, H)))
    W = np.stack([_bf(np.eye(H))] * 3)
    assert np.array_equal(oracle.expert_gemm(rows, [10, 0, 30], W), rows)


def test_runs_follow_the_counts():
    rng = np.random.default_rng(2)
    H, N = 8, 4
    rows = _bf(rng.standard_normal((9, H)))
    W = _bf(rng.standard_normal((3, N, H)))
    out = oracle.expert_gemm(rows, [0, 4, 5], W)
    X, Wf = oracle.bf16_to_f64(rows), oracle.bf16_to_f64(W)
    assert np.array_equal(out[:4], _bf(X[:4] @ Wf[1].T))
    assert np.array_equal(out[4:], _bf(X[4:] @ Wf[2].T))
    assert np.array_equal(oracle.expert_gemm(rows, [0, 4, 5], W, sel=[3, 7]), out[[3, 7]])
