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


def test_ffn_hand_values():
    # one expert, H = F = 1: hidden = silu(x w1) * (x w3), out = hidden * w2
    rows = _bf([[2.0], [-1.0], [0.0]])
    w1, w3, w2 = _bf([[[1.0]]]), _bf([[[3.0]]]), _bf([[[0.5]]])
    hidden, out = oracle.expert_ffn(rows, [3], w1, w3, w2)
    silu = lambda z: z / (1 + np.exp(-z))  # noqa: E731
    want_h = _bf([[silu(2.0) * 6.0], [silu(-1.0) * -3.0], [0.0]])
    assert np.array_equal(hidden, want_h)
    assert np.array_equal(out, _bf(oracle.bf16_to_f64(want_h) * 0.5))


def test_ffn_with_identity_weights():
    rng = np.random.default_rng(3)
    H = 8
    rows = _bf(rng.standard_normal((12, H)))
    eye = np.stack([_bf(np.eye(H))] * 2)
    hidden, out = oracle.expert_ffn(rows, [5, 7], eye, eye, eye)
    X = oracle.bf16_to_f64(rows)
    assert np.array_equal(hidden, _bf(X / (1 + np.exp(-X)) * X))
    assert np.array_equal(out, hidden)


def test_ffn_down_projection_is_the_linear_expert():
    rng = np.random.default_rng(4)
    H, F = 8, 16
    rows = _bf(rng.standard_normal((10, H)))
    w1, w3 = _bf(rng.standard_normal((2, F, H))), _bf(rng.standard_normal((2, F, H)))
    w2 = _bf(rng.standard_normal((2, H, F)))
    hidden, out = oracle.expert_ffn(rows, [4, 6], w1, w3, w2)
    assert np.array_equal(out, oracle.expert_gemm(hidden, [4, 6], w2))
