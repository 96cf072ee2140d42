"""Pins for the oracle's stand-in expert, gate-weighted combine and imbalance
statistics.

Combine y = sum_i G(x)_i E_i(x): MoE survey section 1.1, eq. (1) and step
(4); the pseudo-code's final combine(returned, gates): "混合专家模型跨卡通信
机制解析", section 四.  Statistics: DODOCO summary, section "方法论"; hot/cold
expert ratio: Lina blog post, section "推理".
"""
import numpy as np
import pytest
import torch

from combine_moe_route_17_b300 import workloads as wl


def _f64(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _torch_bf16(v64):
    return torch.from_numpy(np.asarray(v64, np.float64)).to(torch.bfloat16).view(
        torch.int16).numpy().view(np.uint16)


def _pipeline(orc, cfg, inp, logits=None):
    lg = inp["logits"] if logits is None else logits
    idx, w = orc.route_topk(lg, cfg.k, cfg.n_groups, cfg.topk_groups, cfg.group_topn)
    m = orc.dispatch_maps(idx, cfg.E, cfg.R)
    _, recv = orc.dispatch_rows(inp["x"], idx, m, cfg.E, want_send=False)
    out = orc.expert_standin(recv, idx, m["slot_of"], inp["scale"])
    y = orc.combine(out, m["slot_of"], w)
    return idx, w, m, out, y


def test_standin_is_the_bf16_product(orc):
    cfg = wl.small_config(T=64, H=32, E=8, k=2, R=2, seed=1)
    inp = wl.make_inputs(cfg)
    idx, w, m, out, _ = _pipeline(orc, cfg, inp)
    tok = np.repeat(np.arange(cfg.T), cfg.k)
    prod = (_f64(inp["x"][tok]).astype(np.float32) *
            inp["scale"][idx.ravel()][:, None]).astype(np.float32)
    expect = torch.from_numpy(prod).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(out[m["slot_of"].ravel()], expect)


def test_combine_with_unit_experts_is_identity(orc):
    cfg = wl.small_config(T=128, H=64, E=16, k=4, R=4, bias="zipf", bias_param=1.0, seed=3)
    inp = wl.make_inputs(cfg)
    inp["scale"] = np.ones(cfg.E, np.float32)
    *_, y = _pipeline(orc, cfg, inp)
    assert np.array_equal(y, inp["x"])


def test_combine_closed_form_with_equal_gates(orc):
    # Equal logits -> every gate is exactly 1/k (k a power of two), so
    # y = bf16( sum_j bf16(s_j x) / k ) with an exact fp64 sum: a dropped
    # term, a wrong slot or a wrong expert scale changes y.
    E, k, R, T, H = 16, 4, 4, 64, 48
    cfg = wl.small_config(T=T, H=H, E=E, k=k, R=R, seed=6)
    inp = wl.make_inputs(cfg)
    rng = np.random.default_rng(0)
    lg = np.full((T, E), -5.0, np.float32)
    chosen = np.stack([rng.choice(E, k, replace=False) for _ in range(T)])
    lg[np.arange(T)[:, None], chosen] = 1.0
    idx, w, m, out, y = _pipeline(orc, cfg, inp, logits=lg)
    assert (w == np.float32(0.25)).all()
    xs = _f64(inp["x"])
    s = inp["scale"].astype(np.float32)
    terms = np.zeros((T, H))
    for j in range(k):
        prod = (xs.astype(np.float32) * s[idx[:, j]][:, None]).astype(np.float32)
        terms += 0.25 * _f64(_torch_bf16(prod.astype(np.float64)))
    assert np.array_equal(y, _torch_bf16(terms))


def test_combine_matches_closed_form_within_bf16(orc):
    cfg = wl.CONFIGS["c1"].replace(T=512)
    inp = wl.make_inputs(cfg)
    idx, w, m, out, y = _pipeline(orc, cfg, inp)
    gain = (w.astype(np.float64) * inp["scale"][idx].astype(np.float64)).sum(1)
    ref = _f64(inp["x"]) * gain[:, None]
    got = _f64(y)
    # out_j and y are each rounded once to bf16 (unit roundoff u = 2^-8):
    # |y - ref| <= (2u + u^2) |ref| plus the fp32 gate rounding (~1e-7)
    u = 2.0 ** -8
    assert np.all(np.abs(got - ref) <= (2 * u + u * u + 1e-6) * np.abs(ref))


def test_combine_token_range(orc):
    cfg = wl.small_config(T=32, H=16, E=8, k=2, R=2, seed=8)
    inp = wl.make_inputs(cfg)
    idx, w, m, out, y = _pipeline(orc, cfg, inp)
    part = orc.combine(out, m["slot_of"], w, 5, 17)
    assert np.array_equal(part[5:17], y[5:17])
    assert (part[:5] == 0).all() and (part[17:] == 0).all()


# ------------------------------------------------------------------ stats ----

def test_stats_hand_worked(orc):
    # E=8, R=4 (2 experts per rank): rank loads 2, 4, 6, 8 of 20 slots.
    c = np.array([2, 0, 4, 0, 6, 0, 8, 0], np.int32)
    st = orc.imbalance_stats(c, T=20, k=1, R=4)
    assert st["rank_load"].tolist() == [2, 4, 6, 8]
    # sum_i sum_j |L_i - L_j| = 2 * (2+4+6+2+4+2) = 40 ; 2 R sum L = 160
    assert (st["gini_num"], st["gini_den"]) == (40, 160)
    assert st["gini"] == 0.25
    assert st["max_load"] == 8 and st["min_load"] == 0
    assert st["max_over_mean"] == 8 * 8 / 20
    assert st["hot_over_cold"] == float("inf")


def test_gini_matches_the_sorted_rank_formula(orc):
    # textbook form: G = 2 sum_i i x_(i) / (n sum x) - (n + 1) / n, i = 1..n
    rng = np.random.default_rng(2)
    for R in (2, 3, 4, 8, 16):
        E = R * 4
        c = rng.integers(0, 1000, size=E).astype(np.int32)
        st = orc.imbalance_stats(c, T=R, k=1, R=R)  # only the Gini is checked
        L = np.sort(c.reshape(R, 4).sum(1).astype(np.float64))
        g = 2.0 * np.sum(np.arange(1, R + 1) * L) / (R * L.sum()) - (R + 1) / R
        assert st["gini"] == pytest.approx(g, abs=1e-12)


def test_gini_zero_for_equal_rank_loads(orc):
    # logits that send token t to experts 2(t mod 4), 2(t mod 4)+1: every rank
    # receives exactly T k / R rows.
    T, E, k, R = 64, 8, 2, 4
    lg = np.zeros((T, E), np.float32)
    for t in range(T):
        lg[t, 2 * (t % 4)] = 2.0
        lg[t, 2 * (t % 4) + 1] = 1.0
    idx, _ = orc.route_topk(lg, k)
    c = orc.send_counts(idx, E, R)["c"]
    st = orc.imbalance_stats(c, T, k, R)
    assert st["gini"] == 0.0 and st["gini_num"] == 0
    assert st["max_over_mean"] == 1.0 and st["hot_over_cold"] == 1.0


def test_gini_when_one_rank_takes_everything(orc):
    T, E, k = 32, 16, 2
    lg = np.zeros((T, E), np.float32)
    lg[:, :2] = 5.0  # experts 0, 1 live on rank 0 for every R <= 8
    idx, _ = orc.route_topk(lg, k)
    for R in (2, 4, 8):
        c = orc.send_counts(idx, E, R)["c"]
        st = orc.imbalance_stats(c, T, k, R)
        assert st["gini"] == pytest.approx((R - 1) / R, abs=1e-15)


def test_hot_over_cold_of_config_c2_is_about_five(orc):
    # the linear-ramp bias of the c2 workload was chosen for a ~5x hot/cold
    # ratio (the 16-expert inference skew of the Lina post, section "推理").
    cfg = wl.CONFIGS["c2"]
    idx, _ = orc.route_topk(wl.make_logits(cfg), cfg.k)
    c = orc.send_counts(idx, cfg.E, cfg.R)["c"]
    st = orc.imbalance_stats(c, cfg.T, cfg.k, cfg.R)
    assert 4.75 <= st["hot_over_cold"] <= 5.25
