"""Pins of the oracle's capacity-factor variant (MoE system-optimisation
survey, section 1.1 "专家容量", eq. 3: EC = k f T / E; step 2: samples beyond
an expert's capacity are dropped, unused capacity is zero-filled).

Readings: EC is rounded up to whole rows; an expert's slots are counted in
(token, slot) row-major order and the first EC are kept at rows
e*EC + position of a fixed [E][EC][H] buffer; a dropped slot contributes
nothing to the combine (the gates are not renormalised)."""
import numpy as np
import pytest

import oracle
from combine_moe_route_17_b300 import workloads as wl


@pytest.mark.parametrize("T,E,k,f,ec", [(4096, 16, 2, 1.0, 512), (4096, 16, 2, 1.25, 640),
                                        (4096, 16, 2, 0.1, 52), (7, 3, 2, 1.0, 5),
                                        (16384, 64, 6, 1.0, 1536), (100, 8, 1, 0.0, 0)])
def test_capacity_hand_values(T, E, k, f, ec):
    assert oracle.expert_capacity(T, E, k, f) == ec


def test_hand_worked_drops():
    # four tokens, two experts, top-1; expert 0 gets three tokens but holds two
    idx = np.array([[0], [0], [0], [1]], np.int32)
    x = np.array([[0x3F80, 0x4000], [0x4040, 0x4080], [0x40A0, 0x40C0], [0x40E0, 0x4100]],
                 np.uint16)  # 1..8 in bf16
    w = np.ones((4, 1), np.float32)
    m = oracle.capacity_maps(idx, 2, 2)
    assert m["cap_slot"].ravel().tolist() == [0, 1, -1, 2]
    assert m["dropped"].tolist() == [1, 0]
    rows = oracle.capacity_rows(x, m["cap_slot"], 2, 2)
    assert rows.tolist() == [x[0].tolist(), x[1].tolist(), x[3].tolist(), [0, 0]]
    scale = np.array([2.0, 0.5], np.float32)
    out = oracle.capacity_standin(rows, scale, 2, 2)
    y = oracle.capacity_combine(out, m["cap_slot"], w)
    yv = oracle.bf16_to_f64(y)
    assert yv[0].tolist() == [2.0, 4.0] and yv[1].tolist() == [6.0, 8.0]
    assert yv[2].tolist() == [0.0, 0.0]  # every slot dropped
    assert yv[3].tolist() == [3.5, 4.0]
    assert (out[3] == 0).all()  # padding row stays zero


def test_positions_against_brute_force():
    rng = np.random.default_rng(3)
    T, E, k, EC = 50, 5, 3, 4
    idx = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
    m = oracle.capacity_maps(idx, E, EC)
    flat = idx.ravel()
    for n, e in enumerate(flat):
        pos = int(np.sum(flat[:n] == e))  # slots of e before this one, row-major
        want = e * EC + pos if pos < EC else -1
        assert m["cap_slot"].ravel()[n] == want
    for e in range(E):
        assert m["dropped"][e] == max(int(np.sum(flat == e)) - EC, 0)


def test_counting_invariants():
    cfg = wl.small_config(T=640, H=8, E=16, k=4, R=4, bias="zipf", bias_param=1.0, seed=5)
    idx, _ = oracle.route_topk(wl.make_logits(cfg), cfg.k)
    c = oracle.send_counts(idx, cfg.E, cfg.R)["c"]
    for f in (0.25, 0.5, 1.0, 1.5):
        EC = oracle.expert_capacity(cfg.T, cfg.E, cfg.k, f)
        m = oracle.capacity_maps(idx, cfg.E, EC)
        kept = np.minimum(c, EC)
        assert np.array_equal(m["dropped"], c - kept)
        assert int(kept.sum() + m["dropped"].sum()) == cfg.T * cfg.k
        assert int((m["cap_slot"] < 0).sum()) == int(m["dropped"].sum())
        live = np.sort(m["cap_slot"][m["cap_slot"] >= 0])
        assert len(np.unique(live)) == len(live)  # injective onto kept rows


def test_no_drops_matches_the_dropless_path():
    cfg = wl.small_config(T=384, H=48, E=16, k=4, R=4, W=2, bias="linear", bias_param=0.9, seed=6)
    inp = wl.make_inputs(cfg)
    ref = oracle.forward(cfg, inp)
    cap = oracle.forward_capacity(cfg, inp, f=cfg.E / cfg.k)  # EC = T >= every count
    assert cap["EC"] == cfg.T
    assert (cap["cap_slot"] >= 0).all() and (cap["dropped"] == 0).all()
    assert np.array_equal(cap["cap_rows"][cap["cap_slot"].ravel()],
                          np.repeat(inp["x"], cfg.k, axis=0))
    assert np.array_equal(cap["cap_out"][cap["cap_slot"].ravel()],
                          ref["out"][ref["slot_of"].ravel()])
    assert np.array_equal(cap["y"], ref["y"])  # same fp64 sum in j order, one rounding


def test_closed_form_with_drops():
    cfg = wl.small_config(T=256, H=32, E=8, k=3, R=2, bias="zipf", bias_param=1.0, seed=7)
    inp = wl.make_inputs(cfg)
    cap = oracle.forward_capacity(cfg, inp, f=0.6)
    assert cap["dropped"].sum() > 0
    kept = cap["cap_slot"] >= 0
    factor = np.where(kept, cap["w"].astype(np.float64) *
                      inp["scale"][cap["idx"]].astype(np.float64), 0.0).sum(axis=1)
    want = oracle.bf16_to_f64(inp["x"]) * factor[:, None]
    got = oracle.bf16_to_f64(cap["y"])
    # stand-in rounding (2^-9 relative) then the combine's rounding (2^-9)
    assert np.all(np.abs(got - want) <= 2.0 ** -7 * np.abs(want) + 1e-30)
    assert np.all(got[~kept.any(axis=1)] == 0.0)


def test_zero_capacity_drops_everything():
    cfg = wl.small_config(T=64, H=8, E=4, k=2, R=2, seed=8)
    inp = wl.make_inputs(cfg)
    cap = oracle.forward_capacity(cfg, inp, f=0.0)
    assert cap["EC"] == 0 and (cap["cap_slot"] == -1).all()
    assert cap["cap_rows"].shape == (0, cfg.H)
    assert (cap["y"] == 0).all()
