"""Pins for the oracle's send-count matrix, alltoallv offsets and dispatch
layout.

Send-count matrix and Alltoallv counts: "不规则与流水化 AllToAll", table
"经典 vs 不规则" and section "EP 不规则 a2a 的来源"; permute_by_device then
all_to_all: "混合专家模型跨卡通信机制解析", section 四; same-expert rows
contiguous: MoE survey section 1.1 step (2); waves of E/W experts:
"不规则与流水化 AllToAll", section "Wave-Scheduled 流水化".
"""
import numpy as np
import pytest

from combine_moe_route_17_b300 import workloads as wl


def _random_idx(T, E, k, seed, skew=0.0):
    rng = np.random.default_rng(seed)
    lg = rng.standard_normal((T, E)).astype(np.float32)
    lg += (skew * np.arange(E) / E).astype(np.float32)[None, :]
    return lg


def test_hand_worked_counts(orc):
    # T=4 tokens, k=1, E=4 experts, R=2: tokens 0,1 -> source 0; 2,3 -> source 1;
    # experts 0,1 -> rank 0; 2,3 -> rank 1.
    idx = np.array([[3], [0], [2], [3]], np.int32)
    r = orc.send_counts(idx, 4, 2)
    assert r["C"].tolist() == [[1, 0, 0, 1], [0, 0, 1, 1]]
    assert r["c"].tolist() == [1, 0, 1, 2]
    assert r["S"].tolist() == [[1, 1], [0, 2]]
    assert r["send_off"].tolist() == [[0, 1, 2], [0, 0, 2]]
    assert r["recv_off"].tolist() == [[0, 1, 1], [0, 1, 3]]
    assert r["recv_base"].tolist() == [0, 1, 4]
    m = orc.dispatch_maps(idx, 4, 2)
    # recv order (dst, src, expert, token, slot): (0,0,e0,t1) (1,0,e3,t0) (1,1,e2,t2) (1,1,e3,t3)
    assert m["slot_of"].ravel().tolist() == [1, 0, 2, 3]
    assert m["src_row"].tolist() == [1, 0, 2, 3]
    # send order per source (expert, token, slot): s0: t1(e0) t0(e3); s1: t2(e2) t3(e3)
    assert m["send_pos"].ravel().tolist() == [1, 0, 2, 3]


@pytest.mark.parametrize("T,E,k,R", [(64, 8, 2, 2), (96, 12, 3, 4), (40, 16, 4, 8), (16, 4, 4, 1)])
def test_counts_by_direct_enumeration(orc, T, E, k, R):
    idx, _ = orc.route_topk(_random_idx(T, E, k, T + E, skew=2.0), k)
    r = orc.send_counts(idx, E, R)
    C = np.zeros((R, E), np.int64)
    for t in range(T):
        for j in range(k):
            C[t // (T // R), idx[t, j]] += 1
    assert np.array_equal(r["C"], C)
    assert np.array_equal(r["c"], C.sum(0))
    S = C.reshape(R, R, E // R).sum(2)
    assert np.array_equal(r["S"], S)
    assert r["c"].sum() == T * k == r["S"].sum()
    assert (r["S"].sum(1) == (T // R) * k).all()
    for s in range(R):
        assert r["send_off"][s, 0] == 0 and r["send_off"][s, R] == (T // R) * k
        assert np.array_equal(np.diff(r["send_off"][s]), S[s])
    for d in range(R):
        assert np.array_equal(np.diff(r["recv_off"][d]), S[:, d])
    assert np.array_equal(np.diff(r["recv_base"]), S.sum(0))
    assert r["recv_base"][R] == T * k


def _brute_positions(idx, E, R):
    """Positions by counting, for every (t, j), the pairs with a smaller key."""
    T, k = idx.shape
    Tr, Er = T // R, E // R
    pairs = [(t, j, int(idx[t, j])) for t in range(T) for j in range(k)]
    recv_key = {(t, j): (e // Er, t // Tr, e, t, j) for t, j, e in pairs}
    send_key = {(t, j): (t // Tr, e // Er, e, t, j) for t, j, e in pairs}
    slot = np.zeros((T, k), np.int64)
    spos = np.zeros((T, k), np.int64)
    for a in recv_key:
        slot[a] = sum(1 for b in recv_key if recv_key[b] < recv_key[a])
        spos[a] = sum(1 for b in send_key if send_key[b] < send_key[a])
    return slot, spos


@pytest.mark.parametrize("T,E,k,R,seed", [(24, 8, 2, 2, 0), (32, 12, 3, 4, 1), (16, 16, 4, 8, 2),
                                          (12, 6, 6, 3, 3), (20, 4, 1, 1, 4)])
def test_dispatch_positions_by_brute_force(orc, T, E, k, R, seed):
    idx, _ = orc.route_topk(_random_idx(T, E, k, seed, skew=3.0), k)
    m = orc.dispatch_maps(idx, E, R)
    slot, spos = _brute_positions(idx, E, R)
    assert np.array_equal(m["slot_of"], slot)
    assert np.array_equal(m["send_pos"], spos)


def test_dispatch_is_a_bijection_and_copies_rows(orc):
    cfg = wl.small_config(T=256, H=24, E=16, k=4, R=4, W=4, bias="zipf", bias_param=1.0, seed=5)
    inp = wl.make_inputs(cfg)
    idx, _ = orc.route_topk(inp["logits"], cfg.k)
    m = orc.dispatch_maps(idx, cfg.E, cfg.R)
    n = cfg.T * cfg.k
    assert np.array_equal(np.sort(m["slot_of"].ravel()), np.arange(n))
    assert np.array_equal(np.sort(m["send_pos"].ravel()), np.arange(n))
    tok = np.repeat(np.arange(cfg.T), cfg.k).reshape(cfg.T, cfg.k)
    assert np.array_equal(m["src_row"][m["slot_of"]], tok)
    send, recv = orc.dispatch_rows(inp["x"], idx, m, cfg.E)
    assert np.array_equal(recv[m["slot_of"].ravel()], inp["x"][tok.ravel()])
    assert np.array_equal(send[m["send_pos"].ravel()], inp["x"][tok.ravel()])
    # the send rows of source s sit in its own partition
    Tr = cfg.T // cfg.R
    for s in range(cfg.R):
        rows = m["send_pos"][s * Tr:(s + 1) * Tr].ravel()
        assert rows.min() >= s * Tr * cfg.k and rows.max() < (s + 1) * Tr * cfg.k
    # keys (dst, src, expert) never decrease along the recv rows
    r = orc.send_counts(idx, cfg.E, cfg.R)
    e_of = np.empty(n, np.int64)
    e_of[m["slot_of"].ravel()] = idx.ravel()
    src_of = m["src_row"] // Tr
    key = (e_of // (cfg.E // cfg.R)) * cfg.R * cfg.E + src_of * cfg.E + e_of
    assert (np.diff(key) >= 0).all()
    assert np.array_equal(np.bincount(e_of // (cfg.E // cfg.R), minlength=cfg.R),
                          np.diff(r["recv_base"]))


def test_waves_tile_the_buffers(orc):
    cfg = wl.small_config(T=128, H=16, E=16, k=4, R=4, W=8, bias="dirichlet", bias_param=0.3,
                          seed=9)
    inp = wl.make_inputs(cfg)
    idx, _ = orc.route_topk(inp["logits"], cfg.k)
    m = orc.dispatch_maps(idx, cfg.E, cfg.R)
    full_s, full_r = orc.dispatch_rows(inp["x"], idx, m, cfg.E)
    acc_s = np.zeros_like(full_s)
    acc_r = np.zeros_like(full_r)
    touched = np.zeros(cfg.T * cfg.k, np.int64)
    for w in range(cfg.W):
        s_w, r_w = orc.dispatch_rows(inp["x"], idx, m, cfg.E, cfg.W, w, fill=0)
        sel = (idx // (cfg.E // cfg.W) == w).ravel()
        rows = m["slot_of"].ravel()[sel]
        touched[rows] += 1
        acc_r[rows] = r_w[rows]
        acc_s[m["send_pos"].ravel()[sel]] = s_w[m["send_pos"].ravel()[sel]]
        # rows outside the wave were not written
        others = np.setdiff1d(np.arange(cfg.T * cfg.k), rows)
        assert (r_w[others] == 0).all()
    assert (touched == 1).all()
    assert np.array_equal(acc_r, full_r) and np.array_equal(acc_s, full_s)


def test_layout_does_not_depend_on_wave_count(orc):
    # the maps take no W at all; the rows a wave writes are a subset of one layout
    cfg = wl.small_config(T=64, H=8, E=16, k=2, R=2, seed=2)
    inp = wl.make_inputs(cfg)
    idx, _ = orc.route_topk(inp["logits"], cfg.k)
    m = orc.dispatch_maps(idx, cfg.E, cfg.R)
    _, full = orc.dispatch_rows(inp["x"], idx, m, cfg.E, 1, -1)
    for W in (1, 2, 4, 8, 16):
        acc = np.zeros_like(full)
        for w in range(W):
            _, rw = orc.dispatch_rows(inp["x"], idx, m, cfg.E, W, w)
            acc |= rw
        assert np.array_equal(acc, full)


def test_max_over_mean_does_not_depend_on_R(orc):
    # DODOCO summary, section "主要发现" 1: per-expert max/mean is a property of
    # the routing decisions, not of the expert-to-rank map.
    cfg = wl.small_config(T=960, E=16, k=2, bias="zipf", bias_param=1.0, seed=4)
    idx, _ = orc.route_topk(wl.make_logits(cfg), cfg.k)
    vals = set()
    for R in (1, 2, 4, 8, 16):
        c = orc.send_counts(idx, cfg.E, R)["c"]
        vals.add(orc.imbalance_stats(c, cfg.T, cfg.k, R)["max_over_mean"])
    assert len(vals) == 1
