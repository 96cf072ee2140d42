"""Pins of the oracle's expert-major recv layout: rows ordered (destination
rank, expert, source, token, slot) -- with contiguous expert blocks per rank,
(expert, token, slot) -- so each expert's rows are one run (MoE survey,
section 1.1, step 2: samples of the same expert placed contiguously)."""
import numpy as np

import oracle
from combine_moe_route_17_b300 import workloads as wl


def test_rows_against_lexicographic_brute_force():
    rng = np.random.default_rng(4)
    T, E, k = 40, 6, 3
    idx = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
    m = oracle.dispatch_maps_expert_major(idx, E)
    keys = [(idx[t, j], t, j) for t in range(T) for j in range(k)]
    for t in range(T):
        for j in range(k):
            want = sum(1 for key in keys if key < (idx[t, j], t, j))
            assert m["slot_of"][t, j] == want
    assert np.array_equal(m["src_row"][m["slot_of"].ravel()], np.repeat(np.arange(T), k))


def test_is_a_resort_of_the_rank_major_layout():
    cfg = wl.small_config(T=512, H=8, E=32, k=4, R=4, bias="zipf", bias_param=1.0, seed=9)
    idx, _ = oracle.route_topk(wl.make_logits(cfg), cfg.k)
    rm = oracle.dispatch_maps(idx, cfg.E, cfg.R)
    em = oracle.dispatch_maps_expert_major(idx, cfg.E)
    c = oracle.send_counts(idx, cfg.E, cfg.R)
    # same per-rank ranges: expert-major only reorders rows inside a rank
    assert np.array_equal(em["expert_off"][:: cfg.E // cfg.R], c["recv_base"])
    # every expert's rows are one contiguous run of length c_e
    e_of_row = np.empty(cfg.T * cfg.k, np.int64)
    e_of_row[em["slot_of"].ravel()] = idx.ravel()
    assert np.array_equal(np.diff(e_of_row) >= 0, np.ones(cfg.T * cfg.k - 1, bool))
    assert np.array_equal(np.diff(em["expert_off"]), c["c"])
    # rank-major rows of rank d map onto the same range in expert-major order
    d_rm = np.searchsorted(c["recv_base"], rm["slot_of"].ravel(), side="right") - 1
    d_em = np.searchsorted(c["recv_base"], em["slot_of"].ravel(), side="right") - 1
    assert np.array_equal(d_rm, d_em)
