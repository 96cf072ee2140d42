"""GPU parity of the greedy expert placement (MoE survey, section 4.2.2) and
the fitted symmetric-Dirichlet alpha (DODOCO summary, section "方法论")
against the oracle: placement, relabelling and every summary bit-exact; the
relabelled routing, run through the count pass and the statistics, gives the
placed rank loads."""
import math

import numpy as np
import pytest
import torch

import oracle
from combine_moe_route_17_b300 import binding as B
from combine_moe_route_17_b300 import workloads as wl

pytestmark = pytest.mark.gpu


def _gpu_place(c, E, R):
    shape = B.Shape(R, 8, E, 1, R, 1, 1, 0, 0)
    cc = torch.from_numpy(np.ascontiguousarray(c, np.int32)).cuda()
    pl = torch.empty(E, dtype=torch.int32, device="cuda")
    rl = torch.empty(E, dtype=torch.int32, device="cuda")
    out = torch.zeros(8, dtype=torch.float64, device="cuda")
    B.place_experts_greedy(shape, cc, pl, rl, out)
    torch.cuda.synchronize()
    return pl.cpu().numpy(), rl.cpu().numpy(), B.decode_placement(out)


def _check_place(c, E, R):
    pl, rl, st = _gpu_place(c, E, R)
    ref = oracle.place_greedy(c, R)
    assert np.array_equal(pl, ref["placement"])
    assert np.array_equal(rl, ref["relabel"])
    before = oracle.placement_gini(c, np.arange(E) // (E // R), R)
    after = oracle.placement_gini(c, ref["placement"], R)
    assert st["gini_num_before"] == before["gini_num"]
    assert st["gini_num_after"] == after["gini_num"]
    assert st["gini_den"] == before["gini_den"] == after["gini_den"]
    assert st["gini_before"] == before["gini"] and st["gini_after"] == after["gini"]
    lb = np.bincount(np.arange(E) // (E // R), weights=c, minlength=R)
    la = np.bincount(ref["placement"], weights=c, minlength=R)
    assert st["max_rank_load_before"] == int(lb.max())
    assert st["max_rank_load_after"] == int(la.max())
    return ref


@pytest.mark.parametrize("E,R", [(4, 2), (16, 4), (64, 8), (128, 16), (256, 32), (128, 64),
                                 (256, 64), (7, 7), (1, 1)])
def test_placement_on_random_counts(E, R):
    rng = np.random.default_rng(E * 7 + R)
    for trial in range(3):
        c = rng.integers(0, 4000, E).astype(np.int32)
        if trial == 1:
            c[:] = 5  # all ties
        _check_place(c, E, R)


@pytest.mark.parametrize("cfg", [wl.CONFIGS[n] for n in ("c1", "c2", "c3", "c4")]
                         + [c for c in wl.SWEEP if c.T == 8192 and c.W == 1],
                         ids=lambda c: c.name)
def test_placement_and_alpha_on_routed_counts(cfg):
    small = wl.reduced(cfg, T=min(cfg.T, cfg.R * 256))
    idx, _ = oracle.route_topk(wl.make_logits(small), small.k, small.n_groups, small.topk_groups,
                               small.group_topn)
    c = oracle.send_counts(idx, small.E, small.R)["c"]
    ref = _check_place(c, small.E, small.R)
    # alpha, bit-exact
    shape = B.Shape.of(small)
    a = torch.zeros(1, dtype=torch.float64, device="cuda")
    B.dirichlet_alpha(shape, torch.from_numpy(c).cuda(), a)
    torch.cuda.synchronize()
    want = oracle.dirichlet_alpha(c)
    got = float(a.item())
    assert got == want or (math.isinf(got) and math.isinf(want))
    # relabel the routing: the count pass and the statistics see the placement
    from _parity import make_pipeline

    relabelled = ref["relabel"][idx].astype(np.int32)
    inp = {"logits": wl.make_logits(small), "x": np.zeros((small.T, small.H), np.uint16),
           "scale": wl.make_scales(small)}
    p = make_pipeline(small, inp)
    p.idx.copy_(torch.from_numpy(relabelled))
    p.count()
    p.imbalance()
    torch.cuda.synchronize()
    assert B.get_device_error(p.ws) == 0
    la = np.bincount(ref["placement"], weights=c, minlength=small.R).astype(np.int64)
    assert np.array_equal(p.rank_load.cpu().numpy(), la)
    assert p.stats_dict()["gini"] == oracle.placement_gini(c, ref["placement"], small.R)["gini"]


def test_alpha_limits_on_the_gpu():
    shape = B.Shape(64, 8, 8, 1, 1, 1, 1, 0, 0)
    a = torch.zeros(1, dtype=torch.float64, device="cuda")
    for c, want in (([64, 0, 0, 0, 0, 0, 0, 0], 0.0), ([8] * 8, math.inf)):
        B.dirichlet_alpha(shape, torch.tensor(c, dtype=torch.int32, device="cuda"), a)
        torch.cuda.synchronize()
        assert float(a.item()) == want
