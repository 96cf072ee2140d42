"""moe_route_and_count: routing and counts in one launch (each look-back tile
routes its own tokens and histograms them from shared memory) against the two
separate launches and the oracle.  Everything it writes is bit-identical to
moe_route_topk followed by moe_build_send_counts: idx, w, C, c, S, the
offsets, and the per-slot ranks (seen through the dispatch maps)."""
import numpy as np
import pytest
import torch

import oracle
from combine_moe_route_17_b300 import binding as B
from combine_moe_route_17_b300 import workloads as wl

from _parity import assert_counts, assert_maps, assert_routing, make_pipeline

pytestmark = pytest.mark.gpu


def _front(cfg, inp, fuse_route):
    p = make_pipeline(cfg, inp, fuse_route=fuse_route)
    p.slot_of.fill_(-1)
    p.route_count()
    p.dispatch(-1)
    torch.cuda.synchronize()
    assert B.get_device_error(p.ws) == 0
    return p


@pytest.mark.parametrize("name", ["c1", "c2", "c3", "c4"])
def test_one_launch_equals_two_launches_at_full_size(name):
    cfg = wl.CONFIGS[name]
    lg = wl.make_logits(cfg)
    inp = {"logits": lg, "x": np.zeros((cfg.T, cfg.H), np.uint16), "scale": wl.make_scales(cfg)}
    a = _front(cfg, inp, True)
    b = _front(cfg, inp, False)
    assert torch.equal(a.idx, b.idx)
    assert torch.equal(a.w.view(torch.int32), b.w.view(torch.int32))  # bitwise
    for key in a.counts:
        assert torch.equal(a.counts[key], b.counts[key]), key
    assert torch.equal(a.slot_of, b.slot_of)
    assert torch.equal(a.src_row, b.src_row)
    # and the oracle's routing and counts
    ref = oracle.forward(cfg, {"logits": lg}, with_rows=False)
    got = a.results()
    assert_routing(got, ref)
    assert_counts(got, ref)
    assert_maps(got, ref)


@pytest.mark.parametrize("cfg", [
    wl.small_config(T=1200, H=16, E=16, k=2, R=4, W=1, seed=21),     # ragged tiles (Tr = 300)
    wl.small_config(T=96, H=16, E=8, k=3, R=2, W=1, seed=22),        # one partial tile
    wl.small_config(T=777, H=16, E=3, k=1, R=1, W=1, seed=23),       # E % 4 != 0: scalar loads
    wl.small_config(T=512, H=16, E=256, k=16, R=64, W=1, seed=24),   # G = 32, k = 16
    wl.small_config(T=640, H=16, E=64, k=6, R=8, W=1, n_groups=8, topk_groups=3,
                    group_topn=2, seed=25),                           # groups, fused
    wl.small_config(T=384, H=16, E=12, k=3, R=3, W=1, n_groups=4, topk_groups=2,
                    group_topn=3, seed=26),                           # groups, two launches
], ids=lambda c: c.name)
def test_small_shapes_match_the_oracle(cfg):
    inp = wl.make_inputs(cfg)
    ref = oracle.forward(cfg, inp, with_rows=False)
    p = _front(cfg, inp, True)
    got = p.results()
    assert_routing(got, ref)
    assert_counts(got, ref)
    assert_maps(got, ref)
    q = _front(cfg, inp, False)
    assert torch.equal(p.w.view(torch.int32), q.w.view(torch.int32))


def test_repeated_calls_on_one_workspace():
    cfg = wl.small_config(T=2048, H=16, E=64, k=6, R=8, W=1, bias="linear", bias_param=0.874,
                          seed=27)
    inp = wl.make_inputs(cfg)
    ref = oracle.forward(cfg, inp, with_rows=False)
    p = make_pipeline(cfg, inp, fuse_route=True)
    for _ in range(3):
        p.slot_of.fill_(-1)
        for t in p.counts.values():
            t.fill_(-7)
        p.route_count()
        p.dispatch(-1)
        torch.cuda.synchronize()
        assert B.get_device_error(p.ws) == 0
        got = p.results()
        assert_counts(got, ref)
        assert_maps(got, ref)


def test_non_finite_logit_is_reported():
    cfg = wl.small_config(T=256, H=16, E=16, k=2, R=2, W=1, seed=28)
    p = make_pipeline(cfg, wl.make_inputs(cfg), fuse_route=True)
    p.logits[5, 3] = float("inf")
    p.route_count()
    assert B.get_device_error(p.ws) == B.MOE_ERR_DEVICE_CHECK
    assert B.get_device_error(p.ws) == 0


def test_lookback_wait_gives_up_with_timeout():
    """A tile that never publishes its look-back status: its successors'
    bounded waits run out, the launch ends and reports MOE_ERR_TIMEOUT; the
    workspace then works again."""
    cfg = wl.small_config(T=2048, H=16, E=16, k=2, R=2, W=1, seed=29)  # 8 tiles per source
    inp = wl.make_inputs(cfg)
    ref = oracle.forward(cfg, inp, with_rows=False)
    p = make_pipeline(cfg, inp, fuse_route=True)
    B.debug_set_fault(p.ws, tile=2, wait_ns=20_000_000)  # 20 ms
    p.route_count()
    assert B.get_device_error(p.ws) == B.MOE_ERR_TIMEOUT
    B.debug_set_fault(p.ws, tile=-1, wait_ns=0)
    p.route_count()
    p.dispatch(-1)
    torch.cuda.synchronize()
    assert B.get_device_error(p.ws) == 0
    assert np.array_equal(p.counts["C"].cpu().numpy(), ref["C"])
    assert np.array_equal(p.slot_of.cpu().numpy(), ref["slot_of"])


def test_rejects_bad_arguments():
    cfg = wl.small_config(T=64, H=16, E=8, k=2, R=2, W=1)
    p = make_pipeline(cfg, wl.make_inputs(cfg))
    with pytest.raises(B.MoEError) as e:
        B.route_and_count(p.shape, p.logits, p.idx, p.w, p.counts, p.ws[:128])
    assert e.value.status == B.MOE_ERR_INVALID_ARG
