"""GPU parity at the workloads' full sizes, in the launch configuration the
bench times (fused dispatch in W wave calls, stand-in expert, combine,
statistics).  Routing, counts, offsets, row maps and statistics are compared
in full; permuted rows and combine outputs on a seeded sample of tokens that
the oracle evaluates one by one; the bijection of the row maps in full."""
import numpy as np
import pytest
import torch

import oracle
from combine_moe_route_17_b300 import MoEPipeline
from combine_moe_route_17_b300 import binding as B
from combine_moe_route_17_b300 import workloads as wl

from _parity import assert_counts, assert_maps, assert_routing, assert_stats, assert_y

pytestmark = pytest.mark.gpu

FULL = [wl.CONFIGS[n] for n in ("c1", "c2", "c3", "c4")] + [
    next(c for c in wl.SWEEP if c.T == 262144 and c.bias_param == 0.1 and c.W == 16),
    next(c for c in wl.SWEEP if c.T == 512 and c.bias_param == 10.0 and c.W == 4),
    next(c for c in wl.SWEEP if c.T == 32768 and c.bias_param == 1.0 and c.W == 8),
]


def _oracle_y_for_tokens(cfg, inp, ref, toks):
    """The oracle's stand-in expert and combine evaluated for the sampled
    tokens only, on a compact copy of their expert rows."""
    k = cfg.k
    n = len(toks)
    rows = np.repeat(inp["x"][toks], k, axis=0)
    compact = np.arange(n * k, dtype=np.int32).reshape(n, k)
    out = oracle.expert_standin(rows, ref["idx"][toks], compact, inp["scale"])
    return oracle.combine(out, compact, ref["w"][toks])


@pytest.mark.parametrize("cfg", FULL, ids=lambda c: c.name)
def test_full_size_sampled_parity(cfg):
    inp = wl.make_inputs(cfg)
    ref = oracle.forward(cfg, inp, with_rows=False)
    p = MoEPipeline(cfg, device="cuda")
    p.load_inputs(torch.from_numpy(inp["logits"]), torch.from_numpy(inp["x"].view(np.int16)),
                  torch.from_numpy(inp["scale"]))
    p.route_count()
    p.dispatch_waves()
    rng = np.random.default_rng(1234)
    toks = np.unique(np.concatenate([rng.integers(0, cfg.T, size=min(cfg.T, 768)),
                                     [0, cfg.T - 1]])).astype(np.int64)
    slots = torch.from_numpy(ref["slot_of"][toks].reshape(-1).astype(np.int64)).cuda()
    recv_s = p.recv[slots].view(torch.int16).cpu().numpy().view(np.uint16)
    p.expert()
    p.combine()
    p.imbalance()
    torch.cuda.synchronize()
    assert B.get_device_error(p.ws) == 0
    got = p.results()
    assert_routing(got, ref)
    assert_counts(got, ref)
    assert_maps(got, ref)
    assert_stats(got, ref)
    # bijection onto the T*k rows and src_row o slot_of = token, in full
    so = got["slot_of"].reshape(-1)
    assert np.array_equal(np.sort(so), np.arange(cfg.T * cfg.k, dtype=so.dtype))
    assert np.array_equal(got["src_row"][so], np.repeat(np.arange(cfg.T), cfg.k))
    # sampled rows: bit copies of x
    assert np.array_equal(recv_s, np.repeat(inp["x"][toks], cfg.k, axis=0))
    # sampled combine outputs
    assert_y(got["y"][toks], _oracle_y_for_tokens(cfg, inp, ref, toks))


@pytest.mark.parametrize("name", ["c2", "c4"])
def test_full_size_parity_in_the_bench_graph(name):
    """The step exactly as the bench times it: one captured CUDA graph with
    programmatic launches (route, counts, the W dispatch waves, stand-in
    expert, combine) and the statistics on a second stream forked after the
    counts; replayed twice (the second replay must not see stale state)."""
    cfg = wl.CONFIGS[name]
    inp = wl.make_inputs(cfg)
    ref = oracle.forward(cfg, inp, with_rows=False)
    p = MoEPipeline(cfg, device="cuda")
    p.load_inputs(torch.from_numpy(inp["logits"]), torch.from_numpy(inp["x"].view(np.int16)),
                  torch.from_numpy(inp["scale"]))
    s0, side = torch.cuda.Stream(), torch.cuda.Stream()
    s0.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s0):
        p.route_count(s0)
        side.wait_stream(s0)
        p.imbalance(side)
        for w in range(cfg.W):
            p.dispatch(w, s0)
        s0.wait_stream(side)
        p.expert(s0)
        p.combine(s0)
    for _ in range(2):
        p.y.zero_()
        p.slot_of.fill_(-1)
        g.replay()
        torch.cuda.synchronize()
        assert B.get_device_error(p.ws) == 0
        got = p.results()
        assert_routing(got, ref)
        assert_counts(got, ref)
        assert_maps(got, ref)
        assert_stats(got, ref)
    rng = np.random.default_rng(4321)
    toks = np.unique(np.concatenate([rng.integers(0, cfg.T, size=512), [0, cfg.T - 1]]))
    assert_y(got["y"][toks], _oracle_y_for_tokens(cfg, inp, ref, toks))
