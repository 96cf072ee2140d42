"""GPU parity at the workloads' full sizes, in the launch configuration the
bench times (fused dispatch in W wave calls on W streams, stand-in expert,
combine, statistics).  Everything is compared in full: routing, counts,
offsets, row maps and statistics directly; every recv row, every stand-in
output row and every combine output against the oracle evaluated token chunk
by token chunk (its row copy, stand-in and combine over each chunk's tokens,
on the host's cores side by side)."""
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import torch

import oracle
from combine_moe_route_17_b300 import MoEPipeline
from combine_moe_route_17_b300 import binding as B
from combine_moe_route_17_b300 import workloads as wl

from _parity import Y_RTOL, assert_counts, assert_maps, assert_routing, assert_stats, assert_y

pytestmark = pytest.mark.gpu

FULL = [wl.CONFIGS[n] for n in ("c1", "c2", "c3", "c4")] + [
    next(c for c in wl.SWEEP if c.T == 262144 and c.bias_param == 0.1 and c.W == 16),
    next(c for c in wl.SWEEP if c.T == 512 and c.bias_param == 10.0 and c.W == 4),
    next(c for c in wl.SWEEP if c.T == 32768 and c.bias_param == 1.0 and c.W == 8),
]

CHUNK_BYTES = 128 << 20  # rows of one token chunk (k rows per token)


def _oracle_chunk(cfg, inp, ref, a, b, standin):
    """The oracle's rows for tokens [a, b) in compact order (token, slot):
    the recv row copies, or the stand-in expert outputs and the combine."""
    n, k = b - a, cfg.k
    compact = np.arange(n * k, dtype=np.int32).reshape(n, k)
    maps = {"send_pos": compact, "slot_of": compact}
    _, rows = oracle.dispatch_rows(inp["x"][a:b], ref["idx"][a:b], maps, cfg.E,
                                   want_send=False)
    if not standin:
        return rows, None
    out = oracle.expert_standin(rows, ref["idx"][a:b], compact, inp["scale"])
    return out, oracle.combine(out, compact, ref["w"][a:b])


def _oracle_y_for_tokens(cfg, inp, ref, toks):
    """The oracle's row copy, stand-in expert and combine for the sampled
    tokens only, on a compact copy of their expert rows."""
    k = cfg.k
    n = len(toks)
    compact = np.arange(n * k, dtype=np.int32).reshape(n, k)
    maps = {"send_pos": compact, "slot_of": compact}
    _, rows = oracle.dispatch_rows(inp["x"][toks], ref["idx"][toks], maps, cfg.E,
                                   want_send=False)
    out = oracle.expert_standin(rows, ref["idx"][toks], compact, inp["scale"])
    return oracle.combine(out, compact, ref["w"][toks])


def check_rows_in_full(cfg, inp, ref, rows_dev, y_dev=None):
    """Every row of rows_dev (recv layout, T*k rows) against the oracle; with
    y_dev, rows_dev holds the stand-in outputs and every y row is checked
    too.  The GPU rows of a token chunk are gathered through the oracle's
    slot_of (compared in full beforehand), so the chunks cover all T*k rows."""
    T, k, H = cfg.T, cfg.k, cfg.H
    per = max(1, CHUNK_BYTES // (k * H * 2))
    chunks = [(a, min(T, a + per)) for a in range(0, T, per)]
    nthreads = max(1, min(8, len(os.sched_getaffinity(0))))
    standin = y_dev is not None
    bad_rows = bad_y = 0
    with ThreadPoolExecutor(max_workers=nthreads) as ex:
        for g0 in range(0, len(chunks), nthreads):
            group = chunks[g0:g0 + nthreads]
            futs = [ex.submit(_oracle_chunk, cfg, inp, ref, a, b, standin) for a, b in group]
            for (a, b), fut in zip(group, futs):
                sl = torch.from_numpy(ref["slot_of"][a:b].reshape(-1).astype(np.int64))
                got = rows_dev[sl.to(rows_dev.device)].view(torch.int16).cpu().numpy()
                got = got.view(np.uint16)
                want, y_want = fut.result()
                bad_rows += int(np.any(got != want, axis=1).sum())
                if standin:
                    yg = oracle.bf16_to_f64(y_dev[a:b].view(torch.int16).cpu().numpy()
                                            .view(np.uint16))
                    yr = oracle.bf16_to_f64(y_want)
                    bad_y += int((np.abs(yg - yr) > Y_RTOL * np.abs(yr)).sum())
    what = "stand-in output rows" if standin else "recv rows"
    assert bad_rows == 0, f"{bad_rows} of {T * k} {what} differ from the oracle"
    assert bad_y == 0, f"combine: {bad_y} of {T * H} elements outside rel {Y_RTOL}"


@pytest.mark.parametrize("cfg", FULL, ids=lambda c: c.name)
def test_full_size_parity(cfg):
    inp = wl.make_inputs(cfg)
    ref = oracle.forward(cfg, inp, with_rows=False)
    p = MoEPipeline(cfg, device="cuda")
    p.load_inputs(torch.from_numpy(inp["logits"]), torch.from_numpy(inp["x"].view(np.int16)),
                  torch.from_numpy(inp["scale"]))
    p.route_count()
    p.dispatch_waves()
    torch.cuda.synchronize()
    # the row maps first (the row checks gather through them)
    assert np.array_equal(p.slot_of.cpu().numpy(), ref["slot_of"]), "slot_of"
    so = ref["slot_of"].reshape(-1)
    assert np.array_equal(np.sort(so), np.arange(cfg.T * cfg.k, dtype=so.dtype))
    check_rows_in_full(cfg, inp, ref, p.recv)
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
    # src_row o slot_of = token, in full
    assert np.array_equal(got["src_row"][so], np.repeat(np.arange(cfg.T), cfg.k))
    check_rows_in_full(cfg, inp, ref, p.recv, p.y)


@pytest.mark.parametrize("name", ["c2", "c3", "c4"])
def test_full_size_parity_in_the_bench_graph(name):
    """The step exactly as the bench times it: one captured CUDA graph with
    programmatic launches (route, counts, the W dispatch waves on W streams at
    once, stand-in expert, combine) and the statistics on a second stream
    forked after the counts; replayed twice (the second replay must not see
    stale state)."""
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
        p.dispatch_waves(s0)
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
