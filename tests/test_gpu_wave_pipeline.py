"""GPU parity of the wave-pipelined layer ("不规则与流水化 AllToAll", section
"Wave-Scheduled 流水化"): dispatch(w), the experts of wave w and the combine of
the tokens whose last wave is w on three streams, so that dispatch(w+1),
experts(w) and combine(w-1) overlap.  The pipelined step must give the
oracle's rows and y, bit-identical to the sequential step; each per-wave call
must touch only its own rows or tokens."""
import numpy as np
import pytest
import torch

import oracle
from combine_moe_route_17_b300 import binding as B
from combine_moe_route_17_b300 import workloads as wl

from _parity import assert_full_parity, bf16_rows_to_u16, make_pipeline, run_gpu

pytestmark = pytest.mark.gpu

CASES = [
    wl.small_config(T=2400, H=264, E=64, k=6, R=8, W=4, bias="linear", bias_param=0.874, seed=2),
    wl.small_config(T=1600, H=512, E=128, k=8, R=16, W=8, bias="zipf", bias_param=1.0, seed=3),
    wl.small_config(T=1024, H=256, E=256, k=8, R=32, W=16, n_groups=8, topk_groups=4,
                    group_topn=2, bias="dirichlet", bias_param=0.3, seed=4),
    wl.small_config(T=520, H=40, E=32, k=4, R=4, W=16, bias="zipf", bias_param=1.0, seed=6),
    wl.small_config(T=300, H=8, E=1, k=1, R=1, W=1, seed=7),
]


def _last_wave(idx, E, W):
    return (idx // (E // W)).max(axis=1)


def _pipelined(cfg, inp):
    p = make_pipeline(cfg, inp)
    streams = [torch.cuda.current_stream(), torch.cuda.Stream(), torch.cuda.Stream()]
    p.step_pipelined(streams)
    torch.cuda.synchronize()
    assert B.get_device_error(p.ws) == 0
    res = p.results()
    res["out"] = bf16_rows_to_u16(p.recv)
    return res


@pytest.mark.parametrize("cfg", CASES, ids=lambda c: c.name)
def test_pipelined_step_matches_oracle_and_sequential(cfg):
    inp = wl.make_inputs(cfg)
    got = _pipelined(cfg, inp)
    ref = oracle.forward(cfg, inp)
    seq = run_gpu(cfg, inp)
    assert_full_parity(cfg, inp, {**got, "status": 0}, ref, rows=False)
    assert np.array_equal(got["out"], ref["out"]), "expert rows"
    assert np.array_equal(got["out"], seq["out"])
    assert np.array_equal(got["y"], seq["y"])


def test_pipelined_step_at_reduced_c2_in_a_graph():
    cfg = wl.reduced(wl.CONFIGS["c2"], T=8 * 512)
    inp = wl.make_inputs(cfg)
    p = make_pipeline(cfg, inp)
    s0 = torch.cuda.Stream()
    streams = [s0, torch.cuda.Stream(), torch.cuda.Stream()]
    g = torch.cuda.CUDAGraph()
    s0.wait_stream(torch.cuda.current_stream())
    with torch.cuda.graph(g, stream=s0):
        p.step_pipelined(streams)
    p.load_inputs(torch.from_numpy(inp["logits"]), torch.from_numpy(inp["x"].view(np.int16)),
                  torch.from_numpy(inp["scale"]))
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    assert B.get_device_error(p.ws) == 0
    seq = run_gpu(cfg, inp)
    got = p.results()
    assert np.array_equal(got["y"], seq["y"])
    assert np.array_equal(got["slot_of"], seq["slot_of"])


def test_combine_wave_writes_only_the_tokens_whose_last_wave_it_is():
    cfg = CASES[1]
    inp = wl.make_inputs(cfg)
    ref = oracle.forward(cfg, inp, with_rows=False)
    p = make_pipeline(cfg, inp)
    p.route()
    p.count()
    p.dispatch_waves()
    p.expert()
    p.combine()
    torch.cuda.synchronize()
    y_full = p.y.clone()
    lw = _last_wave(ref["idx"], cfg.E, cfg.W)
    p.y.view(torch.int16).fill_(0x7FC0)  # NaN sentinel
    done = np.zeros(cfg.T, bool)
    for w in range(cfg.W):
        p.combine_wave(w)
        torch.cuda.synchronize()
        done |= lw == w
        y = p.y.view(torch.int16).cpu().numpy().view(np.uint16)
        full = y_full.view(torch.int16).cpu().numpy().view(np.uint16)
        assert np.array_equal(y[done], full[done])
        assert (y[~done] == 0x7FC0).all()
    assert done.all()
    assert B.get_device_error(p.ws) == 0


def test_expert_wave_scales_only_its_rows():
    cfg = CASES[0]
    inp = wl.make_inputs(cfg)
    ref = oracle.forward(cfg, inp)
    p = make_pipeline(cfg, inp)
    p.route()
    p.count()
    p.dispatch_waves()
    torch.cuda.synchronize()
    Ew = cfg.E // cfg.W
    wave_of_row = np.empty(cfg.T * cfg.k, np.int64)
    wave_of_row[ref["slot_of"].reshape(-1)] = (ref["idx"] // Ew).reshape(-1)
    scaled = np.zeros(cfg.T * cfg.k, bool)
    for w in range(cfg.W):
        p.expert_wave(w)
        torch.cuda.synchronize()
        scaled |= wave_of_row == w
        rows = bf16_rows_to_u16(p.recv)
        assert np.array_equal(rows[scaled], ref["out"][scaled])
        assert np.array_equal(rows[~scaled], ref["recv"][~scaled])


def test_wave_entry_points_reject_bad_waves():
    cfg = CASES[0]
    inp = wl.make_inputs(cfg)
    p = make_pipeline(cfg, inp)
    for bad in (-2, cfg.W):
        with pytest.raises(B.MoEError) as e:
            p.combine_wave(bad)
        assert e.value.status == B.MOE_ERR_INVALID_ARG
        with pytest.raises(B.MoEError):
            p.expert_wave(bad)


@pytest.mark.parametrize("name", ["c2", "c4"])
def test_pipelined_step_at_full_size_in_a_graph(name):
    """The full-size step as bench.py --wave-scan times it (one captured graph,
    three streams, the workload's own W): y and the row maps bit-identical to
    the sequential step, maps equal to the oracle's in full, and y on sampled
    tokens equal to the oracle's."""
    cfg = wl.CONFIGS[name]
    inp = wl.make_inputs(cfg)
    p = make_pipeline(cfg, inp)
    s0 = torch.cuda.Stream()
    streams = [s0, torch.cuda.Stream(), torch.cuda.Stream()]
    s0.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s0):
        p.step_pipelined(streams)
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    assert B.get_device_error(p.ws) == 0
    y_pipe = p.y.clone()
    slot_pipe = p.slot_of.clone()
    q = make_pipeline(cfg, inp)
    q.route_count()
    q.dispatch_waves()
    q.expert()
    q.combine()
    torch.cuda.synchronize()
    assert torch.equal(y_pipe.view(torch.int16), q.y.view(torch.int16))
    assert torch.equal(slot_pipe, q.slot_of)
    ref = oracle.forward(cfg, {"logits": inp["logits"]}, with_rows=False)
    assert np.array_equal(slot_pipe.cpu().numpy(), ref["slot_of"])
    rng = np.random.default_rng(81)
    toks = np.unique(np.concatenate([rng.integers(0, cfg.T, 384), [0, cfg.T - 1]]))
    k = cfg.k
    compact = np.arange(len(toks) * k, dtype=np.int32).reshape(len(toks), k)
    out = oracle.expert_standin(np.repeat(inp["x"][toks], k, axis=0), ref["idx"][toks], compact,
                                inp["scale"])
    y_ref = oracle.combine(out, compact, ref["w"][toks])
    y = y_pipe.view(torch.int16)[torch.from_numpy(toks).cuda()].cpu().numpy().view(np.uint16)
    from _parity import assert_y

    assert_y(y, y_ref)
