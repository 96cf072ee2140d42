"""GPU parity of the expert-major recv layout (flag MOE_EXPERT_MAJOR): recv
rows ordered (destination rank, expert, source, token, slot), each expert's
rows one run (MoE survey, section 1.1, step 2).  Maps and rows bit-exact
with the oracle, fused and staged; y bit-identical to the rank-major
layout's (the combine follows slot_of); each wave writes one contiguous run."""
import numpy as np
import pytest
import torch

import oracle
from combine_moe_route_17_b300 import MoEPipeline
from combine_moe_route_17_b300 import binding as B
from combine_moe_route_17_b300 import workloads as wl

from _parity import assert_y, bf16_rows_to_u16

pytestmark = pytest.mark.gpu

SHAPES = [
    wl.small_config(T=1200, H=128, E=16, k=2, R=4, W=1, seed=1),
    wl.small_config(T=2400, H=264, E=64, k=6, R=8, W=4, bias="linear", bias_param=0.874, seed=2),
    wl.small_config(T=1600, H=512, E=128, k=8, R=16, W=8, bias="zipf", bias_param=1.0, seed=3),
    wl.small_config(T=1024, H=256, E=256, k=8, R=32, W=16, n_groups=8, topk_groups=4,
                    group_topn=2, bias="dirichlet", bias_param=0.3, seed=4),
    wl.small_config(T=520, H=40, E=32, k=4, R=4, W=16, bias="zipf", bias_param=1.0, seed=6),
]


def _run(cfg, inp, staged):
    p = MoEPipeline(cfg, device="cuda", staged=staged, expert_major=True)
    p.load_inputs(torch.from_numpy(inp["logits"]), torch.from_numpy(inp["x"].view(np.int16)),
                  torch.from_numpy(inp["scale"]))
    p.route()
    p.count()
    p.dispatch_waves()
    torch.cuda.synchronize()
    got = {"slot_of": p.slot_of.cpu().numpy(), "src_row": p.src_row.cpu().numpy(),
           "recv": bf16_rows_to_u16(p.recv), "off": p.expert_offsets().cpu().numpy()}
    p.expert()
    p.combine()
    torch.cuda.synchronize()
    got["y"] = p.y.view(torch.int16).cpu().numpy().view(np.uint16)
    got["status"] = B.get_device_error(p.ws)
    return got


@pytest.mark.parametrize("staged", [False, True], ids=["fused", "staged"])
@pytest.mark.parametrize("cfg", SHAPES, ids=lambda c: c.name)
def test_expert_major_matches_oracle(cfg, staged):
    inp = wl.make_inputs(cfg)
    ref = oracle.forward(cfg, inp)
    em = oracle.dispatch_maps_expert_major(ref["idx"], cfg.E)
    got = _run(cfg, inp, staged)
    assert got["status"] == 0
    assert np.array_equal(got["slot_of"], em["slot_of"])
    assert np.array_equal(got["src_row"], em["src_row"])
    assert np.array_equal(got["off"], em["expert_off"])
    recv = np.zeros_like(got["recv"])
    recv[em["slot_of"].ravel()] = np.repeat(inp["x"], cfg.k, axis=0)
    assert np.array_equal(got["recv"], recv)
    assert_y(got["y"], ref["y"])
    # the same y as the rank-major layout, bit for bit
    from _parity import run_gpu

    assert np.array_equal(got["y"], run_gpu(cfg, inp, staged=staged)["y"])


def test_each_wave_writes_one_contiguous_run():
    cfg = SHAPES[2]
    inp = wl.make_inputs(cfg)
    ref = oracle.forward(cfg, inp, with_rows=False)
    em = oracle.dispatch_maps_expert_major(ref["idx"], cfg.E)
    p = MoEPipeline(cfg, device="cuda", expert_major=True)
    p.load_inputs(torch.from_numpy(inp["logits"]), torch.from_numpy(inp["x"].view(np.int16)),
                  torch.from_numpy(inp["scale"]))
    p.route()
    p.count()
    p.recv.view(torch.int16).fill_(0x7FC0)
    Ew = cfg.E // cfg.W
    off = em["expert_off"]
    want = np.zeros((cfg.T * cfg.k, cfg.H), np.uint16)
    want[em["slot_of"].ravel()] = np.repeat(inp["x"], cfg.k, axis=0)
    for w in range(cfg.W):
        p.dispatch(w)
        torch.cuda.synchronize()
        rows = bf16_rows_to_u16(p.recv)
        hi = off[(w + 1) * Ew]
        assert np.array_equal(rows[:hi], want[:hi])  # waves 0..w: one prefix run
        assert (rows[hi:] == 0x7FC0).all()
    assert B.get_device_error(p.ws) == 0


def test_expert_major_maps_at_full_size():
    cfg = wl.CONFIGS["c3"]
    lg = wl.make_logits(cfg)
    ref = oracle.forward(cfg, {"logits": lg}, with_rows=False)
    em = oracle.dispatch_maps_expert_major(ref["idx"], cfg.E)
    inp = {"logits": lg, "x": wl.make_x(cfg, rows=cfg.T), "scale": wl.make_scales(cfg)}
    p = MoEPipeline(cfg, device="cuda", expert_major=True)
    p.load_inputs(torch.from_numpy(inp["logits"]), torch.from_numpy(inp["x"].view(np.int16)),
                  torch.from_numpy(inp["scale"]))
    p.route()
    p.count()
    p.dispatch_waves()
    torch.cuda.synchronize()
    assert B.get_device_error(p.ws) == 0
    assert np.array_equal(p.slot_of.cpu().numpy(), em["slot_of"])
    assert np.array_equal(p.src_row.cpu().numpy(), em["src_row"])
