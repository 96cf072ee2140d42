"""GPU parity of the capacity-factor variant (MoE survey, section 1.1,
"专家容量", eq. 3 and step 2) against the oracle: the capacity (host), the
per-slot rows or drops and the per-expert drop counts bit-exact, the
[E][EC][H] rows (kept rows bit copies of x, padding zero) and the stand-in
rows bit-exact, the combine within the path's tolerance."""
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
    wl.small_config(T=1200, H=128, E=16, k=2, R=4, seed=1),
    wl.small_config(T=2400, H=264, E=64, k=6, R=8, W=4, bias="linear", bias_param=0.874, seed=2),
    wl.small_config(T=1600, H=512, E=128, k=8, R=16, bias="zipf", bias_param=1.0, seed=3),
    wl.small_config(T=1024, H=256, E=256, k=8, R=32, n_groups=8, topk_groups=4, group_topn=2,
                    bias="dirichlet", bias_param=0.3, seed=4),
    wl.small_config(T=300, H=8, E=1, k=1, R=1, seed=7),
]


def _run(cfg, inp, f):
    p = MoEPipeline(cfg, device="cuda", capacity_factor=f)
    p.load_inputs(torch.from_numpy(inp["logits"]), torch.from_numpy(inp["x"].view(np.int16)),
                  torch.from_numpy(inp["scale"]))
    p.cap_rows.view(torch.int16).fill_(0x7FC0)  # every row must be written
    p.route()
    p.count()
    p.dispatch_capacity()
    torch.cuda.synchronize()
    got = {"EC": p.capacity, "cap_slot": p.cap_slot.cpu().numpy(),
           "dropped": p.dropped.cpu().numpy(), "cap_rows": bf16_rows_to_u16(p.cap_rows)}
    p.expert_capacity()
    p.combine_capacity()
    torch.cuda.synchronize()
    got["cap_out"] = bf16_rows_to_u16(p.cap_rows)
    got["y"] = p.y.view(torch.int16).cpu().numpy().view(np.uint16)
    got["status"] = B.get_device_error(p.ws)
    return got


@pytest.mark.parametrize("f", [0.5, 1.0, 1.25, 3.0])
@pytest.mark.parametrize("cfg", SHAPES, ids=lambda c: c.name)
def test_capacity_path_matches_oracle(cfg, f):
    inp = wl.make_inputs(cfg)
    ref = oracle.forward_capacity(cfg, inp, f)
    got = _run(cfg, inp, f)
    assert got["status"] == 0
    assert got["EC"] == ref["EC"]
    assert np.array_equal(got["cap_slot"], ref["cap_slot"])
    assert np.array_equal(got["dropped"], ref["dropped"])
    assert np.array_equal(got["cap_rows"], ref["cap_rows"])
    assert np.array_equal(got["cap_out"], ref["cap_out"])
    assert_y(got["y"], ref["y"])


def test_zero_capacity_drops_everything():
    cfg = SHAPES[1]
    inp = wl.make_inputs(cfg)
    got = _run(cfg, inp, 0.0)
    assert got["EC"] == 0 and (got["cap_slot"] == -1).all()
    assert (got["y"] == 0).all()
    assert got["status"] == 0


@pytest.mark.parametrize("name,f", [("c2", 1.0), ("c3", 1.25)])
def test_capacity_at_full_size(name, f):
    """Maps and drop counts in full; rows and y on sampled tokens."""
    cfg = wl.CONFIGS[name]
    inp = wl.make_inputs(cfg)
    ref = oracle.forward_capacity(cfg, inp, f, with_rows=False)
    p = MoEPipeline(cfg, device="cuda", capacity_factor=f)
    p.load_inputs(torch.from_numpy(inp["logits"]), torch.from_numpy(inp["x"].view(np.int16)),
                  torch.from_numpy(inp["scale"]))
    p.route()
    p.count()
    p.dispatch_capacity()
    p.expert_capacity()
    p.combine_capacity()
    torch.cuda.synchronize()
    assert B.get_device_error(p.ws) == 0
    assert p.capacity == ref["EC"]
    assert np.array_equal(p.cap_slot.cpu().numpy(), ref["cap_slot"])
    assert np.array_equal(p.dropped.cpu().numpy(), ref["dropped"])
    rng = np.random.default_rng(99)
    toks = np.unique(rng.integers(0, cfg.T, 512))
    cs = ref["cap_slot"][toks]
    rows = bf16_rows_to_u16(p.cap_rows[torch.from_numpy(np.maximum(cs, 0).reshape(-1)).cuda()])
    kept = (cs >= 0).reshape(-1)
    x_rep = np.repeat(inp["x"][toks], cfg.k, axis=0)
    # stand-in rows: bf16(s_e * x) on the kept slots
    compact = np.arange(len(toks) * cfg.k, dtype=np.int32).reshape(len(toks), cfg.k)
    want = oracle.expert_standin(x_rep, ref["idx"][toks], compact, inp["scale"])
    assert np.array_equal(rows[kept], want[kept])
    y = p.y.view(torch.int16).cpu().numpy().view(np.uint16)[toks]
    cslot = np.where(cs >= 0, compact, -1).astype(np.int32)
    assert_y(y, oracle.capacity_combine(want, cslot, ref["w"][toks]))


def test_capacity_host_rejects():
    cfg = SHAPES[0]
    inp = wl.make_inputs(cfg)
    p = MoEPipeline(cfg, device="cuda", capacity_factor=1.0)
    with pytest.raises(B.MoEError):
        B.dispatch_capacity(p.shape, -1, p.x, p.idx, p.ws, p.cap_rows, p.cap_slot)
    with pytest.raises(B.MoEError):
        B.dispatch_capacity(p.shape, 1 << 40, p.x, p.idx, p.ws, p.cap_rows, p.cap_slot)
    with pytest.raises(B.MoEError):
        B.combine_capacity(p.shape, -3, p.cap_rows, p.cap_slot, p.w, p.y)
