"""HostBatchRunner: batches in pinned host memory, two device buffer sets,
copy-in / compute / read-back on three streams.  Every step's y and
statistics must equal those of the plain step on the same batch (bit for
bit) and the oracle's, whatever the overlap of neighbouring steps."""
import numpy as np
import pytest
import torch

import oracle
from combine_moe_route_17_b300 import HostBatchRunner
from combine_moe_route_17_b300 import workloads as wl

from _parity import assert_y, run_gpu

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("fuse_route", [False, True], ids=["two_launches", "route_and_count"])
def test_double_buffered_steps_match_the_plain_step(fuse_route):
    cfg = wl.small_config(T=2400, H=264, E=64, k=6, R=8, W=4, bias="linear", bias_param=0.874,
                          seed=31)
    batches = [wl.make_inputs(cfg, seed=s) for s in (31, 32, 33)]
    for b in batches[1:]:
        b["scale"] = batches[0]["scale"]  # one set of experts
    want = [run_gpu(cfg, b, keep_rows=False) for b in batches]
    runner = HostBatchRunner(cfg, device="cuda", fuse_route=fuse_route)
    runner.load_scale(batches[0]["scale"])
    h_in = [(torch.from_numpy(b["logits"]).pin_memory(),
             torch.from_numpy(b["x"].view(np.int16)).pin_memory()) for b in batches]
    n = 7
    h_y = [torch.empty((cfg.T, cfg.H), dtype=torch.int16).pin_memory() for _ in range(n)]
    h_st = [torch.zeros(8, dtype=torch.float64).pin_memory() for _ in range(n)]
    for i in range(n):
        runner.step(i, *h_in[i % 3], h_y[i], h_st[i])
    runner.join(torch.cuda.current_stream())
    torch.cuda.synchronize()
    runner.check_device_error()
    for i in range(n):
        ref = want[i % 3]
        assert np.array_equal(h_y[i].numpy().view(np.uint16), ref["y"]), f"step {i}"
        assert np.array_equal(h_st[i].numpy(), ref["pipeline"].stats.cpu().numpy()), \
            f"statistics of step {i}"
    ref0 = oracle.forward(cfg, batches[0])
    assert_y(h_y[0].numpy().view(np.uint16), ref0["y"])
