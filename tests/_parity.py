"""Shared helpers of the GPU parity tests: run the CUDA path through the
C-ABI binding and compare with the CPU oracle on the same seeded inputs.

Tolerances:
  indices, counts, offsets, row maps, permuted rows, statistics: bit-exact;
  gate weights: |w_gpu - w_oracle| <= 1e-6 (fp32 expf, fp32 sum and divide on
    the GPU against an fp64 softmax rounded once: the error budget is below
    6e-7 for k <= 16);
  combine: |y_gpu - y_oracle| <= 1e-2 |y_oracle| elementwise (fp32
    accumulation rounded once to bf16 against fp64 rounded once: at most one
    bf16 ulp, 2^-7 relative, apart).
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from combine_moe_route_17_b300 import MoEPipeline
from combine_moe_route_17_b300 import binding as B

W_TOL = 1e-6
Y_RTOL = 1e-2


def bf16_rows_to_u16(t: torch.Tensor) -> np.ndarray:
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def make_pipeline(cfg, inp, staged=False, fuse_route=False, concurrent_waves=True,
                  bulk_copy=False):
    p = MoEPipeline(cfg, device="cuda", staged=staged, fuse_route=fuse_route,
                    concurrent_waves=concurrent_waves, bulk_copy=bulk_copy)
    p.load_inputs(torch.from_numpy(inp["logits"]), torch.from_numpy(inp["x"].view(np.int16)),
                  torch.from_numpy(inp["scale"]))
    return p


def run_gpu(cfg, inp, staged=False, keep_rows=True, waves=True, fuse_route=False,
            concurrent_waves=True, bulk_copy=False):
    p = make_pipeline(cfg, inp, staged, fuse_route, concurrent_waves, bulk_copy)
    p.route_count()
    if waves:
        p.dispatch_waves()
    else:
        p.dispatch(-1)
    torch.cuda.synchronize()
    res = {}
    if keep_rows:
        res["recv"] = bf16_rows_to_u16(p.recv)
        if staged:
            res["send"] = bf16_rows_to_u16(p.send)
            res["send_pos"] = p.send_pos.cpu().numpy()
    p.expert()
    if keep_rows:
        torch.cuda.synchronize()
        res["out"] = bf16_rows_to_u16(p.recv)
    p.combine()
    p.imbalance()
    torch.cuda.synchronize()
    status = B.get_device_error(p.ws)
    res.update(p.results())
    res["status"] = status
    res["pipeline"] = p
    return res


def assert_routing(got, ref):
    assert np.array_equal(got["idx"], ref["idx"]), "routing indices"
    dw = np.abs(got["w"].astype(np.float64) - ref["w"].astype(np.float64))
    assert dw.max(initial=0.0) <= W_TOL, f"gate weights max|dw|={dw.max()}"


def assert_counts(got, ref):
    for key in ("c", "C", "S", "send_off", "recv_off", "recv_base"):
        assert np.array_equal(got[key], ref[key]), key


def assert_maps(got, ref):
    assert np.array_equal(got["slot_of"], ref["slot_of"]), "slot_of"
    assert np.array_equal(got["src_row"], ref["src_row"]), "src_row"


def assert_y(y_gpu_u16, y_ref_u16):
    yg = oracle.bf16_to_f64(y_gpu_u16)
    yr = oracle.bf16_to_f64(y_ref_u16)
    bad = np.abs(yg - yr) > Y_RTOL * np.abs(yr)
    assert not bad.any(), f"combine: {int(bad.sum())} elements outside rel {Y_RTOL}"


def assert_stats(got, ref):
    g, r = got["stats"], ref["stats"]
    for key in ("max_load", "min_load", "gini_num", "gini_den"):
        assert g[key] == r[key], key
    for key in ("max_over_mean", "hot_over_cold", "gini"):
        assert g[key] == r[key] or (np.isinf(g[key]) and np.isinf(r[key])), key
    assert np.array_equal(got["rank_load"], ref["stats"]["rank_load"])


def assert_full_parity(cfg, inp, got, ref, rows=True):
    assert got["status"] == 0, B.status_string(got["status"])
    assert_routing(got, ref)
    assert_counts(got, ref)
    assert_maps(got, ref)
    if rows:
        assert np.array_equal(got["recv"], ref["recv"]), "recv rows"
        assert np.array_equal(got["out"], ref["out"]), "stand-in expert rows"
        if "send" in got:
            assert np.array_equal(got["send"], ref["send"]), "send rows"
            assert np.array_equal(got["send_pos"], ref["send_pos"]), "send_pos"
    assert_y(got["y"], ref["y"])
    assert_stats(got, ref)
