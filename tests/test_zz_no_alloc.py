"""The allocation-free send-count entry point, moe_build_send_counts_noalloc.

It serves callers that cannot call cudaMalloc (a memory planner that needs
the alltoallv counts before any exchange buffer exists, a runtime whose
device memory all belongs to its own pool): they pass only inputs and
outputs, and the scratch is a fixed array inside the library.  These tests
call it through the C ABI and check it against moe_build_send_counts (with a
caller workspace) on two calls in a row, bit for bit, since every output is
an integer count or offset.  The file is collected last so that a run that
stops at the first failure has already run every other test; it also passes
on its own in a fresh process (its first call sets the array up)."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from combine_moe_route_17_b300 import binding as B
from combine_moe_route_17_b300 import workloads as wl

pytestmark = pytest.mark.gpu

OUTS = (("c", torch.int32, lambda c: (c.E,)), ("C", torch.int32, lambda c: (c.R, c.E)),
        ("S", torch.int32, lambda c: (c.R, c.R)),
        ("send_off", torch.int64, lambda c: (c.R, c.R + 1)),
        ("recv_off", torch.int64, lambda c: (c.R, c.R + 1)),
        ("recv_base", torch.int64, lambda c: (c.R + 1,)))


def _outputs(cfg):
    return {n: torch.full(f(cfg), -1, dtype=dt, device="cuda") for n, dt, f in OUTS}


def _idx(cfg):
    idx, _ = oracle.route_topk(wl.make_logits(cfg), cfg.k, cfg.n_groups, cfg.topk_groups,
                               cfg.group_topn)
    return torch.from_numpy(idx).cuda()


def _noalloc(cfg, idx, out):
    L = B.lib()
    shape = B.Shape.of(cfg)
    return L.moe_build_send_counts_noalloc(
        ctypes.byref(shape), idx.data_ptr(), out["c"].data_ptr(), out["C"].data_ptr(),
        out["S"].data_ptr(), out["send_off"].data_ptr(), out["recv_off"].data_ptr(),
        out["recv_base"].data_ptr(), torch.cuda.current_stream().cuda_stream)


def _with_workspace(cfg, idx):
    shape = B.Shape.of(cfg)
    out = _outputs(cfg)
    ws = B.new_workspace(shape)
    B.build_send_counts(shape, idx, out, ws)
    torch.cuda.synchronize()
    assert B.get_device_error(ws) == B.MOE_OK
    return {k: v.cpu().numpy() for k, v in out.items()}


def test_noalloc_counts_match_the_workspace_entry_point_on_two_calls_in_a_row():
    cfgs = [wl.CONFIGS["c2"], wl.CONFIGS["c4"]]
    idxs = [_idx(c) for c in cfgs]
    expect = [_with_workspace(c, i) for c, i in zip(cfgs, idxs)]
    outs = [_outputs(c) for c in cfgs]
    # two calls back to back on one stream: the second reuses the array the
    # first left behind, with another shape
    assert _noalloc(cfgs[0], idxs[0], outs[0]) == B.MOE_OK
    assert _noalloc(cfgs[1], idxs[1], outs[1]) == B.MOE_OK
    torch.cuda.synchronize()
    for cfg, out, exp in zip(cfgs, outs, expect):
        for name in exp:
            assert np.array_equal(out[name].cpu().numpy(), exp[name]), (cfg.name, name)
    # and the same shape twice more, with the array's last contents from above
    for _ in range(2):
        again = _outputs(cfgs[0])
        assert _noalloc(cfgs[0], idxs[0], again) == B.MOE_OK
        torch.cuda.synchronize()
        for name in expect[0]:
            assert np.array_equal(again[name].cpu().numpy(), expect[0][name]), name


def test_noalloc_rejects_shapes_beyond_its_scratch():
    big = wl.CONFIGS["c3"].replace(T=262144)  # needs far more than 4 MiB of scratch
    assert B.workspace_size(B.Shape.of(big)) > (4 << 20)
    L = B.lib()
    shape = B.Shape.of(big)
    fake = 0x100000  # never dereferenced: the size check comes first
    st = L.moe_build_send_counts_noalloc(ctypes.byref(shape), fake, fake, fake, fake, fake,
                                         fake, fake, None)
    assert st == B.MOE_ERR_UNSUPPORTED
