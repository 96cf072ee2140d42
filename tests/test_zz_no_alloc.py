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


def test_noalloc_failure_shows_in_recv_base_and_the_next_call_is_clean():
    """The call returns before its kernel runs, so a failure found on the
    device comes back in the outputs: an expert index out of range (the count
    kernel's own bounds check skips the slot and raises the error) sets
    recv_base[R] = -MOE_ERR_DEVICE_CHECK.  The array's error word is cleared
    by the next call, which then matches the workspace entry point again."""
    cfg = wl.CONFIGS["c2"]
    idx = _idx(cfg)
    bad = idx.clone()
    bad[5, 2] = cfg.E
    out = _outputs(cfg)
    assert _noalloc(cfg, bad, out) == B.MOE_OK
    torch.cuda.synchronize()
    assert int(out["recv_base"][-1]) == -B.MOE_ERR_DEVICE_CHECK
    expect = _with_workspace(cfg, idx)
    for _ in range(2):
        again = _outputs(cfg)
        assert _noalloc(cfg, idx, again) == B.MOE_OK
        torch.cuda.synchronize()
        assert int(again["recv_base"][-1]) == cfg.T * cfg.k
        for name in expect:
            assert np.array_equal(again[name].cpu().numpy(), expect[name]), name


_FIRST_CALL_UNDER_CAPTURE = r"""
import ctypes, sys
import torch
sys.path.insert(0, sys.argv[1])
from combine_moe_route_17_b300 import binding as B
from combine_moe_route_17_b300 import workloads as wl
cfg = wl.CONFIGS["c1"]
shape = B.Shape.of(cfg)
idx = torch.zeros((cfg.T, cfg.k), dtype=torch.int32, device="cuda")
outs = [torch.zeros(n, dtype=dt, device="cuda") for n, dt in
        ((cfg.E, torch.int32), (cfg.R * cfg.E, torch.int32), (cfg.R * cfg.R, torch.int32),
         (cfg.R * (cfg.R + 1), torch.int64), (cfg.R * (cfg.R + 1), torch.int64),
         (cfg.R + 1, torch.int64))]
s = torch.cuda.Stream()
torch.cuda.synchronize()
g = torch.cuda.CUDAGraph()
with torch.cuda.graph(g, stream=s):
    st = B.lib().moe_build_send_counts_noalloc(ctypes.byref(shape), idx.data_ptr(),
                                               *[o.data_ptr() for o in outs], s.cuda_stream)
print("status", st)
"""


def test_noalloc_first_call_under_capture_is_refused():
    """In a fresh process the first call sets the array up (address lookup and
    zero-fill); made on a capturing stream, it is refused and launches
    nothing, so no zero-fill is left to a graph that may never run."""
    import os
    import subprocess
    import sys

    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-c", _FIRST_CALL_UNDER_CAPTURE, root],
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    assert f"status {B.MOE_ERR_INVALID_ARG}" in r.stdout, r.stdout
