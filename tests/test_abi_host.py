"""CPU-only checks of the C ABI: the library loads, exports every symbol the
header declares, and rejects bad shapes and pointers on the host before any
launch (no GPU needed: those paths never reach the CUDA runtime)."""
import ctypes
import os
import re

import pytest

import combine_moe_route_17_b300 as pkg
from combine_moe_route_17_b300 import binding as B
from combine_moe_route_17_b300 import workloads as wl

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe_route.h")


@pytest.fixture(scope="module")
def L():
    from combine_moe_route_17_b300 import build

    build.build()
    return pkg.lib()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:moe_status|const char\*|int)\s+(moe_\w+)\s*\(", src,
                                 flags=re.M)))


def test_header_declares_the_contract():
    names = declared_functions()
    for must in ("moe_workspace_size", "moe_route_topk", "moe_build_send_counts",
                 "moe_dispatch", "moe_combine", "moe_imbalance_stats", "moe_get_device_error",
                 "moe_status_string"):
        assert must in names


def test_library_exports_every_declared_symbol(L):
    for name in declared_functions():
        assert hasattr(L, name), name
        assert name in B.SIGNATURES, f"binding lacks {name}"
    assert set(B.SIGNATURES) == set(declared_functions())
    assert pkg.abi_version() == 1


def test_status_strings(L):
    for code in range(6):
        assert pkg.status_string(code) not in ("", "unknown status")
    assert pkg.status_string(99) == "unknown status"


def _shape(**kw):
    base = dict(T=64, H=64, E=8, k=2, R=2, W=1, n_groups=1, topk_groups=0, group_topn=0)
    base.update(kw)
    return B.Shape(**base)


@pytest.mark.parametrize("kw,code", [
    (dict(T=63), 1), (dict(H=12), 1), (dict(H=0), 1), (dict(E=7), 1), (dict(k=9), 1),
    (dict(W=3), 1), (dict(R=3, T=64, E=9), 1), (dict(R=4, T=64, E=6), 1), (dict(k=0), 1), (dict(T=-2), 1),
    (dict(E=512, R=2), 2), (dict(k=17, E=32), 2), (dict(R=128, E=256, T=128), 2),
    (dict(n_groups=3), 1), (dict(n_groups=4, topk_groups=0, group_topn=1), 1),
    (dict(n_groups=4, topk_groups=1, group_topn=1, k=3), 1),
    (dict(n_groups=4, topk_groups=2, group_topn=3), 1),
    (dict(T=(1 << 27), k=16, E=16, R=1), 2),
])
def test_shape_validation(L, kw, code):
    assert L.moe_validate_shape(ctypes.byref(_shape(**kw))) == code


def test_valid_shapes_and_workspace_size(L):
    for cfg in list(wl.CONFIGS.values()) + wl.SWEEP[::7]:
        s = B.Shape.of(cfg)
        assert L.moe_validate_shape(ctypes.byref(s)) == 0, cfg.name
        n = B.workspace_size(s)
        assert n >= 256 + 4 * cfg.T * cfg.k
        assert n % 256 == 0
    assert B.workspace_size(_shape(T=0)) > 0


def test_calls_reject_bad_arguments_before_launch(L):
    s = _shape()
    sp = ctypes.byref(s)
    fake = 0x100000  # never dereferenced: validation fails first
    # null / misaligned buffers
    assert L.moe_route_topk(sp, None, fake, fake, None, None) == 1
    assert L.moe_route_topk(sp, fake + 2, fake, fake, None, None) == 1
    assert L.moe_build_send_counts(sp, fake, fake, fake, fake, fake, fake, fake, None, 0,
                                   None) == 1
    assert L.moe_build_send_counts(sp, fake, fake, fake, fake, fake, fake, fake, fake, 16,
                                   None) == 1  # workspace too small
    ws_ok = B.workspace_size(s)
    assert L.moe_expert_offsets(sp, fake, ws_ok, None, None) == 1  # no output
    assert L.moe_expert_offsets(sp, fake, ws_ok, fake + 2, None) == 1  # misaligned output
    assert L.moe_expert_offsets(sp, fake, ws_ok - 256, fake, None) == 1  # workspace too small
    assert L.moe_expert_offsets(sp, fake + 16, ws_ok, fake, None) == 1  # workspace misaligned
    assert L.moe_dispatch(sp, fake + 8, fake, fake, ws_ok, -1, 0, None, fake, fake, None, None,
                          None) == 1  # x not 16-byte aligned
    assert L.moe_dispatch(sp, fake, fake, fake, ws_ok, 1, 0, None, fake, fake, None, None,
                          None) == 1  # wave out of range (W = 1)
    big = _shape(H=40000)  # three 80 KB rows per warp exceed the bulk path's buffers
    ws_big = B.workspace_size(big)
    assert L.moe_dispatch(ctypes.byref(big), fake, fake, fake, ws_big, -1, B.MOE_BULK_COPY, None,
                          fake, fake, None, None, None) == 2
    assert L.moe_dispatch(sp, fake, fake, fake, ws_ok, -1, 8, None, fake, fake, None, None,
                          None) == 1  # unknown flag
    assert L.moe_dispatch(sp, fake, fake, fake, ws_ok, -1, 1, None, fake, fake, None, None,
                          None) == 1  # staged without send
    assert L.moe_combine(sp, fake, None, fake, None, 0, 0, None, None, fake, None) == 1
    assert L.moe_combine(sp, fake, fake, fake, None, 0, 1, fake, fake, fake, None) == 1
    assert L.moe_all_to_all(sp, fake, ws_ok, -1, 2, fake, fake + 16, None) == 1
    assert L.moe_all_to_all(sp, fake, ws_ok, -1, 0, fake, fake, None) == 1  # in place
    assert L.moe_imbalance_stats(sp, None, fake, None, None) == 1
    assert L.moe_expert_standin(sp, fake, fake, None, fake, None) == 1
    assert L.moe_get_device_error(None, None) == 1
    assert L.moe_workspace_init(None, 0, None) == 1
    bad = _shape(T=63)
    assert L.moe_route_topk(ctypes.byref(bad), fake, fake, fake, None, None) == 1


def test_python_binding_raises(L):
    import torch

    s = _shape()
    with pytest.raises(ValueError):
        B.route_topk(s, torch.zeros(64, 8), torch.zeros(64, 2, dtype=torch.int32),
                     torch.zeros(64, 2))  # CPU tensors are refused


@pytest.mark.parametrize("f", [0.0, 0.1, 0.5, 1.0, 1.1, 1.25, 1.3333333, 2.0, 3.7])
def test_expert_capacity_matches_the_oracle(L, f):
    """The library's EC = ceil(k f T / E) (host arithmetic, no launch) equals
    the oracle's for every named workload."""
    import oracle

    for cfg in wl.CONFIGS.values():
        assert B.expert_capacity(B.Shape.of(cfg), f) == oracle.expert_capacity(cfg.T, cfg.E,
                                                                               cfg.k, f)


def test_expert_capacity_rejects_bad_factors(L):
    s = B.Shape.of(wl.CONFIGS["c1"])
    for f in (-0.5, float("nan"), 1e9):
        with pytest.raises(B.MoEError):
            B.expert_capacity(s, f)


def test_pack_gated_weights_interleaves_128_row_blocks():
    import torch

    E, F, H = 2, 256, 8
    w1 = torch.arange(E * F * H, dtype=torch.float32).reshape(E, F, H)
    w3 = -w1 - 1
    p = B.pack_gated_weights(w1, w3)
    assert p.shape == (E, 2 * F, H)
    for e in range(E):
        for b in range(F // 128):
            assert torch.equal(p[e, 256 * b:256 * b + 128], w1[e, 128 * b:128 * (b + 1)])
            assert torch.equal(p[e, 256 * b + 128:256 * (b + 1)], w3[e, 128 * b:128 * (b + 1)])
    with pytest.raises(ValueError):
        B.pack_gated_weights(w1[:, :96], w3[:, :96])
