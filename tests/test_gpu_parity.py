"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle on the
same seeded inputs, at sizes the oracle finishes in seconds that span several
look-back tiles per source and a ragged last tile."""
import numpy as np
import pytest
import torch

import oracle
from combine_moe_route_17_b300 import binding as B
from combine_moe_route_17_b300 import workloads as wl

from _parity import assert_full_parity, run_gpu

pytestmark = pytest.mark.gpu

SMALL = [
    # several 128-token tiles per source + a ragged tail (Tr = 300)
    wl.small_config(T=1200, H=128, E=16, k=2, R=4, W=1, seed=1),
    wl.small_config(T=2400, H=264, E=64, k=6, R=8, W=4, bias="linear", bias_param=0.874, seed=2),
    wl.small_config(T=1600, H=512, E=128, k=8, R=16, W=8, bias="zipf", bias_param=1.0, seed=3),
    wl.small_config(T=1024, H=256, E=256, k=8, R=32, W=16, n_groups=8, topk_groups=4,
                    group_topn=2, bias="dirichlet", bias_param=0.3, seed=4),
    wl.small_config(T=1280, H=64, E=128, k=8, R=64, W=16, bias="dirichlet", bias_param=0.1,
                    seed=5),
    # W that splits a rank (E/W < E/R) and W > R
    wl.small_config(T=520, H=40, E=32, k=4, R=4, W=16, bias="zipf", bias_param=1.0, seed=6),
    # extremes of k and E
    wl.small_config(T=300, H=8, E=1, k=1, R=1, W=1, seed=7),
    wl.small_config(T=256, H=24, E=16, k=16, R=2, W=2, seed=8),
    wl.small_config(T=512, H=64, E=256, k=16, R=64, W=256, bias="dirichlet", bias_param=1.0,
                    seed=9),
    wl.small_config(T=777, H=16, E=3, k=1, R=1, W=3, seed=10),
    # group-limited variants
    wl.small_config(T=640, H=32, E=64, k=6, R=8, W=2, n_groups=8, topk_groups=3, group_topn=2,
                    seed=11),
    wl.small_config(T=384, H=16, E=12, k=3, R=3, W=4, n_groups=4, topk_groups=2, group_topn=3,
                    seed=12),
]


@pytest.mark.parametrize("concurrent", [True, False], ids=["concurrent_waves", "waves_in_order"])
@pytest.mark.parametrize("fuse_route", [True, False], ids=["route_and_count", "two_launches"])
@pytest.mark.parametrize("cfg", SMALL, ids=lambda c: c.name)
def test_fused_path_matches_oracle(cfg, fuse_route, concurrent):
    inp = wl.make_inputs(cfg)
    got = run_gpu(cfg, inp, fuse_route=fuse_route, concurrent_waves=concurrent)
    ref = oracle.forward(cfg, inp)
    assert_full_parity(cfg, inp, got, ref)


@pytest.mark.parametrize("staged", [False, True], ids=["fused", "staged"])
@pytest.mark.parametrize("concurrent", [True, False], ids=["concurrent_waves", "waves_in_order"])
@pytest.mark.parametrize("cfg", SMALL, ids=lambda c: c.name)
def test_bulk_copy_path_matches_oracle(cfg, concurrent, staged):
    """MOE_BULK_COPY: the row copies through shared memory by the bulk-copy
    engine give the same rows and maps as the register path and the oracle."""
    inp = wl.make_inputs(cfg)
    got = run_gpu(cfg, inp, staged=staged, concurrent_waves=concurrent, bulk_copy=True)
    ref = oracle.forward(cfg, inp)
    assert_full_parity(cfg, inp, got, ref)


@pytest.mark.parametrize("cfg", SMALL[:6], ids=lambda c: c.name)
def test_staged_path_matches_oracle_and_fused(cfg):
    inp = wl.make_inputs(cfg)
    got = run_gpu(cfg, inp, staged=True)
    ref = oracle.forward(cfg, inp)
    assert_full_parity(cfg, inp, got, ref)
    fused = run_gpu(cfg, inp, staged=False)
    assert np.array_equal(fused["recv"], got["recv"])
    assert np.array_equal(fused["y"], got["y"])


@pytest.mark.parametrize("cfg", [wl.CONFIGS[n] for n in ("c1", "c2", "c3", "c4")],
                         ids=lambda c: c.name)
def test_named_workloads_at_reduced_size(cfg):
    small = wl.reduced(cfg, T=cfg.R * 160).replace(H=min(cfg.H, 512))
    inp = wl.make_inputs(small)
    got = run_gpu(small, inp)
    ref = oracle.forward(small, inp)
    assert_full_parity(small, inp, got, ref)


def test_waves_write_only_their_rows():
    cfg = wl.small_config(T=640, H=64, E=32, k=4, R=4, W=8, bias="zipf", bias_param=1.0, seed=21)
    inp = wl.make_inputs(cfg)
    ref = oracle.forward(cfg, inp)
    from _parity import make_pipeline

    p = make_pipeline(cfg, inp)
    p.route()
    p.count()
    sentinel = torch.full_like(p.recv, float("nan"))
    p.recv.copy_(sentinel)
    p.slot_of.fill_(-7)
    Ew = cfg.E // cfg.W
    seen = np.zeros(cfg.T * cfg.k, bool)
    for w in range(cfg.W):
        p.dispatch(w)
        torch.cuda.synchronize()
        recv = p.recv.view(torch.int16).cpu().numpy().view(np.uint16)
        in_wave = (ref["idx"] // Ew == w)
        rows = ref["slot_of"][in_wave]
        seen[rows] = True
        assert np.array_equal(recv[seen], ref["recv"][seen])
        assert (recv[~seen] == 0x7FC0).all()  # NaN sentinel untouched
        so = p.slot_of.cpu().numpy()
        done = (ref["idx"] // Ew <= w)
        assert np.array_equal(so[done], ref["slot_of"][done])
        assert (so[~done] == -7).all()
    assert seen.all()
    assert B.get_device_error(p.ws) == 0


def test_exchange_round_trip_per_wave():
    cfg = wl.small_config(T=960, H=48, E=64, k=6, R=8, W=16, bias="linear", bias_param=0.9,
                          seed=22)
    inp = wl.make_inputs(cfg)
    ref = oracle.forward(cfg, inp)
    from _parity import make_pipeline

    p = make_pipeline(cfg, inp, staged=True)
    p.route()
    p.count()
    send = torch.zeros_like(p.recv)
    send_pos = torch.empty_like(p.slot_of)
    B.permute_by_device(p.shape, p.x, p.idx, p.ws, send, send_pos)
    recv = torch.zeros_like(p.recv)
    for w in range(cfg.W):
        B.all_to_all(p.shape, p.ws, send, recv, wave=w, direction=0)
    back = torch.zeros_like(p.recv)
    for w in reversed(range(cfg.W)):
        B.all_to_all(p.shape, p.ws, recv, back, wave=w, direction=1)
    torch.cuda.synchronize()
    u16 = lambda t: t.view(torch.int16).cpu().numpy().view(np.uint16)  # noqa: E731
    assert np.array_equal(u16(send), ref["send"])
    assert np.array_equal(send_pos.cpu().numpy(), ref["send_pos"])
    assert np.array_equal(u16(recv), ref["recv"])
    assert np.array_equal(u16(back), ref["send"])
    assert B.get_device_error(p.ws) == 0


def test_workspace_reuse_across_shapes():
    a = wl.small_config(T=1024, H=32, E=32, k=4, R=4, W=2, seed=31)
    b = wl.small_config(T=512, H=32, E=32, k=4, R=4, W=2, seed=32)
    ia, ib = wl.make_inputs(a), wl.make_inputs(b)
    from _parity import make_pipeline

    pa = make_pipeline(a, ia)
    ref_a, ref_b = oracle.forward(a, ia, with_rows=False), oracle.forward(b, ib, with_rows=False)
    pb = make_pipeline(b, ib)
    pb.ws = pa.ws  # one workspace serves both shapes (a's is the larger)
    for p, ref in ((pa, ref_a), (pb, ref_b), (pa, ref_a), (pa, ref_a), (pb, ref_b)):
        p.route()
        p.count()
        p.dispatch_waves()
        torch.cuda.synchronize()
        assert np.array_equal(p.counts["C"].cpu().numpy(), ref["C"])
        assert np.array_equal(p.slot_of.cpu().numpy(), ref["slot_of"])
    assert B.get_device_error(pa.ws) == 0


def test_workspace_reuse_after_a_different_layout():
    """A workspace that served one shape, then another whose look-back status
    region overlaps the first shape's rank array: stale ranks must never
    read as published status words."""
    cfgs = [wl.CONFIGS["c2"], wl.CONFIGS["c4"], wl.CONFIGS["c2"]]
    big = max(B.workspace_size(B.Shape.of(c)) for c in cfgs)
    ws = torch.zeros(big, dtype=torch.uint8, device="cuda")
    for cfg in cfgs:
        lg = wl.make_logits(cfg)
        ref = oracle.forward(cfg, {"logits": lg}, with_rows=False)
        shape = B.Shape.of(cfg)
        idx = torch.from_numpy(ref["idx"]).cuda()
        out = {k: torch.empty(v.shape, dtype=torch.int32 if v.dtype == np.int32 else torch.int64,
                              device="cuda") for k, v in ref.items()
               if k in ("c", "C", "S", "send_off", "recv_off", "recv_base")}
        B.build_send_counts(shape, idx, out, ws)
        torch.cuda.synchronize()
        assert B.get_device_error(ws) == 0
        for k in out:
            assert np.array_equal(out[k].cpu().numpy(), ref[k]), (cfg.name, k)


def test_ties_and_signed_zeros():
    cfg = wl.small_config(T=256, H=16, E=32, k=5, R=4, W=1, seed=41)
    inp = wl.make_inputs(cfg)
    rng = np.random.default_rng(0)
    lg = rng.integers(-2, 3, size=(cfg.T, cfg.E)).astype(np.float32)
    lg[rng.random(lg.shape) < 0.3] = -0.0
    lg[:16] = 0.0  # all-equal rows
    inp["logits"] = lg
    got = run_gpu(cfg, inp)
    ref = oracle.forward(cfg, inp)
    assert_full_parity(cfg, inp, got, ref)
    assert (got["idx"][:16] == np.arange(cfg.k)).all()


def test_all_tokens_to_one_expert():
    cfg = wl.small_config(T=1024, H=32, E=16, k=1, R=4, W=4, seed=42)
    inp = wl.make_inputs(cfg)
    inp["logits"] = np.zeros((cfg.T, cfg.E), np.float32)
    inp["logits"][:, 13] = 1.0
    got = run_gpu(cfg, inp)
    ref = oracle.forward(cfg, inp)
    assert_full_parity(cfg, inp, got, ref)
    assert got["stats"]["hot_over_cold"] == float("inf")
    assert got["stats"]["gini"] == pytest.approx(0.75)


def test_empty_batch():
    cfg = wl.small_config(T=0, H=16, E=8, k=2, R=2, W=2, seed=0)
    inp = wl.make_inputs(cfg)
    got = run_gpu(cfg, inp)
    assert got["status"] == 0
    assert (got["C"] == 0).all() and (got["c"] == 0).all() and (got["S"] == 0).all()
    assert (got["send_off"] == 0).all() and (got["recv_base"] == 0).all()
    st = got["stats"]
    assert st["gini"] == 0.0 and st["max_over_mean"] == 0.0 and st["hot_over_cold"] == 0.0


def test_lookback_wait_gives_up_with_timeout():
    """A tile that never publishes its status: its successors' bounded waits
    run out, the pass ends and reports MOE_ERR_TIMEOUT; the workspace then
    works again."""
    cfg = wl.small_config(T=2048, H=16, E=16, k=2, R=2, W=1, seed=51)  # 8 tiles per source
    inp = wl.make_inputs(cfg)
    ref = oracle.forward(cfg, inp, with_rows=False)
    from _parity import make_pipeline

    p = make_pipeline(cfg, inp)
    p.route()
    B.debug_set_fault(p.ws, tile=2, wait_ns=20_000_000)  # 20 ms
    p.count()
    assert B.get_device_error(p.ws) == B.MOE_ERR_TIMEOUT
    B.debug_set_fault(p.ws, tile=-1, wait_ns=0)
    p.count()
    p.dispatch_waves()
    torch.cuda.synchronize()
    assert B.get_device_error(p.ws) == 0
    assert np.array_equal(p.counts["C"].cpu().numpy(), ref["C"])
    assert np.array_equal(p.slot_of.cpu().numpy(), ref["slot_of"])


def test_device_checks_report_bad_inputs():
    cfg = wl.small_config(T=256, H=16, E=16, k=2, R=2, W=1, seed=52)
    inp = wl.make_inputs(cfg)
    from _parity import make_pipeline

    p = make_pipeline(cfg, inp)
    p.logits[5, 3] = float("nan")
    p.route()
    assert B.get_device_error(p.ws) == B.MOE_ERR_DEVICE_CHECK
    p.idx[7, 1] = cfg.E + 3  # out of range expert index
    p.count()
    assert B.get_device_error(p.ws) == B.MOE_ERR_DEVICE_CHECK
    p.slot_of.fill_(-1)
    p.dispatch(-1)
    assert B.get_device_error(p.ws) == B.MOE_ERR_DEVICE_CHECK
    p.combine()
    assert B.get_device_error(p.ws) == B.MOE_ERR_DEVICE_CHECK
    assert B.get_device_error(p.ws) == 0  # read-and-clear


def test_host_rejects_bad_calls_without_launching():
    cfg = wl.small_config(T=64, H=16, E=8, k=2, R=2, W=1)
    inp = wl.make_inputs(cfg)
    from _parity import make_pipeline

    p = make_pipeline(cfg, inp)
    with pytest.raises(B.MoEError) as e:
        B.dispatch(p.shape, p.x, p.idx, p.ws[:128], p.recv, p.slot_of)
    assert e.value.status == B.MOE_ERR_INVALID_ARG
    with pytest.raises(B.MoEError):
        B.dispatch(p.shape, p.x, p.idx, p.ws, p.recv, p.slot_of, wave=1)
    with pytest.raises(ValueError):
        B.route_topk(p.shape, p.logits.double(), p.idx, p.w)
