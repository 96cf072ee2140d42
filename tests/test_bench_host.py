"""CPU tests of bench.py's host logic: the max-over-ranks aggregation on two
gloo ranks, the reference arm's rank handling, the clock-sample parsing and
the oracle step the CPU baseline times."""
import io
import json
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from combine_moe_route_17_b300 import workloads as wl  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r timed 100 (r + 1) ms over 10 steps of 1000 tokens
        v, ms = bench.aggregate_throughput(100.0 * (rank + 1), 10, 1000, world)
        bench.barrier(world)
        q.put((rank, v, ms))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_on_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for _, v, ms in got:
        # tokens of both ranks over the slowest rank's 200 ms
        assert v == pytest.approx(2 * 10 * 1000 / 0.2)
        assert ms == pytest.approx(20.0)


def test_single_rank_aggregate():
    v, ms = bench.aggregate_throughput(50.0, 5, 100, 1)
    assert v == pytest.approx(500 / 0.05) and ms == pytest.approx(10.0)


def test_reference_arm_only_rank_zero_prints(monkeypatch):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("LOCAL_RANK", "1")
    buf = io.StringIO()
    with redirect_stdout(buf):
        rc = bench.main(["--impl", "reference", "--steps", "1", "--warmup", "0"])
    assert rc == 0 and buf.getvalue() == ""


def test_clock_summary_keeps_the_timed_windows():
    c = bench.ClockSampler("GPU-abc")
    c.sm_max = 2032.0
    c.samples = [
        (0.5, 300.0, ("hw_slowdown",), 90.0),   # before the timed window: left out
        (1.1, 1900.0, ("sw_power_cap",), 800.5),
        (1.2, 1950.0, (), 900.0),
        (1.3, 1960.0, (), 910.0),
        (3.0, 500.0, ("sw_thermal_slowdown",), 95.0),  # after it
    ]
    c.windows = [[1.0, 2.0]]
    s = c.summary()
    assert s["samples"] == 3 and s["sm_mhz"] == 1950 and s["sm_max_mhz"] == 2032
    assert s["reasons"] == ["sw_power_cap"] and s["power_w_max"] == 910.0
    c.windows = [[5.0, 6.0]]
    assert c.summary()["samples"] == 0
    c.windows = []  # nothing marked: every sample counts
    assert c.summary()["samples"] == 5


def test_oracle_step_and_algorithmic_bytes():
    cfg = wl.small_config(T=256, H=64, E=16, k=4, R=4, W=2)
    inp = wl.make_inputs(cfg)
    assert bench.oracle_step(cfg, inp, 128) > 0
    ab = bench.algorithmic_bytes(wl.CONFIGS["c2"])
    # payload dominates: (2 + 2k) T H 2 bytes
    c2 = wl.CONFIGS["c2"]
    assert abs(ab["total"] / ((2 + 2 * c2.k) * c2.T * c2.H * 2) - 1) < 0.02


def test_reference_arm_json_line(monkeypatch):
    monkeypatch.setattr(bench, "oracle_sample_tokens", lambda cfg, s, inp: cfg.R * 8)
    monkeypatch.setattr(wl, "CONFIGS", dict(wl.CONFIGS, c1=wl.CONFIGS["c1"].replace(H=64)))
    buf = io.StringIO()
    with redirect_stdout(buf):
        rc = bench.main(["--impl", "reference", "--steps", "2", "--warmup", "1",
                         "--workload", "c1"])
    assert rc == 0
    line = json.loads(buf.getvalue().strip())
    assert line["impl"] == "reference" and line["unit"] == "tokens/s" and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"


def test_partitioned_oracle_step_is_the_oracle_pass():
    """The all-cores CPU baseline runs the oracle's own functions over the R
    source partitions on threads; its outputs are the whole-batch oracle's."""
    from concurrent.futures import ThreadPoolExecutor

    import numpy as np

    import oracle

    cfg = wl.small_config(T=1200, H=40, E=32, k=4, R=4, W=1, bias="zipf", bias_param=1.0,
                          seed=13)
    inp = wl.make_inputs(cfg)
    ref = oracle.forward(cfg, inp)
    keep = {}
    with ThreadPoolExecutor(max_workers=4) as pool:
        secs = bench.oracle_step_partitions(cfg, inp, cfg.T, pool, 4, keep=keep)
    assert secs > 0
    for key in ("idx", "w", "slot_of", "src_row", "recv", "y", "C", "c", "S", "send_off",
                "recv_off", "recv_base"):
        assert np.array_equal(keep[key], ref[key]), key


def test_profiled_traffic_follows_the_kernel_source(tmp_path, monkeypatch):
    """roofline.traffic comes from a committed ncu summary only while the
    kernel source still has the hash the summary records."""
    src = tmp_path / "k.cu"
    src.write_text("__global__ void k() {}\n")
    prof = tmp_path / "ncu_scatter_c9.md"
    prof.write_text("traffic_bytes_per_launch: 123456\n"
                    f"kernel_source_sha256_16: {bench.file_sha(str(src))}\n")
    monkeypatch.setattr(bench, "PROFILES", str(tmp_path))
    assert bench.profiled_traffic("scatter_rows_kernel", "c9", str(src)) == 123456.0
    src.write_text("__global__ void k() { /* changed */ }\n")
    assert bench.profiled_traffic("scatter_rows_kernel", "c9", str(src)) is None
    assert bench.profiled_traffic("combine_kernel", "c9", str(src)) is None  # no summary


def test_staged_bytes_add_the_send_layout_both_ways():
    cfg = wl.CONFIGS["c2"]
    fused, staged = bench.algorithmic_bytes(cfg), bench.algorithmic_bytes(cfg, staged=True)
    rows = cfg.T * cfg.k * cfg.H * 2
    assert staged["dispatch"] - fused["dispatch"] == 2 * rows + cfg.T * cfg.k * 4
    assert staged["combine"] - fused["combine"] == 2 * rows
    assert staged["route"] == fused["route"] and staged["counts"] == fused["counts"]
