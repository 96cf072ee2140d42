#!/usr/bin/env python3
"""Throughput of the MoE dispatch/combine hot path on one B300 (per GPU).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl cuda|reference]
                    [--workload c2] [--staged]

A step is one pass of the hot path over one batch of the workload: top-k
routing, send counts, dispatch (W wave calls), combine and the imbalance
statistics; the scalar stand-in expert runs between dispatch and combine,
outside the timed intervals.  Each step is timed with CUDA events on the
launching stream; L2 is flushed (a 256 MB write) between steps, outside the
events.  One JSON line goes to stdout on rank 0.

--impl reference times the CPU oracle instead, on the host cores, on the same
workload (the same metric and units).  Under torchrun with N > 1 every rank
runs its own replica of the workload (no data-path collective: the ranks of
the method live inside one GPU's memory), and the value is the tokens of all
ranks over the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from combine_moe_route_17_b300 import workloads as wl  # noqa: E402

METRIC = "dispatch+combine tokens/s and achieved HBM GB/s (fraction of peak) on 1 B300"
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK_HBM_GBS = 6400.0
PROFILES = os.path.join(ROOT, "profiles")
L2_FLUSH_BYTES = 256 << 20


# ------------------------------------------------------------- helpers ----

def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=("cuda", "reference"), default="cuda")
    ap.add_argument("--workload", default="c3",
                    help="c1..c4 (c3, the largest, by default), or sweep (every sweep point)")
    ap.add_argument("--tokens", type=int, default=None, metavar="T",
                    help="run the workload at T tokens (a multiple of R) instead of its own T: "
                         "small cases for profiler captures")
    ap.add_argument("--staged", action="store_true", help="go through the send layout")
    ap.add_argument("--bulk-copy", action="store_true",
                    help="dispatch row copies with the bulk-copy engine through shared memory "
                         "(MOE_BULK_COPY) instead of registers")
    ap.add_argument("--profile-dispatch", action="store_true",
                    help="after the timed run, replay the dispatch phase alone (a graph of the "
                         "W wave calls) once between cudaProfilerStart and cudaProfilerStop, for "
                         "a profiler's range replay of the waves as they run together")
    ap.add_argument("--sequential-waves", action="store_true",
                    help="the W dispatch wave calls one after the other on one stream "
                         "(default: on W streams at once)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--fuse-route", action="store_true",
                    help="route and count in one launch (moe_route_and_count)")
    ap.add_argument("--expert-gemm", action="store_true",
                    help="time the expert-major layer with the tensor-core linear expert")
    ap.add_argument("--wave-expert", choices=("standin", "ffn"), default="standin",
                    help="the expert of --wave-scan: the scalar stand-in or the gated FFN")
    ap.add_argument("--ffn-dim", type=int, default=2048, metavar="F",
                    help="intermediate width of the gated FFN expert timed by --expert-gemm")
    ap.add_argument("--capacity", type=float, default=None, metavar="F",
                    help="time the capacity-factor variant with capacity factor F")
    ap.add_argument("--wave-scan", action="store_true",
                    help="time the wave-pipelined layer for every W dividing E and fit T(W)")
    ap.add_argument("--eager", action="store_true",
                    help="time eager launches instead of a captured CUDA graph")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="CPU work budget of the oracle baseline")
    return ap.parse_args(argv)


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def reduce_max(value: float, world: int) -> float:
    """Max of a float over the ranks of the default process group."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist

    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_throughput(local_ms: float, steps: int, tokens_per_step: int, world: int):
    """Whole-job tokens/s: the tokens of all ranks over the slowest rank's
    timed milliseconds; also that rank's ms per step."""
    ms = reduce_max(local_ms, world)
    return tokens_per_step * steps * world / (ms / 1e3), ms / steps


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def algorithmic_bytes(cfg, staged: bool = False) -> dict:
    """Bytes the fused path must move once per step: logits and gates,
    the slot ids, x once and every recv row once, every expert row once and
    y once, and the row maps.  The staged path also writes and reads the
    send layout in each direction (x -> send -> recv, then recv -> send ->
    y) and writes send_pos."""
    T, H, E, k = cfg.T, cfg.H, cfg.E, cfg.k
    route = T * E * 4 + T * k * 8
    counts = T * k * 4 + T * k * 4
    dispatch = T * H * 2 + T * k * H * 2 + T * k * 8 + T * k * 8
    combine = T * k * H * 2 + T * H * 2 + T * k * 8
    if staged:
        dispatch += 2 * T * k * H * 2 + T * k * 4
        combine += 2 * T * k * H * 2
    return {"route": route, "counts": counts, "dispatch": dispatch, "combine": combine,
            "total": route + counts + dispatch + combine}


def measured_hbm_peak():
    try:
        with open(PEAKS_FILE) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def file_sha(path: str) -> str:
    with open(path, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def profiled_traffic(kernel: str, workload: str, kernel_src: str):
    """DRAM bytes per launch of `kernel` from the committed ncu summary of the
    workload, or None if there is none or the kernel source changed since."""
    short = {"combine_kernel": "combine", "scatter_rows_kernel": "scatter"}.get(kernel, kernel)
    try:
        txt = open(os.path.join(PROFILES, f"ncu_{short}_{workload}.md")).read()
    except OSError:
        return None
    m_b = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", txt)
    m_h = re.search(r"kernel_source_sha256_16:\s*([0-9a-f]+)", txt)
    if not m_b or not m_h or m_h.group(1) != file_sha(kernel_src):
        return None
    return float(m_b.group(1))


class ClockSampler:
    """SM clock, power and clock-event (throttle) reasons of one GPU, polled
    through NVML every ~2 ms on a thread from before the warm-up to the end of
    the timed loops.  summary() keeps the samples taken inside the timed
    windows (mark() opens and closes one), so even a short timed region
    carries its own clock record; nvidia-smi at 20 ms is the fallback when
    NVML cannot be loaded."""

    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
    PERIOD_S = 0.002

    def __init__(self, uuid: str | None, index: int = 0):
        self.uuid = (uuid or "").lower().replace("gpu-", "")
        self.index = index
        self.samples = []  # (perf_counter, sm_mhz, reasons tuple, power_w)
        self.windows = []
        self.sm_max = None
        self.source = None
        self._stop = threading.Event()
        self._t = None
        self._proc = None

    # -- NVML ------------------------------------------------------------
    def _nvml_handle(self):
        import pynvml as nv

        nv.nvmlInit()
        for i in range(nv.nvmlDeviceGetCount()):
            h = nv.nvmlDeviceGetHandleByIndex(i)
            u = nv.nvmlDeviceGetUUID(h)
            u = (u.decode() if isinstance(u, bytes) else u).lower().replace("gpu-", "")
            if self.uuid and u == self.uuid:
                return nv, h
        if nv.nvmlDeviceGetCount() == 1 or not self.uuid:
            return nv, nv.nvmlDeviceGetHandleByIndex(self.index)
        raise RuntimeError("GPU not found by UUID")

    def _poll_nvml(self, nv, h):
        bits = (nv.nvmlClocksEventReasonHwSlowdown, nv.nvmlClocksEventReasonHwThermalSlowdown,
                nv.nvmlClocksEventReasonSwThermalSlowdown, nv.nvmlClocksEventReasonSwPowerCap)
        while not self._stop.is_set():
            t = time.perf_counter()
            try:
                sm = float(nv.nvmlDeviceGetClockInfo(h, nv.NVML_CLOCK_SM))
                r = int(nv.nvmlDeviceGetCurrentClocksEventReasons(h))
                pw = nv.nvmlDeviceGetPowerUsage(h) / 1000.0
            except Exception:  # noqa: BLE001 -- a failed query just skips a sample
                time.sleep(self.PERIOD_S)
                continue
            self.samples.append((t, sm, tuple(n for n, b in zip(self.REASONS, bits) if r & b),
                                 pw))
            time.sleep(self.PERIOD_S)

    # -- nvidia-smi fallback ---------------------------------------------
    def _poll_smi(self):
        q = ("uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
             "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
             "clocks_event_reasons.sw_power_cap")
        self._proc = subprocess.Popen(
            ["nvidia-smi", f"--query-gpu={q}", "--format=csv,noheader,nounits", "-lms=20"],
            stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        for line in self._proc.stdout:
            r = [x.strip() for x in line.split(",")]
            if len(r) != 8 or (self.uuid and self.uuid not in r[0].lower()):
                continue
            try:
                sm, smax, pw = float(r[1]), float(r[2]), float(r[3])
            except ValueError:
                continue
            self.sm_max = smax
            self.samples.append((time.perf_counter(), sm,
                                 tuple(n for i, n in enumerate(self.REASONS)
                                       if r[4 + i] == "Active"), pw))

    def __enter__(self):
        try:
            nv, h = self._nvml_handle()
            self.sm_max = float(nv.nvmlDeviceGetMaxClockInfo(h, nv.NVML_CLOCK_SM))
            self.source = "nvml, every 2 ms"
            self._t = threading.Thread(target=self._poll_nvml, args=(nv, h), daemon=True)
        except Exception as exc:  # noqa: BLE001 -- no NVML: nvidia-smi
            self.source = f"nvidia-smi, every 20 ms (NVML: {type(exc).__name__}: {exc})"[:200]
            self._t = threading.Thread(target=self._poll_smi, daemon=True)
        self._t.start()
        t0 = time.perf_counter()
        while not self.samples and time.perf_counter() - t0 < 2.0:
            time.sleep(0.001)  # the first sample lands before the timed region
        return self

    def mark(self, start: bool):
        if start:
            self.windows.append([time.perf_counter(), None])
        elif self.windows and self.windows[-1][1] is None:
            self.windows[-1][1] = time.perf_counter()

    def __exit__(self, *exc):
        self._stop.set()
        if self._proc is not None:
            self._proc.terminate()
            try:
                self._proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self._proc.kill()
        if self._t is not None:
            self._t.join(timeout=2)

    def summary(self):
        inside = [x for x in self.samples
                  if not self.windows or any(a <= x[0] <= (b if b is not None else float("inf"))
                                             for a, b in self.windows)]
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": self.sm_max, "samples": 0,
                    "reasons": ["no samples inside the timed windows"], "source": self.source,
                    "samples_whole_run": len(self.samples)}
        sm = [x[1] for x in inside]
        return {"sm_mhz": statistics.median(sm), "sm_min_mhz": min(sm),
                "sm_max_mhz": self.sm_max,
                "reasons": sorted({r for x in inside for r in x[2]}),
                "samples": len(inside), "power_w_max": max(x[3] for x in inside),
                "source": self.source,
                "window_s": sum((b or 0) - a for a, b in self.windows)}


# ------------------------------------------------------------ CUDA arm ----

def run_cuda(args, cfg, rank, world, local):
    import torch

    from combine_moe_route_17_b300 import MoEPipeline
    from combine_moe_route_17_b300 import binding as B

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    inp = wl.make_inputs(cfg)
    p = MoEPipeline(cfg, device=dev, staged=args.staged, fuse_route=args.fuse_route,
                    concurrent_waves=not args.sequential_waves, bulk_copy=args.bulk_copy)
    p.load_inputs(torch.from_numpy(inp["logits"]), torch.from_numpy(inp["x"].view(np.int16)),
                  torch.from_numpy(inp["scale"]))
    stream = torch.cuda.current_stream(dev)
    side = torch.cuda.Stream(dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    W = cfg.W
    waves = [-1] if W == 1 else list(range(W))
    # concurrent waves run on W streams at once, so the dispatch phase is
    # timed as one segment; waves in order are timed one by one
    concurrent = W > 1 and p.concurrent_waves and not args.staged
    if concurrent:
        segments = [lambda st: p.dispatch_waves(st)]
    else:
        segments = [lambda st, w=w: p.dispatch(w, st) for w in waves]
    nw = len(segments)
    # event slots: 0 start, 1 after dispatch, 2 before combine, 3 end,
    # 4.. per-wave pairs, then combine pair, route end, counts end, stats pair
    I_CMB, I_RT, I_CT, I_ST = 4 + 2 * nw, 6 + 2 * nw, 7 + 2 * nw, 8 + 2 * nw
    n_ev = 10 + 2 * nw
    # inside the timed intervals: route + counts (one launch when fused), the
    # W dispatch launches, combine, stats; the stand-in expert runs between
    # the two intervals and is not counted
    launches_per_step = (3 if p.fuse_route else 4) + len(waves)
    if args.staged:  # an exchange per wave, and the reverse exchange before the gather
        launches_per_step += len(waves) + 1

    def one_step(ev, st, overlap_stats, per_kernel):
        """One step on stream `st`.  With overlap_stats the statistics run on
        a second stream, forked after the counts and joined before the end
        of the dispatch phase, so they overlap the dispatch waves.  Without
        per_kernel, events mark only the phase boundaries, so consecutive
        kernels keep their programmatic (early-launch) dependencies."""
        ev[0].record(st)
        if p.fuse_route:
            p.route_count(st)
            if per_kernel:
                ev[I_RT].record(st)
                ev[I_CT].record(st)
        else:
            p.route(st)
            if per_kernel:
                ev[I_RT].record(st)
            p.count(st)
            if per_kernel:
                ev[I_CT].record(st)
        if overlap_stats:
            side.wait_stream(st)
            if per_kernel:
                ev[I_ST].record(side)
            p.imbalance(side)
            if per_kernel:
                ev[I_ST + 1].record(side)
        for i, seg in enumerate(segments):
            if per_kernel:
                ev[4 + 2 * i].record(st)
            seg(st)
            if per_kernel:
                ev[5 + 2 * i].record(st)
        if overlap_stats:
            st.wait_stream(side)
        ev[1].record(st)
        p.expert(st)  # harness, outside the timed intervals
        ev[2].record(st)
        if per_kernel:
            ev[I_CMB].record(st)
        p.combine(st)
        if per_kernel:
            ev[I_CMB + 1].record(st)
        if not overlap_stats:
            if per_kernel:
                ev[I_ST].record(st)
            p.imbalance(st)
            if per_kernel:
                ev[I_ST + 1].record(st)
        ev[3].record(st)

    def new_events(external):
        return [torch.cuda.Event(enable_timing=True, external=external) for _ in range(n_ev)]

    def read(ev, per_kernel):
        r = {"step": ev[0].elapsed_time(ev[1]) + ev[2].elapsed_time(ev[3])}
        if per_kernel:
            r.update({"route": ev[0].elapsed_time(ev[I_RT]),
                      "counts": ev[I_RT].elapsed_time(ev[I_CT]),
                      "waves": [ev[4 + 2 * i].elapsed_time(ev[5 + 2 * i]) for i in range(nw)],
                      "combine": ev[I_CMB].elapsed_time(ev[I_CMB + 1]),
                      "stats": ev[I_ST].elapsed_time(ev[I_ST + 1])})
        return r

    props = torch.cuda.get_device_properties(dev)
    # the sampler polls from before the warm-up to the end of the timed loops
    with ClockSampler(str(getattr(props, "uuid", "") or ""), local) as clk:
        for _ in range(args.warmup):
            flush.zero_()
            one_step(new_events(False), stream, False, True)
        torch.cuda.synchronize(dev)
        p.check_device_error()

        # Graph mode: the step (L2 flush first, outside the timed events) is
        # captured as a CUDA graph and replayed; the timing events are record
        # nodes inside it, read back after each replay.  The headline graph has
        # events at the phase boundaries only; a second graph with events around
        # every kernel gives the per-kernel times.
        graphs = None
        if not args.eager:
            try:
                graphs = {}
                for per_kernel in (False, True):
                    gev = new_events(True)
                    graph = torch.cuda.CUDAGraph()
                    cap = torch.cuda.Stream(dev)
                    cap.wait_stream(stream)
                    with torch.cuda.graph(graph, stream=cap):
                        flush.zero_()
                        one_step(gev, cap, True, per_kernel)
                    torch.cuda.synchronize(dev)
                    for _ in range(max(3, min(args.warmup, 20))):
                        graph.replay()
                        torch.cuda.synchronize(dev)
                        read(gev, per_kernel)
                    graphs[per_kernel] = (graph, gev)
            except RuntimeError as exc:  # no event record nodes: eager timing
                print(f"graph capture unavailable ({exc}); timing eager launches", file=sys.stderr)
                graphs = None
                torch.cuda.synchronize(dev)
        p.check_device_error()

        times, ktimes = [], []
        barrier(world)
        torch.cuda.synchronize(dev)
        clk.mark(True)
        t0 = time.perf_counter()
        if graphs is not None:
            graph, gev = graphs[False]
            for _ in range(args.steps):
                graph.replay()
                torch.cuda.synchronize(dev)
                times.append(read(gev, False))
            wall = time.perf_counter() - t0
            graph, gev = graphs[True]
            for _ in range(max(3, min(args.steps, 200))):
                graph.replay()
                torch.cuda.synchronize(dev)
                ktimes.append(read(gev, True))
        else:
            events = [new_events(False) for _ in range(args.steps)]
            for s_ in range(args.steps):
                flush.zero_()
                one_step(events[s_], stream, False, True)
            torch.cuda.synchronize(dev)
            wall = time.perf_counter() - t0
            times = ktimes = [read(e, True) for e in events]
        clk.mark(False)
    barrier(world)
    p.check_device_error()

    step_ms = [t["step"] for t in times]
    disp_ms = [sum(t["waves"]) for t in ktimes]
    comb_ms = [t["combine"] for t in ktimes]
    route_ms = [t["route"] for t in ktimes]
    count_ms = [t["counts"] for t in ktimes]
    stats_ms = [t["stats"] for t in ktimes]
    wave_ms = np.mean(np.array([t["waves"] for t in ktimes]), axis=0).tolist()
    value, ms_per_step = aggregate_throughput(float(np.sum(step_ms)), args.steps, cfg.T, world)
    ab = algorithmic_bytes(cfg, staged=args.staged)
    gbs = ab["total"] / (ms_per_step / 1e3) / 1e9
    peak, peak_kind = measured_hbm_peak()

    # dominant kernel: the larger share of the step, dispatch (W launches) or
    # combine (one launch); achieved = its algorithmic bytes per launch over
    # its mean launch duration
    d_ms, c_ms = float(np.mean(disp_ms)), float(np.mean(comb_ms))
    src_dir = os.path.join(ROOT, "combine_moe_route_17_b300", "csrc")
    if c_ms >= d_ms:
        dom = {"kernel": "exchange_kernel+combine_kernel" if args.staged else "combine_kernel",
               "launches": 2 if args.staged else 1, "ms": c_ms, "bytes": ab["combine"],
               "src": os.path.join(src_dir, "combine.cu")}
    elif args.staged:
        # per wave: the scatter into the send layout and the exchange to recv
        dom = {"kernel": "scatter_rows_kernel+exchange_kernel", "launches": 2 * len(waves),
               "ms": d_ms, "bytes": ab["dispatch"], "src": os.path.join(src_dir, "dispatch.cu")}
    else:
        dom = {"kernel": "scatter_rows_kernel", "launches": len(waves), "ms": d_ms,
               "bytes": ab["dispatch"], "src": os.path.join(src_dir, "dispatch.cu")}
    # with concurrent waves the W launches overlap: launch_ms is the dispatch
    # phase over W, so bytes_per_launch / launch_ms is the phase's own rate
    achieved = dom["bytes"] / (dom["ms"] / 1e3) / 1e9
    traffic = (profiled_traffic(dom["kernel"], args.workload, dom["src"]) if args.tokens is None
               else None)

    result = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32",
        "dtype_note": "fp32 routing and gate-weighted accumulation, int32 counts and "
                      "offsets; the hidden-state rows are bf16 and move as bit copies",
        "data": "synthetic (seeded; routing logits with the workload's bias family)",
        "config": {"workload": cfg.name, "T": cfg.T, "H": cfg.H, "E": cfg.E, "k": cfg.k,
                   "R": cfg.R, "W": cfg.W, "n_groups": cfg.n_groups, "bias": cfg.bias,
                   "bias_param": cfg.bias_param, "seed": cfg.seed,
                   "mode": "staged" if args.staged else "fused",
                   "row_copy": "bulk-copy engine via shared memory" if args.bulk_copy
                   else "registers, 16-byte vectors",
                   "waves": ("concurrent (one stream per wave call)" if concurrent
                             else "in order on one stream" if W > 1 else "one call"),
                   "route": "one launch with the counts" if p.fuse_route
                   else "separate route and count launches",
                   "l2": f"flushed between steps ({L2_FLUSH_BYTES >> 20} MB write)",
                   "launch": "cuda graph, programmatic dependent launches (stats on a "
                   "second stream, overlapping dispatch)" if graphs is not None else "eager",
                   "parallelism": f"replicas{world}" if world > 1 else "single"},
        "gbs": gbs, "frac_of_measured_hbm": gbs / peak,
        "frac_of_nominal_8tbs": gbs / 8000.0,
        "algorithmic_bytes_per_step": ab["total"],
        "per_kernel_ms": {**({"route_and_count": float(np.mean(route_ms))} if p.fuse_route
                             else {"route": float(np.mean(route_ms)),
                                   "counts": float(np.mean(count_ms))}),
                          "dispatch_all_waves": d_ms,
                          "dispatch_per_wave": None if concurrent else wave_ms,
                          "combine": c_ms, "stats": float(np.mean(stats_ms)),
                          "step_median": float(np.median(step_ms)),
                          "step_with_kernel_events": float(np.mean([t["step"] for t in ktimes])),
                          "note": "kernel times from a second graph pass with events around "
                                  "every kernel"},
        "roofline": {"bound": "hbm", "kernel": dom["kernel"], "launches_per_step":
                     dom["launches"], "launches_overlap": bool(concurrent and
                                                               dom["kernel"].startswith("scatter")),
                     "bytes_per_launch": dom["bytes"] / dom["launches"],
                     "launch_ms": dom["ms"] / dom["launches"], "achieved": achieved,
                     "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic,
                     # the DRAM bytes the launch really moves (the profile's
                     # traffic) over its time: how close it runs to the peak
                     # for the bytes it must move
                     "traffic_achieved": (traffic / (dom["ms"] / dom["launches"] / 1e3) / 1e9
                                          if traffic else None),
                     "traffic_frac": (traffic / (dom["ms"] / dom["launches"] / 1e3) / 1e9 / peak
                                      if traffic else None)},
        "gpu_launches": launches_per_step * args.steps,
        "gpu_launches_note": f"{launches_per_step} per step inside the timed intervals; "
                             "the stand-in expert (1 per step) runs between them",
        "wall_s": wall,
        "clocks": clk.summary(),
    }
    if args.profile_dispatch:
        # route and counts first, outside the range; then the dispatch phase alone
        p.route_count(stream)
        cap = torch.cuda.Stream(dev)
        cap.wait_stream(stream)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cap):
            for seg in segments:
                seg(cap)
        flush.zero_()
        torch.cuda.synchronize(dev)
        torch.cuda.profiler.start()
        g.replay()
        torch.cuda.synchronize(dev)
        torch.cuda.profiler.stop()
        p.check_device_error()
        result["profile_dispatch"] = "one replay of the dispatch phase inside a profiler range"
    if not args.no_e2e:
        result["e2e"] = run_e2e(args, cfg, p, inp, dev, world)
    return result


def run_e2e(args, cfg, p, inp, dev, world):
    """Same metric through the same C-ABI calls with the inputs in pinned host
    memory: the H2D copies of logits and x and the D2H read of y and the
    statistics are inside the timed interval of every step.  Reported twice:
    step after step (sequential_value, stand-in expert excluded), and
    double-buffered through HostBatchRunner (value)."""
    import torch

    stream = torch.cuda.current_stream(dev)
    h_logits = torch.from_numpy(inp["logits"]).pin_memory()
    h_x = torch.from_numpy(inp["x"].view(np.int16)).pin_memory()
    h_y = torch.empty((cfg.T, cfg.H), dtype=torch.int16).pin_memory()
    h_stats = torch.empty(8, dtype=torch.float64).pin_memory()
    steps = max(3, min(args.steps, 100))

    def one(ev0, ev1, ev2, ev3):
        ev0.record(stream)
        p.logits.copy_(h_logits, non_blocking=True)
        p.x.view(torch.int16).copy_(h_x, non_blocking=True)
        p.forward_to_experts()
        ev1.record(stream)
        p.expert()
        ev2.record(stream)
        p.combine()
        p.imbalance()
        h_y.copy_(p.y.view(torch.int16), non_blocking=True)
        h_stats.copy_(p.stats, non_blocking=True)
        ev3.record(stream)

    for _ in range(3):
        one(*[torch.cuda.Event(enable_timing=True) for _ in range(4)])
    torch.cuda.synchronize(dev)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps)]
    barrier(world)
    for e in evs:
        one(*e)
    torch.cuda.synchronize(dev)
    ms_seq = sum(e[0].elapsed_time(e[1]) + e[2].elapsed_time(e[3]) for e in evs)
    ms_seq = reduce_max(ms_seq, world)

    # Double-buffered (HostBatchRunner): step i+1's copy-in and step i-1's
    # read-back overlap step i's compute.  Timed from the first copy-in to
    # the last read-back; the stand-in expert runs inside that interval.
    from combine_moe_route_17_b300 import HostBatchRunner

    runner = HostBatchRunner(cfg, device=dev, staged=args.staged, fuse_route=args.fuse_route)
    runner.load_scale(inp["scale"])
    h_ys = [torch.empty((cfg.T, cfg.H), dtype=torch.int16).pin_memory() for _ in range(2)]
    h_sts = [torch.empty(8, dtype=torch.float64).pin_memory() for _ in range(2)]
    for i in range(4):
        runner.step(i, h_logits, h_x, h_ys[i % 2], h_sts[i % 2])
    torch.cuda.synchronize(dev)
    runner.check_device_error()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    t0.record(runner.s_in)
    for i in range(steps):
        runner.step(i, h_logits, h_x, h_ys[i % 2], h_sts[i % 2])
    runner.join(stream)
    t1.record(stream)
    torch.cuda.synchronize(dev)
    runner.check_device_error()
    if not np.array_equal(h_ys[(steps - 1) % 2].numpy(), h_y.numpy()):
        raise RuntimeError("double-buffered steps disagree with the sequential step")
    ms = reduce_max(t0.elapsed_time(t1), world)

    # The link's own rate for the same copies: the step's copy-in and
    # read-back alone, both directions at once, same buffers and streams.
    def copies_only():
        with torch.cuda.stream(runner.s_in):
            runner.pipes[0].logits.copy_(h_logits, non_blocking=True)
            runner.pipes[0].x.view(torch.int16).copy_(h_x, non_blocking=True)
        with torch.cuda.stream(runner.s_out):
            h_ys[1].copy_(runner.pipes[1].y.view(torch.int16), non_blocking=True)
            h_sts[1].copy_(runner.pipes[1].stats, non_blocking=True)
        runner.join(stream)

    copies_only()
    torch.cuda.synchronize(dev)
    l0, l1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    l0.record(stream)
    for _ in range(steps):
        runner.s_in.wait_stream(stream)
        runner.s_out.wait_stream(stream)
        copies_only()
    l1.record(stream)
    torch.cuda.synchronize(dev)
    link_ms = l0.elapsed_time(l1) / steps
    del runner
    bi = cfg.T * cfg.E * 4 + cfg.T * cfg.H * 2
    bo = cfg.T * cfg.H * 2 + 48
    return {"value": cfg.T * steps * world / (ms / 1e3), "unit": "tokens/s",
            "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo, "steps": steps,
            "mode": "double-buffered: copies of neighbouring steps overlap the compute "
                    "(stand-in expert included)",
            "sequential_value": cfg.T * steps * world / (ms_seq / 1e3),
            "link": {"copies_only_ms_per_step": link_ms,
                     "gbs": (bi + bo) / (link_ms / 1e3) / 1e9,
                     "frac": link_ms / (ms / steps),
                     "note": "the same H2D and D2H copies alone, both directions at once"}}


# ---------------------------------------------------------------- sweep ----

def _finite(v):
    """JSON has no infinity: non-finite figures (hot/cold with an idle
    expert) become null."""
    return float(v) if np.isfinite(v) else None


def _spread(vals):
    """mean/std/min/max over the finite values, and how many were not."""
    a = np.asarray(vals, dtype=np.float64)
    f = a[np.isfinite(a)]
    out = {"non_finite": int(a.size - f.size)}
    if f.size:
        out.update(mean=float(f.mean()), std=float(f.std()), min=float(f.min()),
                   max=float(f.max()))
    return out


def run_sweep(args):
    """The sweep workload: T x Dirichlet alpha x W on E=128, k=8, R=64,
    H=4096.  Every point is one captured step (programmatic launches, events
    at the phase boundaries, L2 flushed first), replayed args.steps times;
    x is drawn once per T (it does not depend on alpha or W).  The routing
    statistics are also taken over seeds 0..9 per (T, alpha) for their
    spread (routing, counts and statistics only)."""
    import torch

    from combine_moe_route_17_b300 import MoEPipeline

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    peak, peak_kind = measured_hbm_peak()
    steps = max(3, min(args.steps, 20))  # timed replays per point
    points = []
    by_T = {}
    for c in wl.SWEEP:
        by_T.setdefault(c.T, []).append(c)
    for T in sorted(by_T):
        cfgs = by_T[T]
        base = cfgs[0]
        x = torch.from_numpy(wl.make_x(base).view(np.int16))
        p = MoEPipeline(base.replace(W=1), device=dev)
        p.x.view(torch.int16).copy_(x)
        del x
        for alpha in sorted({c.bias_param for c in cfgs}):
            acfg = base.replace(bias_param=alpha)
            p.logits.copy_(torch.from_numpy(wl.make_logits(acfg)))
            p.scale.copy_(torch.from_numpy(wl.make_scales(acfg)))
            spread = {"max_over_mean": [], "gini": [], "hot_over_cold": [],
                      "gini_after_greedy_placement": [], "alpha_fit": []}
            for seed in range(10):
                p.logits.copy_(torch.from_numpy(wl.make_logits(acfg, seed=seed)))
                p.route_count()
                p.imbalance()
                st = p.stats_dict()
                for key in ("max_over_mean", "gini", "hot_over_cold"):
                    spread[key].append(st[key])
                spread["gini_after_greedy_placement"].append(p.place_greedy()["gini_after"])
                spread["alpha_fit"].append(p.dirichlet_alpha())
            p.logits.copy_(torch.from_numpy(wl.make_logits(acfg)))
            for W in sorted({c.W for c in cfgs if c.bias_param == alpha}):
                cfg = acfg.replace(W=W, name=f"sweep_T{T}_a{alpha:g}_W{W}")
                p.set_waves(W)
                ev = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(4)]
                g = torch.cuda.CUDAGraph()
                cap = torch.cuda.Stream(dev)
                cap.wait_stream(stream)
                with torch.cuda.graph(g, stream=cap):
                    flush.zero_()
                    ev[0].record(cap)
                    p.route_count(cap)
                    p.dispatch_waves(cap)  # the W wave calls at once, one stream each
                    ev[1].record(cap)
                    p.expert(cap)
                    ev[2].record(cap)
                    p.combine(cap)
                    p.imbalance(cap)
                    ev[3].record(cap)
                torch.cuda.synchronize(dev)
                ms = []
                for r in range(steps + 3):
                    g.replay()
                    torch.cuda.synchronize(dev)
                    if r >= 3:
                        ms.append(ev[0].elapsed_time(ev[1]) + ev[2].elapsed_time(ev[3]))
                p.check_device_error()
                st = p.stats_dict()
                placed = p.place_greedy()
                alpha_fit = p.dirichlet_alpha()
                ab = algorithmic_bytes(cfg)
                m = float(np.mean(ms))
                gbs = ab["total"] / (m / 1e3) / 1e9
                points.append({
                    "T": T, "alpha": alpha, "W": W, "ms_per_step": m, "tokens_per_s": T / (m / 1e3),
                    "gbs": gbs, "frac_of_nominal_8tbs": gbs / 8000.0, "frac_of_measured_hbm": gbs / peak,
                    "max_load": st["max_load"], "min_load": st["min_load"],
                    "max_over_mean": st["max_over_mean"],
                    "hot_over_cold": _finite(st["hot_over_cold"]),  # null: an expert got 0
                    "gini": st["gini"],
                    "gini_after_greedy_placement": placed["gini_after"],
                    "max_rank_load_before": placed["max_rank_load_before"],
                    "max_rank_load_after": placed["max_rank_load_after"],
                    "alpha_fit": _finite(alpha_fit),
                    "seeds_0_9": {k: _spread(v) for k, v in spread.items()}})
                del g
        del p
        torch.cuda.empty_cache()
    return {"metric": METRIC, "workload": "sweep", "unit": "tokens/s", "steps": steps,
            "higher_is_better": True, "dtype": "f32", "data": "synthetic (seeded Dirichlet log-bias)",
            "config": {"H": 4096, "E": 128, "k": 8, "R": 64, "T": sorted(by_T),
                       "alpha": [0.1, 1.0, 10.0], "W": [1, 4, 8, 16],
                       "l2": f"flushed between steps ({L2_FLUSH_BYTES >> 20} MB write)",
                       "launch": "cuda graph, programmatic dependent launches; the W dispatch "
                                 "wave calls at once on W streams"},
            "peak": peak, "peak_kind": peak_kind, "points": points}


# ------------------------------------------------------------- capacity ----

def run_capacity(args, cfg):
    """The capacity-factor variant (MoE survey, section 1.1, eq. 3): route,
    counts, capacity dispatch into the fixed [E][EC][H] buffer and the
    capacity combine, timed as a captured graph step like the dropless path
    (stand-in expert between, outside the timed events; L2 flushed first).
    Algorithmic bytes: logits, gates and slot ids, x once, every capacity row
    written once (kept rows and zero padding), every kept row read once by
    the combine, y once and the maps."""
    import torch

    from combine_moe_route_17_b300 import MoEPipeline

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    inp = wl.make_inputs(cfg)
    p = MoEPipeline(cfg, device=dev, capacity_factor=args.capacity)
    p.load_inputs(torch.from_numpy(inp["logits"]), torch.from_numpy(inp["x"].view(np.int16)),
                  torch.from_numpy(inp["scale"]))
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    base = torch.cuda.current_stream(dev)
    cap, side = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    for _ in range(max(3, args.warmup)):
        p.step_capacity()
    torch.cuda.synchronize(dev)
    p.check_device_error()
    ev = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(4)]
    g = torch.cuda.CUDAGraph()
    cap.wait_stream(base)
    with torch.cuda.graph(g, stream=cap):
        flush.zero_()
        ev[0].record(cap)
        p.route_count(cap)
        side.wait_stream(cap)
        p.imbalance(side)
        p.dispatch_capacity(cap)
        cap.wait_stream(side)
        ev[1].record(cap)
        p.expert_capacity(cap)
        ev[2].record(cap)
        p.combine_capacity(cap)
        ev[3].record(cap)
    torch.cuda.synchronize(dev)
    ms = []
    for r in range(args.steps + 3):
        g.replay()
        torch.cuda.synchronize(dev)
        if r >= 3:
            ms.append(ev[0].elapsed_time(ev[1]) + ev[2].elapsed_time(ev[3]))
    p.check_device_error()
    T, H, E, k, EC = cfg.T, cfg.H, cfg.E, cfg.k, p.capacity
    dropped = int(p.dropped.sum().item())
    kept = T * k - dropped
    ab = (T * E * 4 + T * k * 8 + T * k * 8 + T * H * 2 + E * EC * H * 2 + T * k * 12
          + kept * H * 2 + T * H * 2 + T * k * 8)
    m = float(np.mean(ms))
    peak, peak_kind = measured_hbm_peak()
    gbs = ab / (m / 1e3) / 1e9
    return {"metric": METRIC + " -- capacity-factor variant", "value": T / (m / 1e3),
            "unit": "tokens/s", "n_gpus": 1, "steps": args.steps, "ms_per_step": m,
            "higher_is_better": True, "dtype": "f32",
            "data": "synthetic (seeded; routing logits with the workload's bias family)",
            "config": {"workload": cfg.name, "capacity_factor": args.capacity, "capacity": EC,
                       "l2": f"flushed between steps ({L2_FLUSH_BYTES >> 20} MB write)",
                       "launch": "cuda graph, programmatic dependent launches"},
            "dropped_slots": dropped, "dropped_fraction": dropped / (T * k),
            "padding_rows": E * EC - kept, "algorithmic_bytes_per_step": ab, "gbs": gbs,
            "frac_of_measured_hbm": gbs / peak, "frac_of_nominal_8tbs": gbs / 8000.0,
            "peak_kind": peak_kind}


# ---------------------------------------------------------- expert GEMM ----

def run_expert_gemm(args, cfg):
    """The expert-major layer with the tensor-core linear expert (a bf16
    [H][H] weight per expert, seeded on the device): route, counts, the W
    expert-major dispatch waves, moe_expert_gemm and the combine, timed as
    one captured graph (L2 flushed first); the GEMM alone is timed the same
    way, and so is the gated FFN expert (moe_expert_ffn) and its layer.  The
    GEMM's rate is 2*T*k*H*H flops over its time (the FFN's 6*T*k*H*F):
    as a burst of replays against the measured burst bf16 peak, and replayed
    back to back under the power cap against the measured sustained peak."""
    import torch

    from combine_moe_route_17_b300 import MoEPipeline
    from combine_moe_route_17_b300 import binding as B

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    inp = wl.make_inputs(cfg)
    p = MoEPipeline(cfg, device=dev, expert_major=True)
    p.load_inputs(torch.from_numpy(inp["logits"]), torch.from_numpy(inp["x"].view(np.int16)),
                  torch.from_numpy(inp["scale"]))
    gen = torch.Generator(device=dev)
    gen.manual_seed(cfg.seed + 17)
    Wt = (torch.randn((cfg.E, cfg.H, cfg.H), generator=gen, device=dev, dtype=torch.float32)
          / float(np.sqrt(cfg.H))).to(torch.bfloat16)
    out = torch.empty_like(p.recv)
    F = args.ffn_dim
    w13 = (torch.randn((cfg.E, 2 * F, cfg.H), generator=gen, device=dev, dtype=torch.float32)
           / float(np.sqrt(cfg.H))).to(torch.bfloat16)
    w2 = (torch.randn((cfg.E, cfg.H, F), generator=gen, device=dev, dtype=torch.float32)
          / float(np.sqrt(F))).to(torch.bfloat16)
    hidden = torch.empty((cfg.T * cfg.k, F), dtype=torch.bfloat16, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    base = torch.cuda.current_stream(dev)
    cap = torch.cuda.Stream(dev)
    steps = max(3, min(args.steps, 20))

    def gemm(st):
        B.expert_gemm(p.shape, p.recv, Wt, p.counts["c"], out, p.ws, st)

    def ffn(st):
        B.expert_ffn(p.shape, p.recv, w13, w2, p.counts["c"], hidden, out, p.ws, st)

    def ffn_layer(st):
        p.route_count(st)
        p.dispatch_waves(st)
        ffn(st)
        B.combine(p.shape, out, p.slot_of, p.w, p.y, p.ws, stream=st)

    def layer(st):
        p.route_count(st)
        p.dispatch_waves(st)
        gemm(st)
        B.combine(p.shape, out, p.slot_of, p.w, p.y, p.ws, stream=st)

    layer(base)
    torch.cuda.synchronize(dev)
    p.check_device_error()

    def timed(body):
        ev = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(2)]
        g = torch.cuda.CUDAGraph()
        cap.wait_stream(base)
        with torch.cuda.graph(g, stream=cap):
            flush.zero_()
            ev[0].record(cap)
            body(cap)
            ev[1].record(cap)
        torch.cuda.synchronize(dev)
        # burst: `steps` replays right after 3 warm-up replays; sustained:
        # replays back to back for 1.5 s more, the mean of the last second
        # (the 1.1 kW power cap has settled by then)
        burst, tail = [], []
        for r in range(steps + 3):
            g.replay()
            torch.cuda.synchronize(dev)
            if r >= 3:
                burst.append(ev[0].elapsed_time(ev[1]))
        t_start = time.perf_counter()
        while time.perf_counter() - t_start < 1.5:
            g.replay()
            torch.cuda.synchronize(dev)
            if time.perf_counter() - t_start > 0.5:
                tail.append(ev[0].elapsed_time(ev[1]))
        p.check_device_error()
        return float(np.mean(burst)), float(np.mean(tail))

    props = torch.cuda.get_device_properties(dev)
    with ClockSampler(str(getattr(props, "uuid", "") or "")) as clk:
        gemm_ms, gemm_ms_sus = timed(gemm)
        layer_ms, _ = timed(layer)
    with ClockSampler(str(getattr(props, "uuid", "") or "")) as clk_ffn:
        ffn_layer(base)
        torch.cuda.synchronize(dev)
        ffn_ms, ffn_ms_sus = timed(ffn)
        ffn_layer_ms, _ = timed(ffn_layer)
    flops = 2.0 * cfg.T * cfg.k * cfg.H * cfg.H
    ffn_flops = 6.0 * cfg.T * cfg.k * cfg.H * F
    tflops = flops / (gemm_ms / 1e3) / 1e12
    tflops_sus = flops / (gemm_ms_sus / 1e3) / 1e12
    ffn_tflops = ffn_flops / (ffn_ms / 1e3) / 1e12
    ffn_tflops_sus = ffn_flops / (ffn_ms_sus / 1e3) / 1e12
    try:
        peaks = json.load(open(PEAKS_FILE))
        peak, peak_kind = float(peaks["bf16_tflops"]), "measured (burst)"
        peak_sus = float(peaks["bf16_tflops_sustained"])
    except (OSError, KeyError, ValueError):
        peak, peak_kind, peak_sus = 1800.0, "fallback", 1400.0
    return {"metric": "expert-major MoE layer with the tcgen05 linear expert",
            "workload": cfg.name, "unit": "ms", "steps": steps,
            "config": {"T": cfg.T, "H": cfg.H, "E": cfg.E, "k": cfg.k, "R": cfg.R, "W": cfg.W,
                       "expert": "linear, bf16 [H][H] per expert, fp32 accumulation",
                       "l2": f"flushed between steps ({L2_FLUSH_BYTES >> 20} MB write)",
                       "launch": "cuda graph, programmatic dependent launches"},
            "gemm_ms": gemm_ms, "gemm_tflops": tflops,
            "roofline": {"bound": "tensor", "achieved": tflops, "peak": peak,
                         "peak_kind": peak_kind, "unit": "TFLOP/s", "frac": tflops / peak},
            "sustained": {"gemm_ms": gemm_ms_sus, "gemm_tflops": tflops_sus,
                          "peak": peak_sus, "frac": tflops_sus / peak_sus,
                          "ffn_ms": ffn_ms_sus, "ffn_tflops": ffn_tflops_sus,
                          "ffn_frac": ffn_tflops_sus / peak_sus,
                          "note": "replays back to back for 1.5 s, mean of the last second, "
                                  "against the measured sustained bf16 peak"},
            "layer_ms": layer_ms, "layer_tokens_per_s": cfg.T / (layer_ms / 1e3),
            "ffn": {"F": F, "expert": "silu(x W1^T) * (x W3^T) then W2, bf16 weights, fp32 "
                                      "accumulation, bf16 intermediate",
                    "ffn_ms": ffn_ms, "ffn_tflops": ffn_tflops,
                    "frac": ffn_tflops / peak, "layer_ms": ffn_layer_ms,
                    "layer_tokens_per_s": cfg.T / (ffn_layer_ms / 1e3)},
            "clocks": clk.summary(), "clocks_ffn": clk_ffn.summary()}


# ------------------------------------------------------------ wave scan ----

def run_wave_scan(args, cfg):
    """T(W) of the wave-pipelined layer on one workload: for every W that
    divides E (up to 64), one captured step of route, counts and, per wave,
    dispatch(w) / experts(w) / combine of the tokens whose last wave is w on
    three streams ("不规则与流水化 AllToAll", section "Wave-Scheduled 流水化"),
    L2 flushed first.  The sequential layer (every wave dispatched, then the
    experts, then the combine, one stream) is timed beside it, the two steps'
    replays alternating so both see the same clocks.  The pipelined
    times are fitted to T(W) = W*alpha + M/beta + M/(W*beta) with M the
    exchanged bytes (T*k*H*2), giving the model's W* = sqrt(M/(alpha*beta))
    beside the measured best W (section "最优 wave 数")."""
    import torch

    from combine_moe_route_17_b300 import MoEPipeline, wavefit

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    inp = wl.make_inputs(cfg)
    ffn = args.wave_expert == "ffn"
    p = MoEPipeline(cfg.replace(W=1), device=dev, expert_major=ffn)
    p.load_inputs(torch.from_numpy(inp["logits"]), torch.from_numpy(inp["x"].view(np.int16)),
                  torch.from_numpy(inp["scale"]))
    if ffn:
        # the gated FFN expert on the tensor cores, seeded random bf16 weights
        F = args.ffn_dim
        gen = torch.Generator(device=dev)
        gen.manual_seed(cfg.seed + 29)
        w13 = (torch.randn((cfg.E, 2 * F, cfg.H), generator=gen, device=dev)
               / float(np.sqrt(cfg.H))).to(torch.bfloat16)
        w2 = (torch.randn((cfg.E, cfg.H, F), generator=gen, device=dev)
              / float(np.sqrt(F))).to(torch.bfloat16)
        p.set_ffn(w13, w2)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    base = torch.cuda.current_stream(dev)
    s0, s1, s2 = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    steps = max(3, min(args.steps, 50))
    M = cfg.T * cfg.k * cfg.H * 2

    def capture(body):
        ev = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(2)]
        g = torch.cuda.CUDAGraph()
        s0.wait_stream(base)
        with torch.cuda.graph(g, stream=s0):
            flush.zero_()
            ev[0].record(s0)
            body()
            ev[1].record(s0)
        torch.cuda.synchronize(dev)
        return g, ev

    def timed_pair(body_a, body_b):
        """Replays the two captured steps alternately (a, b, a, b, ...), so
        both see the same clocks and power state; mean and spread of each."""
        ga, eva = capture(body_a)
        gb, evb = capture(body_b)
        ma, mb = [], []
        for r in range(steps + 3):
            for g, ev, acc in ((ga, eva, ma), (gb, evb, mb)):
                g.replay()
                torch.cuda.synchronize(dev)
                if r >= 3:
                    acc.append(ev[0].elapsed_time(ev[1]))
        p.check_device_error()
        return (float(np.mean(ma)), float(np.std(ma))), (float(np.mean(mb)), float(np.std(mb)))

    def sequential():
        p.route_count(s0)
        p.dispatch_waves(s0)
        p.expert(s0)
        p.combine(s0)
        p.imbalance(s0)

    points = []
    for W in wavefit.divisor_waves(cfg.E, (1, 2, 4, 8, 16, 32, 64)):
        p.set_waves(W)
        handoff = [torch.cuda.Event() for _ in range(2 * W)]
        (pipe_ms, pipe_sd), (seq_ms, seq_sd) = timed_pair(
            lambda: p.step_pipelined((s0, s1, s2), handoff), sequential)
        points.append({"W": W, "pipelined_ms": pipe_ms, "pipelined_ms_std": pipe_sd,
                       "sequential_ms": seq_ms, "sequential_ms_std": seq_sd})
    f = wavefit.fit([q["W"] for q in points], [q["pipelined_ms"] / 1e3 for q in points], M)
    lin_p = wavefit.fit_linear([q["W"] for q in points], [q["pipelined_ms"] / 1e3 for q in points])
    lin_s = wavefit.fit_linear([q["W"] for q in points], [q["sequential_ms"] / 1e3 for q in points])
    expert = (f"gated FFN experts on the tensor cores (F = {args.ffn_dim}, expert-major rows)"
              if ffn else "stand-in experts")
    return {"metric": "wave-pipelined MoE layer time T(W) (route, counts, W-wave dispatch, "
                      f"{expert}, combine)",
            "workload": cfg.name, "unit": "ms", "steps": steps, "M_bytes": M,
            "config": {"T": cfg.T, "H": cfg.H, "E": cfg.E, "k": cfg.k, "R": cfg.R,
                       "expert": expert,
                       "l2": f"flushed between steps ({L2_FLUSH_BYTES >> 20} MB write)",
                       "launch": "cuda graph, three streams (dispatch / experts / combine)"},
            "points": points,
            "fit": {"alpha_us": f["alpha_s"] * 1e6, "beta_GBps": f["beta_Bps"] / 1e9,
                    "w_star": f["w_star"], "w_best_measured": f["w_best_measured"],
                    "r2": f["r2"], "fitted_ms": [t * 1e3 for t in f["fitted_s"]]},
            "linear_fit": {"pipelined": {"t0_ms": lin_p["t0_s"] * 1e3,
                                         "per_wave_us": lin_p["alpha_s"] * 1e6, "r2": lin_p["r2"]},
                           "sequential": {"t0_ms": lin_s["t0_s"] * 1e3,
                                          "per_wave_us": lin_s["alpha_s"] * 1e6,
                                          "r2": lin_s["r2"]}}}


# ------------------------------------------------------- oracle (CPU) ----

def oracle_step(cfg, inp, toks):
    """One oracle pass over the tokens [0, toks): route, counts, dispatch maps
    and rows, combine and statistics; the stand-in expert runs untimed.
    Returns the timed seconds."""
    import oracle

    sub = cfg.replace(T=toks)
    lg = inp["logits"][:toks]
    x = inp["x"][:toks]
    t0 = time.perf_counter()
    idx, w = oracle.route_topk(lg, sub.k, sub.n_groups, sub.topk_groups, sub.group_topn)
    cnt = oracle.send_counts(idx, sub.E, sub.R)
    maps = oracle.dispatch_maps(idx, sub.E, sub.R)
    _, recv = oracle.dispatch_rows(x, idx, maps, sub.E, want_send=False)
    t1 = time.perf_counter()
    out = oracle.expert_standin(recv, idx, maps["slot_of"], inp["scale"])
    t2 = time.perf_counter()
    oracle.combine(out, maps["slot_of"], w)
    oracle.imbalance_stats(cnt["c"], sub.T, sub.k, sub.R)
    t3 = time.perf_counter()
    return (t1 - t0) + (t3 - t2)


def oracle_step_partitions(cfg, inp, toks, pool, nthreads, keep=None):
    """The same oracle functions run as R independent source-partition tasks
    on `nthreads` threads (ctypes releases the GIL during each call): every
    partition's routing, row copies and combine in parallel; the counts and
    the row maps (O(T k) integer work over all partitions) on one thread
    between them; the stand-in expert untimed.  Returns the timed seconds
    (and, when `keep` is a dict, stores idx, w, the maps, recv and y in it)."""
    import ctypes

    import oracle

    L = oracle.lib()
    sub = cfg.replace(T=toks)
    R, k, H, E = sub.R, sub.k, sub.H, sub.E
    Tr = toks // R
    lg = inp["logits"][:toks]
    x = np.ascontiguousarray(inp["x"][:toks])
    vp = ctypes.c_void_p
    t0 = time.perf_counter()
    parts = list(pool.map(lambda s: oracle.route_topk(lg[s * Tr:(s + 1) * Tr], k, sub.n_groups,
                                                      sub.topk_groups, sub.group_topn),
                          range(R)))
    idx = np.concatenate([q[0] for q in parts])
    w = np.concatenate([q[1] for q in parts])
    cnt = oracle.send_counts(idx, E, R)
    maps = oracle.dispatch_maps(idx, E, R)
    so = maps["slot_of"]
    recv = np.zeros((toks * k, H), np.uint16)

    def rows(s):
        a, b = s * Tr, (s + 1) * Tr
        return L.oracle_dispatch_rows(Tr, H, E, k, 1, -1, idx[a:b], x[a:b], None,
                                      so[a:b].ctypes.data_as(vp), None, recv.ctypes.data_as(vp))

    if any(list(pool.map(rows, range(R)))):
        raise RuntimeError("oracle dispatch_rows rejected a partition")
    t1 = time.perf_counter()
    out = oracle.expert_standin(recv, idx, so, inp["scale"])
    t2 = time.perf_counter()
    y = np.zeros((toks, H), np.uint16)

    def comb(s):
        return L.oracle_combine(toks, H, k, s * Tr, (s + 1) * Tr, out, so, w, y)

    if any(list(pool.map(comb, range(R)))):
        raise RuntimeError("oracle combine rejected a partition")
    oracle.imbalance_stats(cnt["c"], sub.T, sub.k, sub.R)
    t3 = time.perf_counter()
    if keep is not None:
        keep.update(idx=idx, w=w, slot_of=so, src_row=maps["src_row"], recv=recv, y=y, **cnt)
    return (t1 - t0) + (t3 - t2)


def run_cpu_baseline_partitions(cfg, inp, budget_s: float):
    """The oracle over the R source partitions on min(R, usable cores)
    threads: the all-cores figure beside the single-thread one."""
    from concurrent.futures import ThreadPoolExecutor

    import oracle

    oracle.build()
    nthreads = max(1, min(cfg.R, len(os.sched_getaffinity(0))))
    with ThreadPoolExecutor(max_workers=nthreads) as pool:
        probe = max(cfg.R, (min(cfg.T, 4096) // cfg.R) * cfg.R)
        dt = oracle_step_partitions(cfg, inp, probe, pool, nthreads)
        toks = int(probe * (budget_s / 4) / max(dt, 1e-6))
        toks = max(cfg.R, min(cfg.T, (toks // cfg.R) * cfg.R))
        secs, n = 0.0, 0
        while secs < budget_s and n < 50:
            secs += oracle_step_partitions(cfg, inp, toks, pool, nthreads)
            n += 1
    return {"value": toks * n / secs, "unit": "tokens/s", "cores": nthreads, "kind": "oracle",
            "sample": f"{n} oracle steps over tokens [0,{toks}) of {cfg.name} as {cfg.R} "
                      f"source-partition tasks on {nthreads} threads (stand-in expert "
                      f"untimed), {secs:.1f} s; host os.cpu_count()={os.cpu_count()}, "
                      f"affinity={len(os.sched_getaffinity(0))}"}


def oracle_sample_tokens(cfg, seconds_per_step: float, inp) -> int:
    """Largest token count (a multiple of R, at most T) whose oracle step fits
    the per-step budget, from a probe on a small slice."""
    probe = max(cfg.R, (min(cfg.T, 1024) // cfg.R) * cfg.R)
    dt = oracle_step(cfg, inp, probe)
    toks = int(probe * seconds_per_step / max(dt, 1e-6))
    toks = max(cfg.R, min(cfg.T, (toks // cfg.R) * cfg.R))
    return toks


def cpu_cores_used() -> int:
    return 1


def run_cpu_baseline(cfg, inp, budget_s: float):
    """The oracle as it stands on the host: whole-workload steps if they fit
    the budget, else a token prefix; single thread."""
    import oracle

    oracle.build()
    toks = oracle_sample_tokens(cfg, budget_s / 4, inp)
    secs, n = 0.0, 0
    while secs < budget_s and n < 50:
        secs += oracle_step(cfg, inp, toks)
        n += 1
    return {"value": toks * n / secs, "unit": "tokens/s", "cores": cpu_cores_used(),
            "kind": "oracle",
            "sample": f"{n} oracle steps over tokens [0,{toks}) of {cfg.name} "
                      f"(stand-in expert untimed), {secs:.1f} s, one thread; "
                      f"host os.cpu_count()={os.cpu_count()}, "
                      f"affinity={len(os.sched_getaffinity(0))}"}


def run_reference(args, cfg, rank, world):
    import oracle

    if rank != 0:
        return None
    oracle.build()
    inp = wl.make_inputs(cfg)
    budget_total = 150.0
    per_step = budget_total / max(1, args.steps + args.warmup)
    toks = oracle_sample_tokens(cfg, min(per_step, 6.0), inp)
    for _ in range(args.warmup):
        oracle_step(cfg, inp, toks)
    secs = 0.0
    for _ in range(args.steps):
        secs += oracle_step(cfg, inp, toks)
    value = toks * args.steps / secs
    sample = (f"each step: oracle over tokens [0,{toks}) of {cfg.name} (stand-in expert "
              f"untimed), one thread; host os.cpu_count()={os.cpu_count()}")
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": secs / args.steps * 1e3 * cfg.T / toks,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded; routing logits with the workload's bias family)",
            "config": {"workload": cfg.name, "T": cfg.T, "H": cfg.H, "E": cfg.E, "k": cfg.k,
                       "R": cfg.R, "W": cfg.W, "sample_tokens": toks},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cpu_cores_used(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "gpu_launches": 0}


# ------------------------------------------------------------------ main ----

def main(argv=None):
    args = parse_args(argv)
    rank, world, local = dist_env()
    if args.workload == "sweep":
        if args.impl != "cuda" or world > 1:
            raise SystemExit("the sweep runs the CUDA path on one GPU")
        print(json.dumps(run_sweep(args)), flush=True)
        return 0
    cfg = wl.CONFIGS[args.workload]
    if args.tokens is not None:
        if args.tokens <= 0 or args.tokens % cfg.R:
            raise SystemExit(f"--tokens must be a positive multiple of R = {cfg.R}")
        cfg = wl.reduced(cfg, T=args.tokens)
    if args.expert_gemm:
        if args.impl != "cuda" or world > 1:
            raise SystemExit("the expert GEMM layer runs the CUDA path on one GPU")
        print(json.dumps(run_expert_gemm(args, cfg)), flush=True)
        return 0
    if args.capacity is not None:
        if args.impl != "cuda" or world > 1:
            raise SystemExit("the capacity variant runs the CUDA path on one GPU")
        print(json.dumps(run_capacity(args, cfg)), flush=True)
        return 0
    if args.wave_scan:
        if args.impl != "cuda" or world > 1:
            raise SystemExit("the wave scan runs the CUDA path on one GPU")
        print(json.dumps(run_wave_scan(args, cfg)), flush=True)
        return 0
    if world > 1:
        import torch.distributed as dist

        if args.impl == "reference":
            if rank != 0:
                return 0
        else:
            import torch

            torch.cuda.set_device(local)
            dist.init_process_group("nccl")
    if args.impl == "reference":
        res = run_reference(args, cfg, rank, world)
    else:
        res = run_cuda(args, cfg, rank, world, local)
        if rank == 0 and world == 1 and not args.no_cpu_baseline:
            cin = wl.make_inputs(cfg)
            res["cpu_baseline"] = run_cpu_baseline(cfg, cin, args.cpu_seconds)
            res["cpu_baseline_all_cores"] = run_cpu_baseline_partitions(cfg, cin,
                                                                        args.cpu_seconds / 2)
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)
    if world > 1 and args.impl != "reference":
        import torch.distributed as dist

        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
