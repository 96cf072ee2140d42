"""One MoE dispatch/combine pass over device-resident buffers.

``MoEPipeline`` owns the device buffers of one shape (torch allocations) and
runs the forward pass of an expert-parallel MoE layer through the C ABI:

    route_topk -> build_send_counts -> dispatch (W waves) -> expert -> combine
    -> imbalance_stats

("混合专家模型跨卡通信机制解析", section 四: gating, permute_by_device,
all_to_all, local experts, all_to_all, combine; the waves of "不规则与流水化
AllToAll", section "Wave-Scheduled 流水化").  The expert step is the scalar
stand-in ``out = bf16(s_e * recv)``; it is harness work and ``step`` runs it
between dispatch and combine.
"""
from __future__ import annotations

from typing import Optional

import torch

from . import binding as B


class MoEPipeline:
    def __init__(self, cfg, device: str = "cuda", staged: bool = False,
                 capacity_factor: Optional[float] = None, expert_major: bool = False,
                 fuse_route: bool = False, concurrent_waves: bool = True,
                 bulk_copy: bool = False):
        self.cfg = cfg
        self.fuse_route = fuse_route  # route_count(): one launch (moe_route_and_count)
        # dispatch_waves(): the W wave calls on W streams at once
        self.concurrent_waves = concurrent_waves
        self.bulk_copy = bulk_copy  # dispatch row copies with the bulk-copy engine
        self._wave_streams = []
        self.shape = B.Shape.of(cfg)
        B.validate_shape(self.shape)
        self.device = torch.device(device)
        self.staged = staged
        self.expert_major = expert_major  # recv rows ordered (rank, expert, source, token, slot)
        T, H, E, k, R = cfg.T, cfg.H, cfg.E, cfg.k, cfg.R
        dev = self.device
        i32, i64, f32, bf = torch.int32, torch.int64, torch.float32, torch.bfloat16
        self.ws = B.new_workspace(self.shape, dev)
        self.logits = torch.empty((T, E), dtype=f32, device=dev)
        self.x = torch.empty((T, H), dtype=bf, device=dev)
        self.scale = torch.empty(E, dtype=f32, device=dev)
        self.idx = torch.empty((T, k), dtype=i32, device=dev)
        self.w = torch.empty((T, k), dtype=f32, device=dev)
        self.counts = {
            "c": torch.empty(E, dtype=i32, device=dev),
            "C": torch.empty((R, E), dtype=i32, device=dev),
            "S": torch.empty((R, R), dtype=i32, device=dev),
            "send_off": torch.empty((R, R + 1), dtype=i64, device=dev),
            "recv_off": torch.empty((R, R + 1), dtype=i64, device=dev),
            "recv_base": torch.empty(R + 1, dtype=i64, device=dev),
        }
        self.recv = torch.empty((T * k, H), dtype=bf, device=dev)
        self.slot_of = torch.empty((T, k), dtype=i32, device=dev)
        self.src_row = torch.empty(T * k, dtype=i32, device=dev)
        self.send = torch.empty((T * k, H), dtype=bf, device=dev) if staged else None
        self.send_pos = torch.empty((T, k), dtype=i32, device=dev) if staged else None
        self.y = torch.empty((T, H), dtype=bf, device=dev)
        self.stats = torch.zeros(8, dtype=torch.float64, device=dev)  # holds one moe_stats
        # capacity-factor layout: fixed [E][EC][H] rows (EC = ceil(k f T / E))
        self.capacity = None
        if capacity_factor is not None:
            self.capacity = B.expert_capacity(self.shape, capacity_factor)
            self.cap_rows = torch.empty((E * self.capacity, H), dtype=bf, device=dev)
            self.cap_slot = torch.empty((T, k), dtype=i32, device=dev)
            self.dropped = torch.empty(E, dtype=i32, device=dev)
        self.rank_load = torch.empty(R, dtype=i64, device=dev)
        self.w13 = self.w2 = self.hidden = self.out = None  # set_ffn()

    def set_waves(self, W: int):
        """Switches the number of waves; the buffers do not depend on W (a
        wave is a sub-range of every (source, destination) block)."""
        cfg = self.cfg.replace(W=W)
        shape = B.Shape.of(cfg)
        B.validate_shape(shape)
        self.cfg, self.shape = cfg, shape

    # -------------------------------------------------------------- inputs --
    def load_inputs(self, logits, x_bits, scale, non_blocking: bool = False):
        """Copies host (or device) inputs into the device buffers."""
        self.logits.copy_(torch.as_tensor(logits), non_blocking=non_blocking)
        xb = torch.as_tensor(x_bits)
        if xb.dtype != torch.bfloat16:
            xb = xb.view(torch.int16).view(torch.bfloat16) if xb.dtype in (
                torch.int16, torch.uint16) else xb
        self.x.copy_(xb, non_blocking=non_blocking)
        self.scale.copy_(torch.as_tensor(scale), non_blocking=non_blocking)

    # ---------------------------------------------------------------- steps --
    def route(self, stream=None):
        B.route_topk(self.shape, self.logits, self.idx, self.w, self.ws, stream)

    def count(self, stream=None):
        B.build_send_counts(self.shape, self.idx, self.counts, self.ws, stream)

    def route_count(self, stream=None):
        """route then count: two launches, or one (moe_route_and_count) with
        fuse_route."""
        if self.fuse_route:
            B.route_and_count(self.shape, self.logits, self.idx, self.w, self.counts, self.ws,
                              stream)
        else:
            self.route(stream)
            self.count(stream)

    def dispatch(self, wave: int = -1, stream=None):
        B.dispatch(self.shape, self.x, self.idx, self.ws, self.recv, self.slot_of, self.src_row,
                   wave=wave, staged=self.staged, send=self.send, send_pos=self.send_pos,
                   stream=stream, expert_major=self.expert_major, bulk=self.bulk_copy)

    def dispatch_waves(self, stream=None):
        """The W wave calls of one pass.  Once the counts are done the wave
        calls share no data (each writes only its own rows), so with
        concurrent_waves each runs on a stream of its own, forked from
        `stream` and joined back into it: a wave's launch ramp and tail then
        overlap its neighbours' copies instead of idling the GPU.  Otherwise
        they run one after the other on `stream`."""
        W = self.cfg.W
        if W == 1:
            self.dispatch(-1, stream)
            return
        if not self.concurrent_waves:
            for w in range(W):
                self.dispatch(w, stream)
            return
        st = stream if stream is not None else torch.cuda.current_stream(self.device)
        while len(self._wave_streams) < W:
            self._wave_streams.append(torch.cuda.Stream(self.device))
        for w in range(W):
            ws_ = self._wave_streams[w]
            ws_.wait_stream(st)
            self.dispatch(w, ws_)
        for w in range(W):
            st.wait_stream(self._wave_streams[w])

    def set_ffn(self, w13: torch.Tensor, w2: torch.Tensor):
        """Makes the gated FFN expert (moe_expert_ffn) the expert of expert()
        and expert_wave(): w13 bf16 [E][2F][H] (binding.pack_gated_weights),
        w2 bf16 [E][H][F], on the device.  Its output rows go to ``out``,
        which the combine then reads.  Needs the expert-major layout."""
        if not self.expert_major:
            raise ValueError("the tensor-core expert reads the expert-major layout")
        T, H, E, k = self.cfg.T, self.cfg.H, self.cfg.E, self.cfg.k
        F = int(w2.shape[2])
        if tuple(w13.shape) != (E, 2 * F, H) or tuple(w2.shape) != (E, H, F):
            raise ValueError("w13 must be [E][2F][H] and w2 [E][H][F]")
        self.w13, self.w2 = w13, w2
        self.hidden = torch.empty((T * k, F), dtype=torch.bfloat16, device=self.device)
        self.out = torch.empty((T * k, H), dtype=torch.bfloat16, device=self.device)

    @property
    def expert_rows(self) -> torch.Tensor:
        """The rows the combine reads: the FFN's output, or recv (the stand-in
        expert works in place)."""
        return self.out if self.w13 is not None else self.recv

    def expert(self, stream=None):
        if self.w13 is not None:
            B.expert_ffn(self.shape, self.recv, self.w13, self.w2, self.counts["c"], self.hidden,
                         self.out, self.ws, stream)
        else:
            B.expert_standin(self.shape, self.idx, self.slot_of, self.scale, self.recv, stream)

    def combine(self, stream=None):
        if self.staged:
            B.combine(self.shape, self.expert_rows, None, self.w, self.y, self.ws, staged=True,
                      staging=self.send, send_pos=self.send_pos, stream=stream,
                      expert_major=self.expert_major)
        else:
            B.combine(self.shape, self.expert_rows, self.slot_of, self.w, self.y, self.ws,
                      stream=stream)

    def imbalance(self, stream=None):
        B.imbalance_stats(self.shape, self.counts["c"], self.stats, self.rank_load, stream)

    def expert_wave(self, wave: int, stream=None):
        if self.w13 is not None:
            B.expert_ffn(self.shape, self.recv, self.w13, self.w2, self.counts["c"], self.hidden,
                         self.out, self.ws, stream, wave=wave)
        else:
            B.expert_standin_wave(self.shape, self.idx, self.slot_of, self.scale, self.recv, wave,
                                  stream)

    def combine_wave(self, wave: int, stream=None):
        B.combine_wave(self.shape, self.expert_rows, self.slot_of, self.idx, self.w, self.y,
                       self.ws, wave, stream)

    def step_pipelined(self, streams, events=None):
        """One step with the waves pipelined over three streams ("不规则与流水化
        AllToAll", section "Wave-Scheduled 流水化"): dispatch(w) on streams[0],
        the experts of wave w on streams[1] once dispatch(w) is done, and the
        combine of the tokens whose last wave is w on streams[2] once the
        experts of wave w are done; so dispatch(w+1), experts(w) and
        combine(w-1) overlap.  `events` (optional) holds 2*W CUDA events to
        use for the hand-offs.  The statistics run on streams[0] after the
        counts.  Ends with streams[0] waiting for the other two."""
        import torch

        s0, s1, s2 = streams
        W = self.cfg.W
        ev = events or [torch.cuda.Event() for _ in range(2 * W)]
        self.route_count(s0)
        self.imbalance(s0)
        for w in range(W):
            self.dispatch(w, s0)
            ev[2 * w].record(s0)
            s1.wait_event(ev[2 * w])
            self.expert_wave(w, s1)
            ev[2 * w + 1].record(s1)
            s2.wait_event(ev[2 * w + 1])
            self.combine_wave(w, s2)
        s0.wait_stream(s1)
        s0.wait_stream(s2)

    def dispatch_capacity(self, stream=None):
        B.dispatch_capacity(self.shape, self.capacity, self.x, self.idx, self.ws, self.cap_rows,
                            self.cap_slot, self.dropped, stream)

    def expert_capacity(self, stream=None):
        B.expert_standin_capacity(self.shape, self.capacity, self.idx, self.cap_slot, self.scale,
                                  self.cap_rows, stream)

    def combine_capacity(self, stream=None):
        B.combine_capacity(self.shape, self.capacity, self.cap_rows, self.cap_slot, self.w,
                           self.y, self.ws, stream)

    def step_capacity(self, stream=None):
        """route, counts, capacity dispatch, stand-in expert, capacity combine,
        statistics."""
        self.route(stream)
        self.count(stream)
        self.dispatch_capacity(stream)
        self.expert_capacity(stream)
        self.combine_capacity(stream)
        self.imbalance(stream)

    def place_greedy(self, stream=None) -> dict:
        """Greedy expert placement of the current counts (device), returned
        with its Gini / largest-load summaries (synchronises)."""
        E = self.cfg.E
        dev = self.device
        if not hasattr(self, "placement"):
            self.placement = torch.empty(E, dtype=torch.int32, device=dev)
            self.relabel = torch.empty(E, dtype=torch.int32, device=dev)
            self.placement_out = torch.zeros(8, dtype=torch.float64, device=dev)
        B.place_experts_greedy(self.shape, self.counts["c"], self.placement, self.relabel,
                               self.placement_out, stream)
        return B.decode_placement(self.placement_out)

    def dirichlet_alpha(self, stream=None) -> float:
        """Fitted symmetric-Dirichlet alpha of the current counts (synchronises)."""
        if not hasattr(self, "alpha_out"):
            self.alpha_out = torch.zeros(1, dtype=torch.float64, device=self.device)
        B.dirichlet_alpha(self.shape, self.counts["c"], self.alpha_out, stream)
        return float(self.alpha_out.item())

    def expert_offsets(self, stream=None) -> torch.Tensor:
        """First recv row of every expert in the expert-major layout, int32
        [E+1]: the table the count pass computed (moe_expert_offsets)."""
        off = torch.empty(self.cfg.E + 1, dtype=torch.int32, device=self.device)
        B.expert_offsets(self.shape, self.ws, off, stream)
        return off

    def forward_to_experts(self, stream=None):
        self.route_count(stream)
        self.dispatch_waves(stream)

    def step(self, stream=None):
        """route, counts, dispatch, stand-in expert, combine, statistics."""
        self.forward_to_experts(stream)
        self.expert(stream)
        self.combine(stream)
        self.imbalance(stream)

    # ------------------------------------------------------------ results --
    def check_device_error(self, stream=None):
        st = B.get_device_error(self.ws, stream)
        if st != B.MOE_OK:
            raise B.MoEError(st, "device-side check")

    def stats_dict(self) -> dict:
        return B.decode_stats(self.stats)

    def results(self) -> dict:
        """Every output copied to the host (numpy)."""
        out = {"idx": self.idx, "w": self.w, "slot_of": self.slot_of, "src_row": self.src_row,
               **self.counts, "rank_load": self.rank_load}
        res = {k: v.cpu().numpy() for k, v in out.items()}
        res["y"] = self.y.view(torch.int16).cpu().numpy().view("uint16")
        res["stats"] = self.stats_dict()
        return res


class HostBatchRunner:
    """Steps over batches that live in pinned host memory, overlapping the
    copies of neighbouring steps with the compute of the current one.

    Two ``MoEPipeline`` buffer sets alternate.  Step i copies its logits and
    x into set i % 2 on an input stream, runs route, counts, the W dispatch
    waves, the stand-in expert, the combine and the statistics on a compute
    stream, and reads y and the statistics back on an output stream.  Events
    keep each set's buffers in order: the copy-in of step i waits for the
    compute of step i - 2 (which read that set's inputs), and the compute of
    step i waits for the read-back of step i - 2 (which read that set's y).
    So step i+1's host-to-device copy and step i-1's device-to-host copy run
    while step i computes, on a full-duplex link.
    """

    def __init__(self, cfg, device="cuda", **pipeline_kw):
        self.device = torch.device(device)
        self.pipes = [MoEPipeline(cfg, device=self.device, **pipeline_kw) for _ in range(2)]
        self.s_in, self.s_comp, self.s_out = (torch.cuda.Stream(self.device) for _ in range(3))
        self._comp_done = [None, None]
        self._out_done = [None, None]

    def load_scale(self, scale):
        for p in self.pipes:
            p.scale.copy_(torch.as_tensor(scale))

    def step(self, i: int, h_logits: torch.Tensor, h_x: torch.Tensor, h_y: torch.Tensor,
             h_stats: torch.Tensor):
        """Enqueues step i: h_logits fp32 [T][E] and h_x bf16 bits int16
        [T][H] in, h_y int16 [T][H] and h_stats float64 [8] out, all pinned.
        Returns the event that marks the end of its read-back."""
        b = i % 2
        p = self.pipes[b]
        if self._comp_done[b] is not None:
            self.s_in.wait_event(self._comp_done[b])
        with torch.cuda.stream(self.s_in):
            p.logits.copy_(h_logits, non_blocking=True)
            p.x.view(torch.int16).copy_(h_x, non_blocking=True)
        in_done = torch.cuda.Event()
        in_done.record(self.s_in)

        self.s_comp.wait_event(in_done)
        if self._out_done[b] is not None:
            self.s_comp.wait_event(self._out_done[b])
        st = self.s_comp
        p.forward_to_experts(st)
        p.expert(st)
        p.combine(st)
        p.imbalance(st)
        comp_done = torch.cuda.Event()
        comp_done.record(st)
        self._comp_done[b] = comp_done

        self.s_out.wait_event(comp_done)
        with torch.cuda.stream(self.s_out):
            h_y.copy_(p.y.view(torch.int16), non_blocking=True)
            h_stats.copy_(p.stats, non_blocking=True)
        out_done = torch.cuda.Event()
        out_done.record(self.s_out)
        self._out_done[b] = out_done
        return out_done

    def join(self, stream):
        """Makes `stream` wait for everything enqueued so far."""
        for s in (self.s_in, self.s_comp, self.s_out):
            stream.wait_stream(s)

    def check_device_error(self):
        for p in self.pipes:
            p.check_device_error()
