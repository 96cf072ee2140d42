"""Python binding of the C ABI in include/moe_route.h (ctypes).

Argument marshalling only: every step of the path runs in the CUDA kernels of
lib/libmoe_route.so.  torch supplies device memory and streams.  There is no
CPU fallback: if the library is missing the first call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "lib", "libmoe_route.so")

MOE_OK = 0
MOE_ERR_INVALID_ARG = 1
MOE_ERR_UNSUPPORTED = 2
MOE_ERR_CUDA = 3
MOE_ERR_TIMEOUT = 4
MOE_ERR_DEVICE_CHECK = 5
MOE_STAGED = 1
MOE_EXPERT_MAJOR = 2
MOE_BULK_COPY = 4

_STATUS_NAMES = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED",
                 3: "MOE_ERR_CUDA", 4: "MOE_ERR_TIMEOUT", 5: "MOE_ERR_DEVICE_CHECK"}


class MoEError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {_STATUS_NAMES.get(status, status)}")


class Shape(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("H", ctypes.c_int32), ("E", ctypes.c_int32),
                ("k", ctypes.c_int32), ("R", ctypes.c_int32), ("W", ctypes.c_int32),
                ("n_groups", ctypes.c_int32), ("topk_groups", ctypes.c_int32),
                ("group_topn", ctypes.c_int32)]

    @classmethod
    def of(cls, cfg) -> "Shape":
        return cls(cfg.T, cfg.H, cfg.E, cfg.k, cfg.R, cfg.W, cfg.n_groups,
                   cfg.topk_groups, cfg.group_topn)


class Stats(ctypes.Structure):
    _fields_ = [("max_load", ctypes.c_int32), ("min_load", ctypes.c_int32),
                ("gini_num", ctypes.c_int64), ("gini_den", ctypes.c_int64),
                ("max_over_mean", ctypes.c_double), ("hot_over_cold", ctypes.c_double),
                ("gini", ctypes.c_double)]


STATS_BYTES = ctypes.sizeof(Stats)


class Placement(ctypes.Structure):
    _fields_ = [("gini_num_before", ctypes.c_int64), ("gini_num_after", ctypes.c_int64),
                ("gini_den", ctypes.c_int64), ("max_rank_load_before", ctypes.c_int64),
                ("max_rank_load_after", ctypes.c_int64), ("gini_before", ctypes.c_double),
                ("gini_after", ctypes.c_double)]


PLACEMENT_BYTES = ctypes.sizeof(Placement)

# Exported symbol -> argument types (every entry returns moe_status unless noted).
_vp, _i, _u, _sz, _u64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_uint, ctypes.c_size_t, ctypes.c_uint64
_SP = ctypes.POINTER(Shape)
SIGNATURES = {
    "moe_validate_shape": [_SP],
    "moe_workspace_size": [_SP, ctypes.POINTER(ctypes.c_size_t)],
    "moe_workspace_init": [_vp, _sz, _vp],
    "moe_route_topk": [_SP, _vp, _vp, _vp, _vp, _vp],
    "moe_build_send_counts": [_SP, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp],
    "moe_build_send_counts_noalloc": [_SP, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp],
    "moe_route_and_count": [_SP, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp],
    "moe_expert_offsets": [_SP, _vp, _sz, _vp, _vp],
    "moe_dispatch": [_SP, _vp, _vp, _vp, _sz, _i, _u, _vp, _vp, _vp, _vp, _vp, _vp],
    "moe_permute_by_device": [_SP, _vp, _vp, _vp, _sz, _i, _vp, _vp, _vp, _vp],
    "moe_all_to_all": [_SP, _vp, _sz, _i, _i, _vp, _vp, _vp],
    "moe_combine": [_SP, _vp, _vp, _vp, _vp, _sz, _u, _vp, _vp, _vp, _vp],
    "moe_imbalance_stats": [_SP, _vp, _vp, _vp, _vp],
    "moe_expert_standin": [_SP, _vp, _vp, _vp, _vp, _vp],
    "moe_expert_standin_wave": [_SP, _vp, _vp, _vp, _i, _vp, _vp],
    "moe_combine_wave": [_SP, _vp, _vp, _vp, _vp, _vp, _i, _vp, _vp],
    "moe_expert_capacity": [_SP, ctypes.c_double, ctypes.POINTER(ctypes.c_int64)],
    "moe_dispatch_capacity": [_SP, ctypes.c_int64, _vp, _vp, _vp, _sz, _vp, _vp, _vp, _vp],
    "moe_expert_standin_capacity": [_SP, ctypes.c_int64, _vp, _vp, _vp, _vp, _vp],
    "moe_combine_capacity": [_SP, ctypes.c_int64, _vp, _vp, _vp, _vp, _vp, _vp],
    "moe_place_experts_greedy": [_SP, _vp, _vp, _vp, _vp, _vp],
    "moe_expert_gemm": [_SP, _vp, _vp, _i, _vp, _vp, _vp, _vp],
    "moe_expert_ffn": [_SP, _vp, _vp, _vp, _i, _vp, _vp, _vp, _vp, _vp],
    "moe_expert_gemm_wave": [_SP, _vp, _vp, _i, _vp, _vp, _i, _vp, _vp],
    "moe_expert_ffn_wave": [_SP, _vp, _vp, _vp, _i, _vp, _vp, _vp, _i, _vp, _vp],
    "moe_dirichlet_alpha": [_SP, _vp, _vp, _vp],
    "moe_get_device_error": [_vp, _vp],
    "moe_debug_set_fault": [_vp, _i, _u64, _vp],
    "moe_status_string": [_i],
    "moe_abi_version": [],
}

_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return LIB_PATH


def lib():
    """Loads libmoe_route.so (after torch, so both share one CUDA runtime)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"CUDA library {LIB_PATH} is missing; build it with "
                    "`python -m combine_moe_route_17_b300.build` (no CPU fallback exists)")
            L = ctypes.CDLL(LIB_PATH)
            for name, args in SIGNATURES.items():
                fn = getattr(L, name)
                fn.argtypes = args
                fn.restype = ctypes.c_int
            L.moe_status_string.restype = ctypes.c_char_p
            _lib = L
    return _lib


def _check(status: int, what: str):
    if status != MOE_OK:
        raise MoEError(status, what)


def _stream(stream: Optional[torch.cuda.Stream]) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _p(t: Optional[torch.Tensor], dtype=None, what: str = "") -> Optional[int]:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{what}: expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{what}: expected a contiguous tensor")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{what}: expected {dtype}, got {t.dtype}")
    return t.data_ptr() or None


def _bf16(t, what):
    if t is None:
        return None
    if t.dtype not in (torch.bfloat16, torch.int16, torch.uint16):
        raise ValueError(f"{what}: expected bf16 rows, got {t.dtype}")
    return _p(t, None, what)


def validate_shape(shape: Shape):
    _check(lib().moe_validate_shape(ctypes.byref(shape)), "moe_validate_shape")


def workspace_size(shape: Shape) -> int:
    n = ctypes.c_size_t(0)
    _check(lib().moe_workspace_size(ctypes.byref(shape), ctypes.byref(n)), "moe_workspace_size")
    return int(n.value)


def new_workspace(shape: Shape, device="cuda", stream=None) -> torch.Tensor:
    nbytes = workspace_size(shape)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=device)
    _check(lib().moe_workspace_init(ws.data_ptr(), nbytes, _stream(stream)), "moe_workspace_init")
    return ws


def route_topk(shape, logits, idx, w, ws=None, stream=None):
    _check(lib().moe_route_topk(ctypes.byref(shape), _p(logits, torch.float32, "logits"),
                                _p(idx, torch.int32, "idx"), _p(w, torch.float32, "w"),
                                _p(ws, torch.uint8, "workspace"), _stream(stream)),
           "moe_route_topk")


def build_send_counts(shape, idx, counts: dict, ws, stream=None):
    _check(lib().moe_build_send_counts(
        ctypes.byref(shape), _p(idx, torch.int32, "idx"),
        _p(counts["c"], torch.int32, "expert_counts"), _p(counts["C"], torch.int32, "C"),
        _p(counts["S"], torch.int32, "S"), _p(counts["send_off"], torch.int64, "send_off"),
        _p(counts["recv_off"], torch.int64, "recv_off"),
        _p(counts["recv_base"], torch.int64, "recv_base"),
        _p(ws, torch.uint8, "workspace"), ws.numel(), _stream(stream)), "moe_build_send_counts")


def route_and_count(shape, logits, idx, w, counts: dict, ws, stream=None):
    """route_topk then build_send_counts, fused into one launch where it can be."""
    _check(lib().moe_route_and_count(
        ctypes.byref(shape), _p(logits, torch.float32, "logits"), _p(idx, torch.int32, "idx"),
        _p(w, torch.float32, "w"), _p(counts["c"], torch.int32, "expert_counts"),
        _p(counts["C"], torch.int32, "C"), _p(counts["S"], torch.int32, "S"),
        _p(counts["send_off"], torch.int64, "send_off"),
        _p(counts["recv_off"], torch.int64, "recv_off"),
        _p(counts["recv_base"], torch.int64, "recv_base"),
        _p(ws, torch.uint8, "workspace"), ws.numel(), _stream(stream)), "moe_route_and_count")


def expert_offsets(shape, ws, expert_off, stream=None):
    """expert_off int32 [E+1]: the first expert-major row of every expert,
    from the table the count pass left in the workspace."""
    _check(lib().moe_expert_offsets(ctypes.byref(shape), _p(ws, torch.uint8, "workspace"),
                                    ws.numel(), _p(expert_off, torch.int32, "expert_off"),
                                    _stream(stream)), "moe_expert_offsets")


def _flags(staged, expert_major, bulk=False):
    return ((MOE_STAGED if staged else 0) | (MOE_EXPERT_MAJOR if expert_major else 0)
            | (MOE_BULK_COPY if bulk else 0))


def dispatch(shape, x, idx, ws, recv, slot_of, src_row=None, wave=-1, staged=False, send=None,
             send_pos=None, stream=None, expert_major=False, bulk=False):
    _check(lib().moe_dispatch(
        ctypes.byref(shape), _bf16(x, "x"), _p(idx, torch.int32, "idx"),
        _p(ws, torch.uint8, "workspace"), ws.numel(), int(wave),
        _flags(staged, expert_major, bulk),
        _bf16(send, "send"), _bf16(recv, "recv"), _p(slot_of, torch.int32, "slot_of"),
        _p(src_row, torch.int32, "src_row"), _p(send_pos, torch.int32, "send_pos"),
        _stream(stream)), "moe_dispatch")


def permute_by_device(shape, x, idx, ws, send, send_pos, slot_of=None, wave=-1, stream=None):
    _check(lib().moe_permute_by_device(
        ctypes.byref(shape), _bf16(x, "x"), _p(idx, torch.int32, "idx"),
        _p(ws, torch.uint8, "workspace"), ws.numel(), int(wave), _bf16(send, "send"),
        _p(send_pos, torch.int32, "send_pos"), _p(slot_of, torch.int32, "slot_of"),
        _stream(stream)), "moe_permute_by_device")


def all_to_all(shape, ws, src, dst, wave=-1, direction=0, stream=None):
    _check(lib().moe_all_to_all(ctypes.byref(shape), _p(ws, torch.uint8, "workspace"), ws.numel(),
                                int(wave), int(direction), _bf16(src, "src"), _bf16(dst, "dst"),
                                _stream(stream)), "moe_all_to_all")


def combine(shape, expert_out, slot_of, w, y, ws=None, staged=False, staging=None,
            send_pos=None, stream=None, expert_major=False):
    _check(lib().moe_combine(
        ctypes.byref(shape), _bf16(expert_out, "expert_out"), _p(slot_of, torch.int32, "slot_of"),
        _p(w, torch.float32, "w"), _p(ws, torch.uint8, "workspace"),
        0 if ws is None else ws.numel(), _flags(staged, expert_major), _bf16(staging, "staging"),
        _p(send_pos, torch.int32, "send_pos"), _bf16(y, "y"), _stream(stream)), "moe_combine")


def imbalance_stats(shape, expert_counts, stats_dev, rank_load=None, stream=None):
    if stats_dev.numel() * stats_dev.element_size() < STATS_BYTES:
        raise ValueError("stats buffer too small")
    _check(lib().moe_imbalance_stats(
        ctypes.byref(shape), _p(expert_counts, torch.int32, "expert_counts"),
        _p(stats_dev, None, "stats"), _p(rank_load, torch.int64, "rank_load"), _stream(stream)),
        "moe_imbalance_stats")


def expert_standin_wave(shape, idx, slot_of, scale, rows, wave=-1, stream=None):
    _check(lib().moe_expert_standin_wave(ctypes.byref(shape), _p(idx, torch.int32, "idx"),
                                         _p(slot_of, torch.int32, "slot_of"),
                                         _p(scale, torch.float32, "scale"), int(wave),
                                         _bf16(rows, "rows"), _stream(stream)),
           "moe_expert_standin_wave")


def combine_wave(shape, expert_out, slot_of, idx, w, y, ws=None, wave=-1, stream=None):
    _check(lib().moe_combine_wave(ctypes.byref(shape), _bf16(expert_out, "expert_out"),
                                  _p(slot_of, torch.int32, "slot_of"), _p(idx, torch.int32, "idx"),
                                  _p(w, torch.float32, "w"), _p(ws, torch.uint8, "workspace"),
                                  int(wave), _bf16(y, "y"), _stream(stream)), "moe_combine_wave")


def expert_capacity(shape, capacity_factor: float) -> int:
    ec = ctypes.c_int64()
    _check(lib().moe_expert_capacity(ctypes.byref(shape), float(capacity_factor),
                                     ctypes.byref(ec)), "moe_expert_capacity")
    return int(ec.value)


def dispatch_capacity(shape, capacity, x, idx, ws, cap_rows, cap_slot, dropped=None, stream=None):
    _check(lib().moe_dispatch_capacity(
        ctypes.byref(shape), int(capacity), _bf16(x, "x"), _p(idx, torch.int32, "idx"),
        _p(ws, torch.uint8, "workspace"), ws.numel(), _bf16(cap_rows, "cap_rows"),
        _p(cap_slot, torch.int32, "cap_slot"), _p(dropped, torch.int32, "dropped"),
        _stream(stream)), "moe_dispatch_capacity")


def expert_standin_capacity(shape, capacity, idx, cap_slot, scale, cap_rows, stream=None):
    _check(lib().moe_expert_standin_capacity(
        ctypes.byref(shape), int(capacity), _p(idx, torch.int32, "idx"),
        _p(cap_slot, torch.int32, "cap_slot"), _p(scale, torch.float32, "scale"),
        _bf16(cap_rows, "cap_rows"), _stream(stream)), "moe_expert_standin_capacity")


def combine_capacity(shape, capacity, cap_out, cap_slot, w, y, ws=None, stream=None):
    _check(lib().moe_combine_capacity(
        ctypes.byref(shape), int(capacity), _bf16(cap_out, "cap_out"),
        _p(cap_slot, torch.int32, "cap_slot"), _p(w, torch.float32, "w"),
        _p(ws, torch.uint8, "workspace"), _bf16(y, "y"), _stream(stream)),
        "moe_combine_capacity")


def expert_gemm(shape, rows, weights, expert_counts, out, ws=None, stream=None, wave=-1):
    """out[r] = rows[r] @ weights[e(r)].T on the tensor cores; weights bf16
    [E][N][H], rows the expert-major recv rows; wave >= 0 runs only that
    wave's experts."""
    N = int(weights.shape[1])
    if wave < 0:
        _check(lib().moe_expert_gemm(ctypes.byref(shape), _bf16(rows, "rows"),
                                     _bf16(weights, "weights"), N,
                                     _p(expert_counts, torch.int32, "expert_counts"),
                                     _bf16(out, "out"), _p(ws, torch.uint8, "workspace"),
                                     _stream(stream)), "moe_expert_gemm")
        return
    _check(lib().moe_expert_gemm_wave(ctypes.byref(shape), _bf16(rows, "rows"),
                                      _bf16(weights, "weights"), N,
                                      _p(expert_counts, torch.int32, "expert_counts"),
                                      _bf16(out, "out"), int(wave),
                                      _p(ws, torch.uint8, "workspace"), _stream(stream)),
           "moe_expert_gemm_wave")


def pack_gated_weights(w1: torch.Tensor, w3: torch.Tensor) -> torch.Tensor:
    """[E][F][H] gate and up weights -> the [E][2F][H] layout moe_expert_ffn
    reads: per expert, F/128 blocks of 128 rows of W1 then the same 128 rows
    of W3 (a layout change only)."""
    E, F, H = w1.shape
    if w3.shape != w1.shape or F % 128:
        raise ValueError("w1 and w3 must both be [E][F][H] with F % 128 == 0")
    return torch.stack([w1.reshape(E, F // 128, 128, H), w3.reshape(E, F // 128, 128, H)],
                       dim=2).reshape(E, 2 * F, H).contiguous()


def expert_ffn(shape, rows, w13, w2, expert_counts, hidden, out, ws=None, stream=None,
               wave=-1):
    """Gated FFN expert on the expert-major rows (see pack_gated_weights);
    wave >= 0 runs only that wave's experts."""
    F = int(w2.shape[2])
    _check(lib().moe_expert_ffn_wave(ctypes.byref(shape), _bf16(rows, "rows"), _bf16(w13, "w13"),
                                     _bf16(w2, "w2"), F,
                                     _p(expert_counts, torch.int32, "expert_counts"),
                                     _bf16(hidden, "hidden"), _bf16(out, "out"), int(wave),
                                     _p(ws, torch.uint8, "workspace"), _stream(stream)),
           "moe_expert_ffn_wave")


def place_experts_greedy(shape, expert_counts, placement, relabel, out, stream=None):
    """out: a device buffer of at least PLACEMENT_BYTES (e.g. float64 [8])."""
    if out.numel() * out.element_size() < PLACEMENT_BYTES:
        raise ValueError("placement output buffer too small")
    _check(lib().moe_place_experts_greedy(
        ctypes.byref(shape), _p(expert_counts, torch.int32, "expert_counts"),
        _p(placement, torch.int32, "placement"), _p(relabel, torch.int32, "relabel"),
        _p(out, None, "placement stats"), _stream(stream)), "moe_place_experts_greedy")


def decode_placement(out: torch.Tensor) -> dict:
    raw = bytes(out.cpu().numpy().tobytes()[:PLACEMENT_BYTES])
    st = Placement.from_buffer_copy(raw)
    return {f: getattr(st, f) for f, _ in Placement._fields_}


def dirichlet_alpha(shape, expert_counts, out, stream=None):
    """out: a device float64 tensor of at least one element."""
    _check(lib().moe_dirichlet_alpha(ctypes.byref(shape),
                                     _p(expert_counts, torch.int32, "expert_counts"),
                                     _p(out, torch.float64, "alpha"), _stream(stream)),
           "moe_dirichlet_alpha")


def decode_stats(stats_host: torch.Tensor) -> dict:
    raw = bytes(stats_host.cpu().numpy().tobytes()[:STATS_BYTES])
    st = Stats.from_buffer_copy(raw)
    return {f: getattr(st, f) for f, _ in Stats._fields_}


def expert_standin(shape, idx, slot_of, scale, rows, stream=None):
    _check(lib().moe_expert_standin(ctypes.byref(shape), _p(idx, torch.int32, "idx"),
                                    _p(slot_of, torch.int32, "slot_of"),
                                    _p(scale, torch.float32, "scale"), _bf16(rows, "rows"),
                                    _stream(stream)), "moe_expert_standin")


def get_device_error(ws, stream=None) -> int:
    """Synchronises the stream; returns and clears the workspace error word."""
    return int(lib().moe_get_device_error(_p(ws, torch.uint8, "workspace"), _stream(stream)))


def debug_set_fault(ws, tile: int, wait_ns: int = 0, stream=None):
    _check(lib().moe_debug_set_fault(_p(ws, torch.uint8, "workspace"), int(tile), int(wait_ns),
                                     _stream(stream)), "moe_debug_set_fault")


def status_string(status: int) -> str:
    return lib().moe_status_string(int(status)).decode()


def abi_version() -> int:
    return int(lib().moe_abi_version())
