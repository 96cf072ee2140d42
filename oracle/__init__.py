"""CPU oracle for MoE expert-parallel dispatch and combine -- TEST INFRASTRUCTURE.

Plain, slow, single-threaded reference of what the dispatch/combine hot path
computes, written from the source pages (see ``moe_oracle.c`` for the
per-function citations).  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg and reference arm of ``bench.py`` may import it.  It shares no code with the
CUDA library; both sides only share the seeded input generators.

Parity status of each function:
  route_topk        pinned (brute force over k-subsets, library stable sort,
                    hand-built ties; weights: sum to 1, k=1 exact)
  send_counts       pinned (direct enumeration, invariants)
  dispatch_maps     pinned (O(n^2) lexicographic rank counting on tiny inputs)
  dispatch_rows     pinned (bit copies checked against x through the maps)
  expert_standin    pinned (torch's bf16 cast of the fp32 products)
  combine           pinned (closed form x * sum_j w_j s_j, identity when s = 1)
  imbalance_stats   pinned (hand-computed loads, Gini = 0 / (R-1)/R cases)
  bf16_from_double  pinned (torch's bf16 cast on fp32 inputs; exact ties)
  cost_model        pinned (the pages' printed W* example, calculus argmin)
  expert_capacity   pinned (hand values of eq. 3)
  capacity_maps     pinned (hand-worked drops; brute-force positions; no drops
                    at large f; kept + dropped = T*k)
  capacity_rows     pinned (kept rows are x, padding zero)
  capacity_standin  pinned (equals expert_standin on the kept rows)
  capacity_combine  pinned (equals combine when nothing is dropped; closed form
                    x * sum over kept j of w_j s_j; all dropped gives 0)
  place_greedy      pinned (hand-worked placements; E/R experts per rank; the
                    greedy max load within 4/3 of the brute-force optimum)
  placement_gini    pinned (contiguous placement equals imbalance_stats' Gini)
  dispatch_maps_expert_major  pinned (O(n^2) lexicographic ranks; a
                    re-sort of the rank-major rows; contiguous expert runs)
  expert_gemm       pinned (hand-computed 2x2 products; identity weights give
                    the rows back; experts own consecutive runs)
  expert_ffn        pinned (silu's closed values; identity gate/up/down weights;
                    the down projection equals expert_gemm on the intermediate)
  dirichlet_alpha   pinned (0 and +inf limits; the moment equation solved in
                    floating point from the shares; consistency on simulated
                    Dirichlet-multinomial counts)
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

from .cost_model import (  # noqa: F401
    wave_time, optimal_waves, optimal_waves_integer, p95_link_load_page,
    p95_link_load_exact_excess,
)

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_HDR = os.path.join(_HERE, "moe_oracle.h")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math", "-ffp-contract=off",
          "-fno-strict-aliasing", "-Wall"]


def build(force: bool = False) -> str:
    """Compile the oracle with gcc into oracle/_build/liboracle.so."""
    os.makedirs(_BUILD, exist_ok=True)
    newest = max(os.path.getmtime(_SRC), os.path.getmtime(_HDR))
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < newest:
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", *CFLAGS, "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _P(dt):
    return np.ctypeslib.ndpointer(dtype=dt, flags="C_CONTIGUOUS")


class _Stats(ctypes.Structure):
    _fields_ = [("max_load", ctypes.c_int32), ("min_load", ctypes.c_int32),
                ("gini_num", ctypes.c_int64), ("gini_den", ctypes.c_int64),
                ("max_over_mean", ctypes.c_double), ("hot_over_cold", ctypes.c_double),
                ("gini", ctypes.c_double)]


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            i32, i64, f32, f64, u16 = (_P(np.int32), _P(np.int64), _P(np.float32),
                                       _P(np.float64), _P(np.uint16))
            ci, vp = ctypes.c_int, ctypes.c_void_p
            L.oracle_bf16_from_double.argtypes = [ctypes.c_double]
            L.oracle_bf16_from_double.restype = ctypes.c_uint16
            L.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
            L.oracle_bf16_to_double.restype = ctypes.c_double
            L.oracle_bf16_round_array.argtypes = [f64, u16, ctypes.c_int64]
            L.oracle_route_topk.argtypes = [ci] * 6 + [f32, i32, f32]
            L.oracle_send_counts.argtypes = [ci] * 4 + [i32, i32, i32, i32, i64, i64, i64]
            L.oracle_dispatch_maps.argtypes = [ci] * 4 + [i32, vp, vp, vp]
            L.oracle_dispatch_rows.argtypes = [ci] * 6 + [i32, u16, vp, vp, vp, vp]
            L.oracle_expert_standin.argtypes = [ci] * 3 + [i32, i32, f32, u16, u16]
            L.oracle_combine.argtypes = [ci] * 5 + [u16, i32, f32, u16]
            L.oracle_imbalance_stats.argtypes = [ci] * 4 + [i32, ctypes.POINTER(_Stats), vp]
            i64s = ctypes.c_int64
            L.oracle_expert_capacity.argtypes = [ci, ci, ci, ctypes.c_double]
            L.oracle_expert_capacity.restype = i64s
            L.oracle_capacity_maps.argtypes = [ci, ci, ci, i64s, i32, i32, i32]
            L.oracle_capacity_rows.argtypes = [ci, ci, ci, ci, i64s, u16, i32, u16]
            L.oracle_capacity_standin.argtypes = [ci, ci, i64s, f32, u16, u16]
            L.oracle_capacity_combine.argtypes = [ci, ci, ci, u16, i32, f32, u16]
            L.oracle_dispatch_maps_expert_major.argtypes = [ci, ci, ci, i32, i32, vp, i64]
            L.oracle_dispatch_maps_expert_major.restype = ctypes.c_int
            L.oracle_place_greedy.argtypes = [ci, ci, i32, i32, i32]
            L.oracle_placement_gini.argtypes = [ci, ci, i32, i32, ctypes.POINTER(i64s),
                                                ctypes.POINTER(i64s),
                                                ctypes.POINTER(ctypes.c_double)]
            L.oracle_dirichlet_alpha.argtypes = [ci, i32, ctypes.POINTER(ctypes.c_double)]
            for name in ("oracle_place_greedy", "oracle_placement_gini",
                         "oracle_dirichlet_alpha"):
                getattr(L, name).restype = ctypes.c_int
            for name in ("oracle_route_topk", "oracle_send_counts", "oracle_dispatch_maps",
                         "oracle_dispatch_rows", "oracle_expert_standin", "oracle_combine",
                         "oracle_imbalance_stats", "oracle_capacity_maps",
                         "oracle_capacity_rows", "oracle_capacity_standin",
                         "oracle_capacity_combine"):
                getattr(L, name).restype = ctypes.c_int
            _lib = L
    return _lib


def _check(rc, what):
    if rc != 0:
        raise ValueError(f"oracle {what} rejected its arguments (rc={rc})")


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


# ------------------------------------------------------------------ bf16 ----

def bf16_from_double(v: float) -> int:
    return int(lib().oracle_bf16_from_double(float(v)))


def bf16_round(v) -> np.ndarray:
    """Round an array of reals (fp64) to bf16 bit patterns (uint16)."""
    a = np.ascontiguousarray(v, dtype=np.float64)
    out = np.empty(a.shape, dtype=np.uint16)
    lib().oracle_bf16_round_array(a.reshape(-1), out.reshape(-1), a.size)
    return out


def bf16_to_f64(bits) -> np.ndarray:
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


# --------------------------------------------------------------- routing ----

def route_topk(logits: np.ndarray, k: int, n_groups: int = 1, topk_groups: int = 0,
               group_topn: int = 0):
    """idx int32 [T][k] (selection order), w fp32 [T][k]."""
    lg = np.ascontiguousarray(logits, dtype=np.float32)
    T, E = lg.shape
    idx = np.empty((T, k), dtype=np.int32)
    w = np.empty((T, k), dtype=np.float32)
    _check(lib().oracle_route_topk(T, E, k, n_groups, topk_groups, group_topn, lg, idx, w),
           "route_topk")
    return idx, w


def send_counts(idx: np.ndarray, E: int, R: int) -> dict:
    ix = np.ascontiguousarray(idx, dtype=np.int32)
    T, k = ix.shape
    out = {
        "C": np.empty((R, E), np.int32), "c": np.empty(E, np.int32),
        "S": np.empty((R, R), np.int32), "send_off": np.empty((R, R + 1), np.int64),
        "recv_off": np.empty((R, R + 1), np.int64), "recv_base": np.empty(R + 1, np.int64),
    }
    _check(lib().oracle_send_counts(T, E, k, R, ix, out["C"], out["c"], out["S"],
                                    out["send_off"], out["recv_off"], out["recv_base"]),
           "send_counts")
    return out


def dispatch_maps(idx: np.ndarray, E: int, R: int) -> dict:
    ix = np.ascontiguousarray(idx, dtype=np.int32)
    T, k = ix.shape
    send_pos = np.empty((T, k), np.int32)
    slot_of = np.empty((T, k), np.int32)
    src_row = np.full(T * k, -1, np.int32)
    _check(lib().oracle_dispatch_maps(T, E, k, R, ix, _ptr(send_pos), _ptr(slot_of),
                                      _ptr(src_row)), "dispatch_maps")
    return {"send_pos": send_pos, "slot_of": slot_of, "src_row": src_row}


def dispatch_rows(x: np.ndarray, idx: np.ndarray, maps: dict, E: int, W: int = 1,
                  wave: int = -1, want_send: bool = True, want_recv: bool = True,
                  fill: int = 0):
    """Permuted bf16 rows: (send, recv), each uint16 [T*k][H] or None.  Rows a
    wave does not touch keep ``fill``."""
    xx = np.ascontiguousarray(x, dtype=np.uint16)
    ix = np.ascontiguousarray(idx, dtype=np.int32)
    T, H = xx.shape
    k = ix.shape[1]
    send = np.full((T * k, H), fill, np.uint16) if want_send else None
    recv = np.full((T * k, H), fill, np.uint16) if want_recv else None
    _check(lib().oracle_dispatch_rows(T, H, E, k, W, wave, ix, xx, _ptr(maps["send_pos"]),
                                      _ptr(maps["slot_of"]), _ptr(send), _ptr(recv)),
           "dispatch_rows")
    return send, recv


def expert_standin(recv: np.ndarray, idx: np.ndarray, slot_of: np.ndarray,
                   scale: np.ndarray) -> np.ndarray:
    rv = np.ascontiguousarray(recv, dtype=np.uint16)
    ix = np.ascontiguousarray(idx, dtype=np.int32)
    so = np.ascontiguousarray(slot_of, dtype=np.int32)
    T, k = ix.shape
    H = rv.shape[1]
    out = np.zeros_like(rv)
    _check(lib().oracle_expert_standin(T, H, k, ix, so,
                                       np.ascontiguousarray(scale, dtype=np.float32), rv, out),
           "expert_standin")
    return out


def combine(out: np.ndarray, slot_of: np.ndarray, w: np.ndarray, t0: int = 0,
            t1: int | None = None) -> np.ndarray:
    """y uint16 [T][H]; rows outside [t0, t1) are left 0."""
    ov = np.ascontiguousarray(out, dtype=np.uint16)
    so = np.ascontiguousarray(slot_of, dtype=np.int32)
    ww = np.ascontiguousarray(w, dtype=np.float32)
    T, k = so.shape
    H = ov.shape[1]
    t1 = T if t1 is None else t1
    y = np.zeros((T, H), np.uint16)
    _check(lib().oracle_combine(T, H, k, t0, t1, ov, so, ww, y), "combine")
    return y


def imbalance_stats(c: np.ndarray, T: int, k: int, R: int) -> dict:
    cc = np.ascontiguousarray(c, dtype=np.int32)
    E = cc.shape[0]
    st = _Stats()
    rl = np.empty(R, np.int64)
    _check(lib().oracle_imbalance_stats(T, E, k, R, cc, ctypes.byref(st), _ptr(rl)),
           "imbalance_stats")
    return {"max_load": st.max_load, "min_load": st.min_load, "gini_num": st.gini_num,
            "gini_den": st.gini_den, "max_over_mean": st.max_over_mean,
            "hot_over_cold": st.hot_over_cold, "gini": st.gini, "rank_load": rl}


# ------------------------------------------------------------ capacity ----

def expert_capacity(T: int, E: int, k: int, f: float) -> int:
    """EC = ceil(k * f * T / E) (MoE survey section 1.1, eq. 3)."""
    ec = lib().oracle_expert_capacity(T, E, k, float(f))
    if ec < 0:
        raise ValueError("expert_capacity rejected its arguments")
    return int(ec)


def capacity_maps(idx: np.ndarray, E: int, EC: int) -> dict:
    """cap_slot int32 [T][k] (row e*EC + position, -1 if dropped) and
    dropped int32 [E]."""
    ix = np.ascontiguousarray(idx, dtype=np.int32)
    T, k = ix.shape
    cap_slot = np.empty((T, k), np.int32)
    dropped = np.empty(E, np.int32)
    _check(lib().oracle_capacity_maps(T, E, k, EC, ix, cap_slot, dropped), "capacity_maps")
    return {"cap_slot": cap_slot, "dropped": dropped}


def capacity_rows(x: np.ndarray, cap_slot: np.ndarray, E: int, EC: int) -> np.ndarray:
    xx = np.ascontiguousarray(x, dtype=np.uint16)
    cs = np.ascontiguousarray(cap_slot, dtype=np.int32)
    T, H = xx.shape
    rows = np.empty((E * EC, H), np.uint16)
    _check(lib().oracle_capacity_rows(T, H, E, cs.shape[1], EC, xx, cs, rows), "capacity_rows")
    return rows


def capacity_standin(rows: np.ndarray, scale: np.ndarray, E: int, EC: int) -> np.ndarray:
    rv = np.ascontiguousarray(rows, dtype=np.uint16)
    out = np.empty_like(rv)
    _check(lib().oracle_capacity_standin(rv.shape[1], E, EC,
                                         np.ascontiguousarray(scale, dtype=np.float32), rv, out),
           "capacity_standin")
    return out


def capacity_combine(out: np.ndarray, cap_slot: np.ndarray, w: np.ndarray) -> np.ndarray:
    ov = np.ascontiguousarray(out, dtype=np.uint16)
    cs = np.ascontiguousarray(cap_slot, dtype=np.int32)
    T, k = cs.shape
    H = ov.shape[1]
    y = np.empty((T, H), np.uint16)
    _check(lib().oracle_capacity_combine(T, H, k, ov, cs, np.ascontiguousarray(w, np.float32), y),
           "capacity_combine")
    return y


def forward_capacity(cfg, inputs: dict, f: float, with_rows: bool = True) -> dict:
    """Routing, counts and the capacity-factor dispatch / stand-in / combine."""
    idx, w = route_topk(inputs["logits"], cfg.k, cfg.n_groups, cfg.topk_groups,
                        cfg.group_topn)
    EC = expert_capacity(cfg.T, cfg.E, cfg.k, f)
    res = {"idx": idx, "w": w, "EC": EC, **send_counts(idx, cfg.E, cfg.R),
           **capacity_maps(idx, cfg.E, EC)}
    if with_rows:
        rows = capacity_rows(inputs["x"], res["cap_slot"], cfg.E, EC)
        out = capacity_standin(rows, inputs["scale"], cfg.E, EC)
        res.update(cap_rows=rows, cap_out=out, y=capacity_combine(out, res["cap_slot"], w))
    return res


# ------------------------------------------------ expert-major layout ----

def dispatch_maps_expert_major(idx: np.ndarray, E: int) -> dict:
    """slot_of / src_row of the expert-major recv layout and expert_off [E+1]."""
    ix = np.ascontiguousarray(idx, dtype=np.int32)
    T, k = ix.shape
    slot_of = np.empty((T, k), np.int32)
    src_row = np.full(T * k, -1, np.int32)
    off = np.empty(E + 1, np.int64)
    _check(lib().oracle_dispatch_maps_expert_major(T, E, k, ix, slot_of, _ptr(src_row), off),
           "dispatch_maps_expert_major")
    return {"slot_of": slot_of, "src_row": src_row, "expert_off": off}


def expert_gemm(rows: np.ndarray, counts: np.ndarray, weights: np.ndarray,
                sel: np.ndarray | None = None) -> np.ndarray:
    """A linear expert on expert-major rows (MoE survey section 1.1, step 3):
    out[r] = bf16_RN(rows[r] . weights[e(r)][n]) computed in fp64, where expert
    e owns rows [sum_{e'<e} c_e', sum_{e'<=e} c_e').  ``sel`` limits the
    computation to those row indices (returns their rows only)."""
    rv = np.ascontiguousarray(rows, dtype=np.uint16)
    cc = np.asarray(counts, dtype=np.int64)
    off = np.concatenate([[0], np.cumsum(cc)])
    W = bf16_to_f64(np.ascontiguousarray(weights, dtype=np.uint16))  # [E][N][H]
    idx = np.arange(rv.shape[0]) if sel is None else np.asarray(sel, dtype=np.int64)
    e_of = np.searchsorted(off, idx, side="right") - 1
    X = bf16_to_f64(rv[idx])
    out = np.empty((len(idx), W.shape[1]), np.float64)
    for e in np.unique(e_of):
        m = e_of == e
        out[m] = X[m] @ W[e].T
    return bf16_round(out)


def expert_ffn(rows: np.ndarray, counts: np.ndarray, w1: np.ndarray, w3: np.ndarray,
               w2: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """A gated FFN expert on expert-major rows (MoE survey section 1.1, step 3):
    hidden = bf16_RN(silu(x W1_e^T) * (x W3_e^T)) with silu(z) = z / (1 +
    exp(-z)), then out = bf16_RN(hidden W2_e^T), all in fp64.  w1, w3 [E][F][H],
    w2 [E][H][F].  Returns (hidden, out) as bf16 bits."""
    rv = np.ascontiguousarray(rows, dtype=np.uint16)
    cc = np.asarray(counts, dtype=np.int64)
    off = np.concatenate([[0], np.cumsum(cc)])
    X = bf16_to_f64(rv)
    W1, W3, W2 = (bf16_to_f64(np.ascontiguousarray(w, dtype=np.uint16)) for w in (w1, w3, w2))
    F, H = W1.shape[1], W2.shape[1]
    hidden = np.zeros((rv.shape[0], F), np.uint16)
    out = np.zeros((rv.shape[0], H), np.uint16)
    for e in range(len(cc)):
        lo, hi = off[e], off[e + 1]
        if hi == lo:
            continue
        g = X[lo:hi] @ W1[e].T
        u = X[lo:hi] @ W3[e].T
        hidden[lo:hi] = bf16_round(g / (1.0 + np.exp(-g)) * u)
        out[lo:hi] = bf16_round(bf16_to_f64(hidden[lo:hi]) @ W2[e].T)
    return hidden, out


# ------------------------------------------------- placement and alpha ----

def place_greedy(c: np.ndarray, R: int) -> dict:
    """placement int32 [E] (rank of each expert) and relabel int32 [E]."""
    cc = np.ascontiguousarray(c, dtype=np.int32)
    E = cc.shape[0]
    placement = np.empty(E, np.int32)
    relabel = np.empty(E, np.int32)
    _check(lib().oracle_place_greedy(E, R, cc, placement, relabel), "place_greedy")
    return {"placement": placement, "relabel": relabel}


def placement_gini(c: np.ndarray, placement: np.ndarray, R: int) -> dict:
    cc = np.ascontiguousarray(c, dtype=np.int32)
    pl = np.ascontiguousarray(placement, dtype=np.int32)
    num, den, g = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_double()
    _check(lib().oracle_placement_gini(cc.shape[0], R, cc, pl, ctypes.byref(num),
                                       ctypes.byref(den), ctypes.byref(g)), "placement_gini")
    return {"gini_num": num.value, "gini_den": den.value, "gini": g.value}


def dirichlet_alpha(c: np.ndarray) -> float:
    cc = np.ascontiguousarray(c, dtype=np.int32)
    a = ctypes.c_double()
    _check(lib().oracle_dirichlet_alpha(cc.shape[0], cc, ctypes.byref(a)), "dirichlet_alpha")
    return a.value


# --------------------------------------------------------- whole forward ----

def forward(cfg, inputs: dict, with_rows: bool = True) -> dict:
    """Every output of one dispatch/combine pass for workload ``cfg``."""
    idx, w = route_topk(inputs["logits"], cfg.k, cfg.n_groups, cfg.topk_groups,
                        cfg.group_topn)
    cnt = send_counts(idx, cfg.E, cfg.R)
    maps = dispatch_maps(idx, cfg.E, cfg.R)
    res = {"idx": idx, "w": w, **cnt, **maps,
           "stats": imbalance_stats(cnt["c"], cfg.T, cfg.k, cfg.R)}
    if with_rows:
        send, recv = dispatch_rows(inputs["x"], idx, maps, cfg.E)
        out = expert_standin(recv, idx, maps["slot_of"], inputs["scale"])
        res.update(send=send, recv=recv, out=out,
                   y=combine(out, maps["slot_of"], w))
    return res
