"""GPU parity of the gated FFN expert (moe_expert_ffn: two persistent
tensor-core launches; the first pairs gate and up columns in one 256-column
TMEM accumulator and applies silu(g) * u in its epilogue) against the oracle.

Tolerance of the intermediate, from the arithmetic.  The gate g = x W1^T and
the up value u = x W3^T are fp32 sums of exact bf16 products, each off by at
most dg = K 2^-22 sum|x w1| (du likewise).  |silu'| < 1.1, so the fp32
h = silu(g) u is off by at most 1.1 |u| dg + |silu(g)| du plus a few fp32
roundings of silu and the product (2^-18 |h| covers them); both sides then
round to bf16, up to a full ulp (2^-7 relative) apart.  The bound doubles the
absolute terms for the second-order products.  The down projection is checked
on the GPU's own intermediate with the linear expert's bound."""
import numpy as np
import pytest
import torch

import oracle
from combine_moe_route_17_b300 import MoEPipeline
from combine_moe_route_17_b300 import binding as B
from combine_moe_route_17_b300 import workloads as wl

from _parity import bf16_rows_to_u16

pytestmark = pytest.mark.gpu


def _bf(a):
    return oracle.bf16_round(np.asarray(a, dtype=np.float64))


def _to_dev(u16):
    return torch.from_numpy(np.ascontiguousarray(u16).view(np.int16)).cuda().view(torch.bfloat16)


def _weights(E, H, F, seed):
    rng = np.random.default_rng(seed)
    w1 = _bf(rng.standard_normal((E, F, H)) / np.sqrt(H))
    w3 = _bf(rng.standard_normal((E, F, H)) / np.sqrt(H))
    w2 = _bf(rng.standard_normal((E, H, F)) / np.sqrt(F))
    return w1, w3, w2


def _ffn_dev(shape, rows_d, w1, w3, w2, counts_d, ws):
    n = shape.T * shape.k
    F = w1.shape[1]
    w13 = B.pack_gated_weights(_to_dev(w1), _to_dev(w3))
    hidden = torch.full((n, F), float("nan"), dtype=torch.bfloat16, device="cuda")
    out = torch.full((n, shape.H), float("nan"), dtype=torch.bfloat16, device="cuda")
    B.expert_ffn(shape, rows_d, w13, _to_dev(w2), counts_d, hidden, out, ws)
    torch.cuda.synchronize()
    assert B.get_device_error(ws) == 0
    return bf16_rows_to_u16(hidden), bf16_rows_to_u16(out)


def _row_expert(counts, n):
    off = np.concatenate([[0], np.cumsum(counts)])
    return np.searchsorted(off, np.arange(n), side="right") - 1


def _assert_hidden(got, rows, counts, w1, w3):
    n, K = rows.shape
    ref = oracle.bf16_to_f64(oracle.expert_ffn(rows, counts, w1, w3,
                                               np.zeros((len(counts), K, w1.shape[1]),
                                                        np.uint16))[0])
    X = oracle.bf16_to_f64(rows)
    W1, W3 = oracle.bf16_to_f64(w1), oracle.bf16_to_f64(w3)
    e_of = _row_expert(counts, n)
    g = np.stack([W1[e_of[i]] @ X[i] for i in range(n)])
    u = np.stack([W3[e_of[i]] @ X[i] for i in range(n)])
    dg = K * 2.0 ** -22 * np.stack([np.abs(W1[e_of[i]]) @ np.abs(X[i]) for i in range(n)])
    du = K * 2.0 ** -22 * np.stack([np.abs(W3[e_of[i]]) @ np.abs(X[i]) for i in range(n)])
    silu = g / (1.0 + np.exp(-g))
    bound = (2.0 ** -7 + 2.0 ** -18) * np.abs(ref) + 2.0 * (1.1 * np.abs(u) * dg +
                                                          (np.abs(silu) + 1.1 * dg) * du)
    h = oracle.bf16_to_f64(got)
    bad = ~(np.abs(h - ref) <= bound)
    assert not bad.any(), f"{int(bad.sum())} of {bad.size} intermediate values outside the bound"


def _assert_down(got_out, got_hidden, counts, w2):
    ref = oracle.bf16_to_f64(oracle.expert_gemm(got_hidden, counts, w2))
    Hd = np.abs(oracle.bf16_to_f64(got_hidden))
    W2 = np.abs(oracle.bf16_to_f64(w2))
    e_of = _row_expert(counts, got_hidden.shape[0])
    absdot = np.stack([W2[e_of[i]] @ Hd[i] for i in range(len(e_of))])
    K = got_hidden.shape[1]
    g = oracle.bf16_to_f64(got_out)
    bad = ~(np.abs(g - ref) <= 2.0 ** -7 * np.abs(ref) + K * 2.0 ** -22 * absdot)
    assert not bad.any(), f"{int(bad.sum())} of {bad.size} outputs outside the bound"


def _case(counts, H, F, seed):
    rng = np.random.default_rng(seed)
    E, n = len(counts), int(sum(counts))
    rows = _bf(rng.standard_normal((n, H)))
    w1, w3, w2 = _weights(E, H, F, seed + 100)
    shape = B.Shape(n, H, E, 1, 1, 1, 1, 0, 0)
    ws = B.new_workspace(shape, "cuda")
    hid, out = _ffn_dev(shape, _to_dev(rows), w1, w3, w2,
                        torch.tensor(counts, dtype=torch.int32, device="cuda"), ws)
    return rows, (w1, w3, w2), hid, out


@pytest.mark.parametrize("counts,H,F", [([128], 128, 128),
                                        ([0, 130, 1, 300, 77], 256, 384),
                                        ([500, 3, 129], 512, 256),
                                        ([64] * 8, 1024, 512)])
def test_ffn_matches_oracle(counts, H, F):
    rows, (w1, w3, w2), hid, out = _case(counts, H, F, seed=len(counts) + H)
    _assert_hidden(hid, rows, counts, w1, w3)
    _assert_down(out, hid, counts, w2)


def test_gate_and_up_pairing():
    """One-hot weights pick distinct columns: g = 8 x[f] (so silu(g) ~ g) and
    u = x[(f + 1 + e) mod H], with x in [1, 5).  Swapping the gate and up
    halves (silu(u) g ~ sigmoid(u) g u), pairing columns of other 128-row
    blocks, or taking another expert's weights all move h far outside the
    bound."""
    counts, H, F = [130, 126], 256, 256
    rng = np.random.default_rng(9)
    rows = _bf(1.0 + 4.0 * rng.random((sum(counts), H)))
    w1 = np.zeros((2, F, H), np.uint16)
    w3 = np.zeros((2, F, H), np.uint16)
    for e in range(2):
        for f in range(F):
            w1[e, f] = _bf(np.eye(1, H, f)[0] * 8.0)
            w3[e, f] = _bf(np.eye(1, H, (f + 1 + e) % H)[0])
    w2 = np.zeros((2, H, F), np.uint16)
    shape = B.Shape(sum(counts), H, 2, 1, 1, 1, 1, 0, 0)
    ws = B.new_workspace(shape, "cuda")
    hid, _ = _ffn_dev(shape, _to_dev(rows), w1, w3, w2,
                      torch.tensor(counts, dtype=torch.int32, device="cuda"), ws)
    _assert_hidden(hid, rows, counts, w1, w3)


def test_ffn_layer():
    """route -> counts -> expert-major dispatch -> gated FFN expert -> combine."""
    cfg = wl.small_config(T=1024, H=256, E=8, k=2, R=4, W=1, bias="zipf", bias_param=1.0,
                          seed=7)
    F = 384
    inp = wl.make_inputs(cfg)
    ref = oracle.forward(cfg, inp, with_rows=False)
    em = oracle.dispatch_maps_expert_major(ref["idx"], cfg.E)
    w1, w3, w2 = _weights(cfg.E, cfg.H, F, 8)
    p = MoEPipeline(cfg, device="cuda", expert_major=True)
    p.load_inputs(torch.from_numpy(inp["logits"]), torch.from_numpy(inp["x"].view(np.int16)),
                  torch.from_numpy(inp["scale"]))
    p.route()
    p.count()
    p.dispatch_waves()
    hid, out = _ffn_dev(p.shape, p.recv, w1, w3, w2, p.counts["c"], p.ws)
    recv = np.zeros((cfg.T * cfg.k, cfg.H), np.uint16)
    recv[em["slot_of"].ravel()] = np.repeat(inp["x"], cfg.k, axis=0)
    _assert_hidden(hid, recv, ref["c"], w1, w3)
    _assert_down(out, hid, ref["c"], w2)


def test_ffn_rejects_unsupported_shapes():
    shape = B.Shape(128, 128, 1, 1, 1, 1, 1, 0, 0)
    x = torch.zeros((128, 128), dtype=torch.bfloat16, device="cuda")
    w13 = torch.zeros((1, 192, 128), dtype=torch.bfloat16, device="cuda")
    w2 = torch.zeros((1, 128, 96), dtype=torch.bfloat16, device="cuda")  # F = 96
    hid = torch.zeros((128, 96), dtype=torch.bfloat16, device="cuda")
    out = torch.zeros((128, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(B.MoEError) as e:
        B.expert_ffn(shape, x, w13, w2, torch.tensor([128], dtype=torch.int32, device="cuda"),
                     hid, out)
    assert e.value.status == B.MOE_ERR_UNSUPPORTED


def _wave_rows(counts, W):
    off = np.concatenate([[0], np.cumsum(counts)])
    Ew = len(counts) // W
    return [(int(off[w * Ew]), int(off[(w + 1) * Ew])) for w in range(W)]


@pytest.mark.parametrize("kind", ["linear", "ffn"])
def test_wave_calls_reproduce_the_all_expert_call(kind):
    """moe_expert_gemm_wave / moe_expert_ffn_wave for w = 0..W-1: after wave w
    the rows of waves <= w equal the all-expert call's bit for bit, and the
    rows of later waves are untouched."""
    counts, H, F, W = [130, 0, 257, 64, 1, 300, 128, 77], 256, 256, 4
    rng = np.random.default_rng(41)
    E, n = len(counts), sum(counts)
    rows = _to_dev(_bf(rng.standard_normal((n, H))))
    shape = B.Shape(n, H, E, 1, 1, W, 1, 0, 0)
    ws = B.new_workspace(shape, "cuda")
    cnt = torch.tensor(counts, dtype=torch.int32, device="cuda")
    if kind == "linear":
        Wt = _to_dev(_bf(rng.standard_normal((E, H, H)) / np.sqrt(H)))

        def run(out, wave):
            B.expert_gemm(shape, rows, Wt, cnt, out, ws, wave=wave)
    else:
        w1, w3, w2 = _weights(E, H, F, 42)
        w13 = B.pack_gated_weights(_to_dev(w1), _to_dev(w3))
        w2d = _to_dev(w2)
        hidden = torch.empty((n, F), dtype=torch.bfloat16, device="cuda")

        def run(out, wave):
            B.expert_ffn(shape, rows, w13, w2d, cnt, hidden, out, ws, wave=wave)

    full = torch.empty((n, H), dtype=torch.bfloat16, device="cuda")
    run(full, -1)
    want = bf16_rows_to_u16(full)
    out = torch.full((n, H), float("nan"), dtype=torch.bfloat16, device="cuda")
    spans = _wave_rows(counts, W)
    for w in range(W):
        run(out, w)
        torch.cuda.synchronize()
        got = bf16_rows_to_u16(out)
        hi = spans[w][1]
        assert np.array_equal(got[:hi], want[:hi]), f"wave {w}"
        assert (got[hi:] == 0x7FC0).all(), f"wave {w} wrote rows of a later wave"
    assert B.get_device_error(ws) == 0
    with pytest.raises(B.MoEError) as e:
        run(out, W)
    assert e.value.status == B.MOE_ERR_INVALID_ARG


def test_pipelined_ffn_layer_equals_the_sequential_layer():
    """route/counts, then per wave dispatch(w) -> FFN experts(w) ->
    combine of the tokens whose last wave is w on three streams: y equals
    the sequential layer's bit for bit, and the oracle's combine of the
    GPU's expert rows within the combine tolerance."""
    cfg = wl.small_config(T=2048, H=256, E=16, k=4, R=4, W=4, bias="zipf", bias_param=1.0,
                          seed=43)
    F = 256
    inp = wl.make_inputs(cfg)
    w1, w3, w2 = _weights(cfg.E, cfg.H, F, 44)
    ys = []
    for pipelined in (False, True):
        p = MoEPipeline(cfg, device="cuda", expert_major=True)
        p.load_inputs(torch.from_numpy(inp["logits"]), torch.from_numpy(inp["x"].view(np.int16)),
                      torch.from_numpy(inp["scale"]))
        p.set_ffn(B.pack_gated_weights(_to_dev(w1), _to_dev(w3)), _to_dev(w2))
        if pipelined:
            streams = [torch.cuda.Stream() for _ in range(3)]
            streams[0].wait_stream(torch.cuda.current_stream())
            p.step_pipelined(streams)
            torch.cuda.current_stream().wait_stream(streams[0])
        else:
            p.route_count()
            p.dispatch_waves()
            p.expert()
            p.combine()
        torch.cuda.synchronize()
        assert B.get_device_error(p.ws) == 0
        ys.append(p.y.view(torch.int16).cpu().numpy().view(np.uint16))
        out = bf16_rows_to_u16(p.out)
    assert np.array_equal(ys[0], ys[1])
    ref = oracle.forward(cfg, inp, with_rows=False)
    em = oracle.dispatch_maps_expert_major(ref["idx"], cfg.E)
    y_ref = oracle.bf16_to_f64(oracle.combine(out, em["slot_of"], ref["w"]))
    y = oracle.bf16_to_f64(ys[1])
    o = np.abs(oracle.bf16_to_f64(out))[em["slot_of"]]
    absdot = np.einsum("tk,tkh->th", np.abs(ref["w"].astype(np.float64)), o)
    assert np.all(np.abs(y - y_ref) <= 2.0 ** -7 * np.abs(y_ref) + cfg.k * 2.0 ** -22 * absdot)
