"""GPU parity of the tensor-core linear expert (moe_expert_gemm: TMA,
tcgen05.mma into TMEM, tcgen05.ld) on expert-major rows against the oracle.

Tolerance, from the arithmetic: products of bf16 are exact in fp32; the fp32
sum of K of them, in the tensor core's order, is off by at most
K * 2^-23 * sum|a b| (a generous bound); each side then rounds once to bf16
(unit roundoff 2^-8), and the two roundings can land a full bf16 ulp apart,
2^-7 relative; so |gpu - oracle| <= 2^-7 |oracle| + K * 2^-22 * sum|a b|.
Identity weights make every sum exact: there the result is bit-exact."""
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


def _gemm(counts, H, N, seed=0, identity=False, sel=None):
    rng = np.random.default_rng(seed)
    E = len(counts)
    n = int(sum(counts))
    rows = _bf(rng.standard_normal((n, H)))
    if identity:
        W = np.stack([_bf(np.eye(N, H))] * E)
    else:
        W = _bf(rng.standard_normal((E, N, H)) / np.sqrt(H))
    shape = B.Shape(max(n, 1), H, E, 1, 1, 1, 1, 0, 0)
    out = torch.full((max(n, 1), N), float("nan"), dtype=torch.bfloat16, device="cuda")
    rows_d = torch.zeros((max(n, 1), H), dtype=torch.bfloat16, device="cuda")
    rows_d[:n] = _to_dev(rows)
    ws = B.new_workspace(shape, "cuda")
    B.expert_gemm(shape, rows_d, _to_dev(W), torch.tensor(counts, dtype=torch.int32,
                                                           device="cuda"), out, ws)
    torch.cuda.synchronize()
    assert B.get_device_error(ws) == 0
    got = bf16_rows_to_u16(out)[:n]
    return rows, W, got


def _assert_within_bound(got, rows, W, counts, sel=None):
    idx = np.arange(rows.shape[0]) if sel is None else np.asarray(sel)
    ref = oracle.bf16_to_f64(oracle.expert_gemm(rows, counts, W, sel=idx))
    off = np.concatenate([[0], np.cumsum(counts)])
    e_of = np.searchsorted(off, idx, side="right") - 1
    X = np.abs(oracle.bf16_to_f64(rows[idx]))
    Wa = np.abs(oracle.bf16_to_f64(W))
    absdot = np.stack([X[i] @ Wa[e_of[i]].T for i in range(len(idx))])
    K = rows.shape[1]
    g = oracle.bf16_to_f64(got[idx])
    bad = np.abs(g - ref) > 2.0 ** -7 * np.abs(ref) + K * 2.0 ** -22 * absdot
    assert not bad.any(), f"{int(bad.sum())} of {bad.size} outside the bound"


def test_one_tile_one_k_block():
    rows, W, got = _gemm([128], 64, 128, seed=1)
    _assert_within_bound(got, rows, W, [128])


def test_identity_weights_are_bit_exact():
    counts = [130, 0, 7, 256]
    rows, W, got = _gemm(counts, 256, 256, identity=True, seed=2)
    assert np.array_equal(got, rows)


@pytest.mark.parametrize("counts,H,N", [([0, 130, 1, 300, 77], 256, 256),
                                        ([500, 3, 129], 512, 384),
                                        ([64] * 16, 1024, 128)])
def test_ragged_experts(counts, H, N):
    rows, W, got = _gemm(counts, H, N, seed=len(counts))
    _assert_within_bound(got, rows, W, counts)


def test_layer_with_the_gemm_expert():
    """route -> counts -> expert-major dispatch -> tensor-core expert -> combine."""
    cfg = wl.small_config(T=2048, H=256, E=16, k=4, R=4, W=2, bias="zipf", bias_param=1.0,
                          seed=5)
    inp = wl.make_inputs(cfg)
    ref = oracle.forward(cfg, inp, with_rows=False)
    em = oracle.dispatch_maps_expert_major(ref["idx"], cfg.E)
    rng = np.random.default_rng(6)
    W = _bf(rng.standard_normal((cfg.E, cfg.H, cfg.H)) / np.sqrt(cfg.H))
    p = MoEPipeline(cfg, device="cuda", expert_major=True)
    p.load_inputs(torch.from_numpy(inp["logits"]), torch.from_numpy(inp["x"].view(np.int16)),
                  torch.from_numpy(inp["scale"]))
    out = torch.empty_like(p.recv)
    p.route()
    p.count()
    p.dispatch_waves()
    B.expert_gemm(p.shape, p.recv, _to_dev(W), p.counts["c"], out, p.ws)
    B.combine(p.shape, out, p.slot_of, p.w, p.y, p.ws)
    torch.cuda.synchronize()
    assert B.get_device_error(p.ws) == 0
    recv = np.zeros((cfg.T * cfg.k, cfg.H), np.uint16)
    recv[em["slot_of"].ravel()] = np.repeat(inp["x"], cfg.k, axis=0)
    got_out = bf16_rows_to_u16(out)
    _assert_within_bound(got_out, recv, W, ref["c"])
    # the combine of the GPU expert rows, against the oracle's combine of them
    y_ref = oracle.bf16_to_f64(oracle.combine(got_out, em["slot_of"], ref["w"]))
    y = oracle.bf16_to_f64(p.y.view(torch.int16).cpu().numpy().view(np.uint16))
    o = np.abs(oracle.bf16_to_f64(got_out))[em["slot_of"]]  # [T][k][H]
    absdot = np.einsum("tk,tkh->th", np.abs(ref["w"].astype(np.float64)), o)
    assert np.all(np.abs(y - y_ref) <= 2.0 ** -7 * np.abs(y_ref) + cfg.k * 2.0 ** -22 * absdot)


def test_gemm_rejects_unsupported_shapes():
    shape = B.Shape(128, 96, 1, 1, 1, 1, 1, 0, 0)  # H % 64 != 0
    x = torch.zeros((128, 96), dtype=torch.bfloat16, device="cuda")
    W = torch.zeros((1, 128, 96), dtype=torch.bfloat16, device="cuda")
    out = torch.zeros((128, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(B.MoEError) as e:
        B.expert_gemm(shape, x, W, torch.tensor([128], dtype=torch.int32, device="cuda"), out)
    assert e.value.status == B.MOE_ERR_UNSUPPORTED
