"""The tensor-core experts at the workloads' full sizes, in the launch
configuration bench.py --expert-gemm times: route, counts, the expert-major
dispatch waves, then moe_expert_gemm (a bf16 [H][H] weight per expert) and
moe_expert_ffn (F = 2048), with seeded N(0, 1/fan-in) weights drawn on the
device.  Sampled rows of a few experts (the busiest, a small one, the last
one with rows, a random one; their first, last and random rows) against the
oracle's fp64 products, with the bounds of the small-size tests."""
import numpy as np
import pytest
import torch

import oracle
from combine_moe_route_17_b300 import MoEPipeline
from combine_moe_route_17_b300 import binding as B
from combine_moe_route_17_b300 import workloads as wl

pytestmark = pytest.mark.gpu

F = 2048


def _u16(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def _layer(cfg):
    inp = wl.make_inputs(cfg)
    p = MoEPipeline(cfg, device="cuda", expert_major=True)
    p.load_inputs(torch.from_numpy(inp["logits"]), torch.from_numpy(inp["x"].view(np.int16)),
                  torch.from_numpy(inp["scale"]))
    p.route_count()
    p.dispatch_waves()
    torch.cuda.synchronize()
    assert B.get_device_error(p.ws) == 0
    return p


def _sample(counts, rng):
    """(expert, row within the expert) pairs of a few experts."""
    c = np.asarray(counts)
    busy = int(np.argmax(c))
    nz = np.flatnonzero(c)
    small = int(nz[np.argmin(c[nz])])
    last = int(nz[-1])
    pick = []
    for e in sorted({busy, small, last, int(rng.choice(nz))}):
        n = int(c[e])
        rows = np.unique(np.concatenate([[0, n - 1], rng.integers(0, n, size=min(n, 24))]))
        pick += [(e, int(r)) for r in rows]
    return pick


def _bound_ok(got, ref, X, Wt, K):
    absdot = np.abs(X) @ np.abs(Wt).T
    return np.abs(got - ref) <= 2.0 ** -7 * np.abs(ref) + K * 2.0 ** -22 * absdot


@pytest.mark.parametrize("name", ["c2", "c4"])
def test_linear_expert_at_full_size(name):
    cfg = wl.CONFIGS[name]
    p = _layer(cfg)
    gen = torch.Generator(device="cuda")
    gen.manual_seed(cfg.seed + 17)
    Wt = (torch.randn((cfg.E, cfg.H, cfg.H), generator=gen, device="cuda", dtype=torch.float32)
          / float(np.sqrt(cfg.H))).to(torch.bfloat16)
    out = torch.empty_like(p.recv)
    B.expert_gemm(p.shape, p.recv, Wt, p.counts["c"], out, p.ws)
    torch.cuda.synchronize()
    assert B.get_device_error(p.ws) == 0
    counts = p.counts["c"].cpu().numpy()
    off = np.concatenate([[0], np.cumsum(counts)])
    pick = _sample(counts, np.random.default_rng(71))
    idx = torch.tensor([off[e] + r for e, r in pick], dtype=torch.int64, device="cuda")
    x = _u16(p.recv[idx])
    got = oracle.bf16_to_f64(_u16(out[idx]))
    experts = np.array([e for e, _ in pick])
    for e in np.unique(experts):
        sel = np.flatnonzero(experts == e)
        W_e = _u16(Wt[int(e)])
        ref = oracle.bf16_to_f64(oracle.expert_gemm(x[sel], [len(sel)], W_e[None]))
        ok = _bound_ok(got[sel], ref, oracle.bf16_to_f64(x[sel]), oracle.bf16_to_f64(W_e), cfg.H)
        assert ok.all(), f"expert {e}: {int((~ok).sum())} outputs outside the bound"


@pytest.mark.parametrize("name", ["c2", "c4"])
def test_ffn_expert_at_full_size(name):
    cfg = wl.CONFIGS[name]
    p = _layer(cfg)
    gen = torch.Generator(device="cuda")
    gen.manual_seed(cfg.seed + 17)
    w13 = (torch.randn((cfg.E, 2 * F, cfg.H), generator=gen, device="cuda")
           / float(np.sqrt(cfg.H))).to(torch.bfloat16)
    w2 = (torch.randn((cfg.E, cfg.H, F), generator=gen, device="cuda")
          / float(np.sqrt(F))).to(torch.bfloat16)
    hidden = torch.empty((cfg.T * cfg.k, F), dtype=torch.bfloat16, device="cuda")
    out = torch.empty_like(p.recv)
    B.expert_ffn(p.shape, p.recv, w13, w2, p.counts["c"], hidden, out, p.ws)
    torch.cuda.synchronize()
    assert B.get_device_error(p.ws) == 0
    counts = p.counts["c"].cpu().numpy()
    off = np.concatenate([[0], np.cumsum(counts)])
    pick = _sample(counts, np.random.default_rng(72))
    idx = torch.tensor([off[e] + r for e, r in pick], dtype=torch.int64, device="cuda")
    x = oracle.bf16_to_f64(_u16(p.recv[idx]))
    h_gpu = _u16(hidden[idx])
    o_gpu = oracle.bf16_to_f64(_u16(out[idx]))
    H = cfg.H
    experts = np.array([e for e, _ in pick])
    for e in np.unique(experts):
        sel = np.flatnonzero(experts == e)
        blocks = _u16(w13[int(e)]).reshape(F // 128, 2, 128, H)
        W1 = oracle.bf16_to_f64(blocks[:, 0].reshape(F, H))
        W3 = oracle.bf16_to_f64(blocks[:, 1].reshape(F, H))
        W2 = _u16(w2[int(e)])
        xs = x[sel]
        g, u = xs @ W1.T, xs @ W3.T
        silu = g / (1.0 + np.exp(-g))
        ref_h = oracle.bf16_to_f64(oracle.bf16_round(silu * u))
        dg = H * 2.0 ** -22 * (np.abs(xs) @ np.abs(W1).T)
        du = H * 2.0 ** -22 * (np.abs(xs) @ np.abs(W3).T)
        bound = (2.0 ** -7 + 2.0 ** -18) * np.abs(ref_h) + 2.0 * (1.1 * np.abs(u) * dg +
                                                                (np.abs(silu) + 1.1 * dg) * du)
        h = oracle.bf16_to_f64(h_gpu[sel])
        assert (np.abs(h - ref_h) <= bound).all(), f"expert {e}: intermediate outside the bound"
        ref_o = oracle.bf16_to_f64(oracle.expert_gemm(h_gpu[sel], [len(sel)], W2[None]))
        ok = _bound_ok(o_gpu[sel], ref_o, h, oracle.bf16_to_f64(W2), F)
        assert ok.all(), f"expert {e}: {int((~ok).sum())} outputs outside the bound"
