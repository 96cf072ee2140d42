"""GPU parity at the size limits of the path.

1. Row addresses past 2^31 16-byte vectors: T = 589824 tokens of H = 4096
   (recv holds T*k = 4.7 M rows, 38.7 GB), so row * H/8 passes 2^31.
   Routing, counts, offsets and row maps are compared with the oracle in
   full; permuted rows and combine outputs on sampled tokens, the ones that
   own the last rows among them.
2. The slot limit: T*k = 2^31 - 65536 (T = 134213632, k = E = 16, H = 8).
   With k = E every token takes every expert, so the results have closed
   forms: idx[t] is the stable descending argsort of the logits, w their
   softmax, c_e = T, C[s][e] = T/R, the recv row of (t, e) is
   recv_base[d] + recv_off[d][s] + (e - d E/R) T/R + (t - s T/R), and
   y = bf16(sum_j w_j bf16(s_e x)).  All of it is checked at full size, in
   chunks, with library routines (torch sort, softmax, gathers) on the GPU.

The hidden states are a fixed bit pattern made on the device (finite
positive bf16 values), since the dispatch only copies bits; the oracle
computes the same pattern for its sampled tokens."""
import numpy as np
import pytest
import torch

import oracle
from combine_moe_route_17_b300 import MoEPipeline
from combine_moe_route_17_b300 import binding as B
from combine_moe_route_17_b300 import workloads as wl

from _parity import W_TOL, assert_counts, assert_maps, assert_routing, assert_y

pytestmark = pytest.mark.gpu

CHUNK = 1 << 22  # tokens per checking chunk


def _pattern(t0, t1, H, device):
    """x[t][h] bits = (t * 131 + h * 7) mod 251 + 16000: bf16 in [0.25, 1)."""
    t = torch.arange(t0, t1, device=device, dtype=torch.int64).view(-1, 1)
    h = torch.arange(H, device=device, dtype=torch.int64).view(1, -1)
    return ((t * 131 + h * 7) % 251 + 16000).to(torch.int16)


def _fill_x(p, T, H):
    for t0 in range(0, T, CHUNK):
        t1 = min(T, t0 + CHUNK)
        p.x.view(torch.int16)[t0:t1] = _pattern(t0, t1, H, p.x.device)


def _free(p):
    del p
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def test_row_addresses_past_2_to_the_31_vectors():
    cfg = wl.small_config(T=589824, H=4096, E=128, k=8, R=64, W=16, bias="dirichlet",
                          bias_param=1.0, seed=61)
    lg = wl.make_logits(cfg)
    scale = wl.make_scales(cfg)
    ref = oracle.forward(cfg, {"logits": lg}, with_rows=False)
    p = MoEPipeline(cfg, device="cuda")
    p.logits.copy_(torch.from_numpy(lg))
    p.scale.copy_(torch.from_numpy(scale))
    _fill_x(p, cfg.T, cfg.H)
    p.route_count()
    p.dispatch_waves()
    torch.cuda.synchronize()
    got = {key: v.cpu().numpy() for key, v in
           {"idx": p.idx, "w": p.w, "slot_of": p.slot_of, "src_row": p.src_row,
            **p.counts}.items()}
    assert B.get_device_error(p.ws) == 0
    assert_routing(got, ref)
    assert_counts(got, ref)
    assert_maps(got, ref)
    assert int(got["slot_of"].max()) * (cfg.H // 8) >= 1 << 31  # the case is what it says
    # sampled tokens: random ones and the owners of the last 64 rows
    rng = np.random.default_rng(62)
    last = got["src_row"][-64:]
    toks = np.unique(np.concatenate([rng.integers(0, cfg.T, 256), last, [0, cfg.T - 1]]))
    slots = torch.from_numpy(got["slot_of"][toks].reshape(-1).astype(np.int64)).cuda()
    rows = p.recv.view(torch.int16)[slots].cpu().numpy().view(np.uint16)
    x_s = np.concatenate([_pattern(int(t), int(t) + 1, cfg.H, "cpu").numpy().view(np.uint16)
                          for t in toks])
    assert np.array_equal(rows, np.repeat(x_s, cfg.k, axis=0))
    p.expert()
    p.combine()
    torch.cuda.synchronize()
    assert B.get_device_error(p.ws) == 0
    y = p.y.view(torch.int16)[torch.from_numpy(toks).cuda()].cpu().numpy().view(np.uint16)
    compact = np.arange(len(toks) * cfg.k, dtype=np.int32).reshape(len(toks), cfg.k)
    out = oracle.expert_standin(np.repeat(x_s, cfg.k, axis=0), ref["idx"][toks], compact, scale)
    assert_y(y, oracle.combine(out, compact, ref["w"][toks]))
    _free(p)


def test_slot_limit_closed_forms():
    R, E, k, H = 4, 16, 16, 8
    T = (1 << 27) - (1 << 12)
    assert T * k < 1 << 31 and T * k >= (1 << 31) - (1 << 16)
    cfg = wl.small_config(T=T, H=H, E=E, k=k, R=R, W=2, seed=63)
    dev = torch.device("cuda")
    p = MoEPipeline(cfg, device=dev)
    gen = torch.Generator(device=dev)
    gen.manual_seed(63)
    for t0 in range(0, T, CHUNK):
        t1 = min(T, t0 + CHUNK)
        p.logits[t0:t1] = torch.randn((t1 - t0, E), generator=gen, device=dev)
    p.scale.copy_(torch.from_numpy(wl.make_scales(cfg)))
    _fill_x(p, T, H)
    p.route_count()
    p.dispatch_waves()
    p.imbalance()
    torch.cuda.synchronize()
    assert B.get_device_error(p.ws) == 0

    Tr, Er = T // R, E // R
    c = p.counts
    assert (c["c"] == T).all() and (c["C"] == Tr).all() and (c["S"] == Tr * Er).all()
    d_ar = torch.arange(R + 1, device=dev, dtype=torch.int64)
    assert torch.equal(c["send_off"], (d_ar * Tr * Er).expand(R, R + 1))
    assert torch.equal(c["recv_off"], (d_ar * Tr * Er).expand(R, R + 1))
    assert torch.equal(c["recv_base"], d_ar * T * Er)
    st = p.stats_dict()
    assert st["max_load"] == T and st["min_load"] == T and st["gini"] == 0.0
    assert st["max_over_mean"] == 1.0 and st["hot_over_cold"] == 1.0

    recv64 = p.recv.view(torch.int64).view(T * k, 2)
    x64 = p.x.view(torch.int64).view(T, 2)
    for t0 in range(0, T, CHUNK):
        t1 = min(T, t0 + CHUNK)
        lg = p.logits[t0:t1]
        want_idx = torch.sort(lg, dim=1, descending=True, stable=True).indices
        idx = p.idx[t0:t1].long()
        assert torch.equal(idx, want_idx), f"idx of tokens [{t0}, {t1})"
        lsel = torch.gather(lg, 1, idx).double()
        want_w = torch.softmax(lsel, dim=1)
        assert (p.w[t0:t1].double() - want_w).abs().max().item() <= W_TOL
        t = torch.arange(t0, t1, device=dev, dtype=torch.int64).view(-1, 1)
        s = t // Tr
        d = idx // Er
        want_slot = d * T * Er + s * Tr * Er + (idx - d * Er) * Tr + (t - s * Tr)
        slot = p.slot_of[t0:t1].long()
        assert torch.equal(slot, want_slot), f"slot_of of tokens [{t0}, {t1})"
        flat = slot.view(-1)
        assert torch.equal(p.src_row[flat].long().view(-1, k), t.expand(-1, k))
        assert torch.equal(recv64[flat].view(-1, k, 2), x64[t0:t1].view(-1, 1, 2).expand(-1, k, 2))
    del recv64, x64

    p.expert()
    p.combine()
    torch.cuda.synchronize()
    assert B.get_device_error(p.ws) == 0
    xb = p.x.view(torch.bfloat16)
    for t0 in range(0, T, CHUNK):
        t1 = min(T, t0 + CHUNK)
        idx = p.idx[t0:t1].long()
        sc = p.scale[idx]  # [n][k]
        out = (sc.unsqueeze(2) * xb[t0:t1].float().unsqueeze(1)).to(torch.bfloat16).double()
        want = (p.w[t0:t1].double().unsqueeze(2) * out).sum(dim=1)
        y = p.y[t0:t1].double()
        assert ((y - want).abs() <= 1e-2 * want.abs()).all(), f"y of tokens [{t0}, {t1})"
    _free(p)
