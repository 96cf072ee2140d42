"""Seeded synthetic workloads for MoE dispatch/combine.

This module only draws random inputs; it holds none of the routing, counting,
permutation or combine arithmetic.  Both the CUDA path and the CPU oracle
consume the arrays it returns, so the GPU never re-derives random numbers.

Workload families (shapes and logit distributions of the irregular-AllToAll
page, section "EP 不规则 a2a 的来源", and of the DODOCO summary, section
"方法论", which studies uniform "mock" routing against skewed routing):

* ``uniform``   logits ~ N(0,1) i.i.d. (near-uniform routing, the mock case)
* ``linear``    logits = z + gamma * pi(e) / (E-1): a linear log-popularity ramp
                over a random expert permutation pi; gamma sets the hot/cold ratio
* ``zipf``      logits = z - s * ln(pi(e) + 1): Zipf(s) popularity, random order
* ``dirichlet`` logits = z + ln(max(p_e, 1e-30)), p ~ Dirichlet(alpha * 1_E)

Random streams: ``numpy.random.SeedSequence(seed).spawn(4)`` gives independent
generators for x, z, the bias and the stand-in expert scales s_e.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np

__all__ = [
    "MoEConfig",
    "CONFIGS",
    "SWEEP",
    "make_inputs",
    "make_logits",
    "make_x",
    "make_scales",
    "bf16_bits_from_f32",
]


@dataclasses.dataclass(frozen=True)
class MoEConfig:
    """One workload: problem shape plus the logit family and seed."""

    name: str
    T: int  # tokens
    H: int  # hidden size (bf16 elements per row)
    E: int  # experts
    k: int  # experts per token
    R: int  # virtual expert-parallel ranks (partitions of one GPU's HBM)
    W: int = 1  # waves of the exchange
    n_groups: int = 1  # 1 = plain top-k; >1 = group-limited routing
    topk_groups: int = 0  # groups kept by group-limited routing
    group_topn: int = 0  # experts whose logits are summed into a group score
    bias: str = "uniform"  # uniform | linear | zipf | dirichlet
    bias_param: float = 0.0  # gamma (linear), s (zipf) or alpha (dirichlet)
    seed: int = 0

    def replace(self, **kw) -> "MoEConfig":
        return dataclasses.replace(self, **kw)

    @property
    def slots(self) -> int:
        return self.T * self.k

    def shape_tuple(self):
        return (self.T, self.H, self.E, self.k, self.R, self.W,
                self.n_groups, self.topk_groups, self.group_topn)


# Hot/cold ratio ~5x (the inference-side skew the Lina post reports for a
# 16-expert MoE, section "推理"): gamma for the linear log-popularity ramp was
# found by bisection on seed 0 so that max/min expert load of the routed
# tokens is 5 +- 0.25; a CPU test re-checks that property.
LINEAR_GAMMA_C2 = 0.874

CONFIGS = {
    "c1": MoEConfig("c1_T4096_H1024_E16_k2_R4_W1", T=4096, H=1024, E=16, k=2, R=4, W=1,
                    bias="uniform"),
    "c2": MoEConfig("c2_T16384_H2048_E64_k6_R8_W4", T=16384, H=2048, E=64, k=6, R=8, W=4,
                    bias="linear", bias_param=LINEAR_GAMMA_C2),
    "c3": MoEConfig("c3_T65536_H4096_E128_k8_R16_W8", T=65536, H=4096, E=128, k=8, R=16, W=8,
                    bias="zipf", bias_param=1.0),
    "c4": MoEConfig("c4_T32768_H7168_E256g8_k8_R32_W16", T=32768, H=7168, E=256, k=8, R=32,
                    W=16, n_groups=8, topk_groups=4, group_topn=2,
                    bias="dirichlet", bias_param=0.3),
}


def _sweep():
    out = []
    for T in (512, 2048, 8192, 32768, 131072, 262144):
        for alpha in (0.1, 1.0, 10.0):
            for W in (1, 4, 8, 16):
                out.append(MoEConfig(f"sweep_T{T}_a{alpha:g}_W{W}", T=T, H=4096, E=128, k=8,
                                     R=64, W=W, bias="dirichlet", bias_param=alpha))
    return out


SWEEP = _sweep()


def _streams(seed: int):
    ss = np.random.SeedSequence(seed)
    return [np.random.default_rng(c) for c in ss.spawn(4)]


def bf16_bits_from_f32(a: np.ndarray) -> np.ndarray:
    """Round fp32 samples to bf16 (nearest-even, via torch's CPU cast) and
    return the 16-bit patterns as uint16."""
    import torch

    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def make_bias(cfg: MoEConfig, rng: np.random.Generator) -> np.ndarray:
    E = cfg.E
    if cfg.bias == "uniform":
        return np.zeros(E, dtype=np.float32)
    if cfg.bias == "linear":
        pi = rng.permutation(E).astype(np.float64)
        return (cfg.bias_param * pi / max(E - 1, 1)).astype(np.float32)
    if cfg.bias == "zipf":
        pi = rng.permutation(E).astype(np.float64)
        return (-cfg.bias_param * np.log(pi + 1.0)).astype(np.float32)
    if cfg.bias == "dirichlet":
        p = rng.dirichlet(np.full(E, cfg.bias_param, dtype=np.float64))
        return np.log(np.maximum(p, 1e-30)).astype(np.float32)
    raise ValueError(f"unknown bias family {cfg.bias!r}")


def make_logits(cfg: MoEConfig, seed: Optional[int] = None) -> np.ndarray:
    """fp32 router logits [T][E] = fp32(z) + fp32(bias)."""
    seed = cfg.seed if seed is None else seed
    _, rz, rb, _ = _streams(seed)
    z = rz.standard_normal((cfg.T, cfg.E), dtype=np.float32)
    b = make_bias(cfg, rb)
    return (z + b[None, :]).astype(np.float32)


def make_x(cfg: MoEConfig, seed: Optional[int] = None, rows: Optional[int] = None) -> np.ndarray:
    """bf16 hidden states [T][H] (uint16 bit patterns) = bf16_RN(N(0,1) fp32).

    ``rows`` draws only the first ``rows`` tokens; they equal the first rows of
    the full draw (numpy fills the samples sequentially, chunks or not)."""
    seed = cfg.seed if seed is None else seed
    rx, _, _, _ = _streams(seed)
    T = cfg.T if rows is None else rows
    out = np.empty((T, cfg.H), dtype=np.uint16)
    step = max(1, (1 << 24) // cfg.H)  # ~64 MB of fp32 per chunk
    for t0 in range(0, T, step):
        t1 = min(T, t0 + step)
        out[t0:t1] = bf16_bits_from_f32(rx.standard_normal((t1 - t0, cfg.H), dtype=np.float32))
    return out


def make_scales(cfg: MoEConfig, seed: Optional[int] = None) -> np.ndarray:
    """Stand-in expert scales s_e ~ U(0.5, 1.5), fp32 [E]."""
    seed = cfg.seed if seed is None else seed
    _, _, _, rs = _streams(seed)
    return (rs.random(cfg.E, dtype=np.float32) + np.float32(0.5)).astype(np.float32)


def make_inputs(cfg: MoEConfig, seed: Optional[int] = None, with_x: bool = True) -> dict:
    """All inputs of one workload: logits, x (bf16 bits) and scales."""
    d = {"logits": make_logits(cfg, seed), "scale": make_scales(cfg, seed)}
    if with_x:
        d["x"] = make_x(cfg, seed)
    return d


def small_config(T=64, H=64, E=8, k=2, R=2, W=1, n_groups=1, topk_groups=0, group_topn=0,
                 bias="uniform", bias_param=0.0, seed=0) -> MoEConfig:
    return MoEConfig(f"small_T{T}_H{H}_E{E}_k{k}_R{R}_W{W}_g{n_groups}", T=T, H=H, E=E, k=k,
                     R=R, W=W, n_groups=n_groups, topk_groups=topk_groups,
                     group_topn=group_topn, bias=bias, bias_param=bias_param, seed=seed)


def reduced(cfg: MoEConfig, T: int) -> MoEConfig:
    """The same family at a smaller token count (T must keep T % R == 0)."""
    assert T % cfg.R == 0
    return cfg.replace(name=f"{cfg.name}_T{T}", T=T)

