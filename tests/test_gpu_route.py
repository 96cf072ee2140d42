"""GPU parity of moe_route_topk alone, over every launch geometry the library
picks from (E, n_groups, group_topn) and both logits load paths.

The sub-warp kernel gives each token G lanes of EPL contiguous experts, so
the shapes below cover every (EPL, G) pair, group-limited routing whose
groups are one lane, several lanes, or many lanes, group sums of the top 1
to 4 logits, and the shapes that go to the one-warp-per-token kernel (groups
that split a lane, group_topn > 4).  Each shape runs on N(0,1) logits and on
tie-heavy integer logits with signed zeros, against the oracle: indices
bit-exact, weights within 1e-6."""
import numpy as np
import pytest
import torch

import oracle
from combine_moe_route_17_b300 import binding as B

from _parity import W_TOL

pytestmark = pytest.mark.gpu

# (E, k, n_groups, topk_groups, group_topn)
SHAPES = [
    (1, 1, 1, 0, 0), (3, 2, 1, 0, 0), (6, 3, 1, 0, 0), (8, 8, 1, 0, 0), (16, 2, 1, 0, 0),
    (24, 5, 1, 0, 0), (32, 4, 1, 0, 0), (64, 6, 1, 0, 0), (100, 7, 1, 0, 0),
    (128, 8, 1, 0, 0), (200, 16, 1, 0, 0), (256, 8, 1, 0, 0), (256, 16, 1, 0, 0),
    # groups of whole lanes (EPL = 4 up to E = 128, 8 above)
    (256, 8, 8, 4, 2), (256, 8, 8, 4, 1), (256, 8, 8, 3, 3), (256, 8, 4, 2, 4),
    (256, 8, 2, 1, 2), (256, 8, 32, 5, 2), (128, 8, 4, 2, 2), (128, 6, 16, 3, 4),
    (64, 6, 8, 3, 2), (64, 6, 16, 2, 4), (32, 4, 8, 2, 1), (16, 3, 2, 1, 3), (48, 6, 6, 3, 2),
    # groups that the one-warp-per-token kernel takes
    (12, 3, 4, 2, 3), (64, 4, 32, 2, 2), (256, 8, 8, 4, 5), (48, 6, 16, 4, 2),
]


def _logits(T, E, kind, seed):
    rng = np.random.default_rng(seed)
    if kind == "normal":
        return rng.standard_normal((T, E)).astype(np.float32)
    lg = rng.integers(-2, 3, size=(T, E)).astype(np.float32)
    lg[rng.random(lg.shape) < 0.3] = -0.0
    lg[: min(T, 8)] = 0.0
    return lg


def _route_gpu(E, k, ng, tg, gn, lg, offset=0):
    T = lg.shape[0]
    shape = B.Shape(T, 8, E, k, 1, 1, ng, tg, gn)
    flat = torch.empty(T * E + offset, dtype=torch.float32, device="cuda")
    flat[offset:] = torch.from_numpy(lg.reshape(-1)).cuda()
    logits = flat[offset:].view(T, E)
    idx = torch.full((T, k), -1, dtype=torch.int32, device="cuda")
    w = torch.full((T, k), -1.0, dtype=torch.float32, device="cuda")
    ws = B.new_workspace(shape, "cuda")
    B.route_topk(shape, logits, idx, w, ws)
    torch.cuda.synchronize()
    assert B.get_device_error(ws) == 0
    return idx.cpu().numpy(), w.cpu().numpy()


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "E%d_k%d_g%d_%d_%d" % s)
@pytest.mark.parametrize("kind", ["normal", "ties"])
def test_route_geometries_match_oracle(shape, kind):
    E, k, ng, tg, gn = shape
    T = 777  # ragged against every tokens-per-warp and tokens-per-block count
    lg = _logits(T, E, kind, seed=E * 131 + k)
    ref_idx, ref_w = oracle.route_topk(lg, k, ng, tg, gn)
    idx, w = _route_gpu(E, k, ng, tg, gn, lg)
    assert np.array_equal(idx, ref_idx)
    assert np.abs(w - ref_w).max() <= W_TOL


@pytest.mark.parametrize("shape", [(64, 6, 1, 0, 0), (256, 8, 8, 4, 2)],
                         ids=lambda s: "E%d_g%d" % (s[0], s[2]))
def test_route_unaligned_logits_take_the_scalar_loads(shape):
    """A logits pointer 4 bytes past a 16-byte boundary cannot take 16-byte
    loads; the result is the same."""
    E, k, ng, tg, gn = shape
    lg = _logits(500, E, "normal", seed=7)
    ref_idx, ref_w = oracle.route_topk(lg, k, ng, tg, gn)
    idx, w = _route_gpu(E, k, ng, tg, gn, lg, offset=1)
    assert np.array_equal(idx, ref_idx)
    assert np.abs(w - ref_w).max() <= W_TOL
