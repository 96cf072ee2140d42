"""Pins for the oracle's bf16 rounding (round to nearest, ties to even)."""
import numpy as np
import torch


def _torch_bits(f32):
    t = torch.from_numpy(np.ascontiguousarray(f32, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_matches_torch_cast_on_fp32_inputs(orc):
    rng = np.random.default_rng(1)
    parts = [
        rng.standard_normal(20000).astype(np.float32),
        (rng.standard_normal(5000) * 1e30).astype(np.float32),
        (rng.standard_normal(5000) * 1e-38).astype(np.float32),  # subnormal range
        (rng.standard_normal(5000) * 1e-42).astype(np.float32),
        np.array([0.0, -0.0, np.inf, -np.inf, 3.3e38, -3.3e38, 3.4e38, 1.0, -1.0],
                 dtype=np.float32),
    ]
    # every bf16 value plus a mid-point (exact tie) and a quarter-point above it
    allb = np.arange(0, 1 << 16, dtype=np.uint32)
    base = (allb << 16).view(np.float32)
    fin = np.isfinite(base)
    parts += [base[fin], (allb[fin] << 16 | 0x8000).view(np.float32),
              (allb[fin] << 16 | 0x4000).view(np.float32),
              (allb[fin] << 16 | 0xC000).view(np.float32)]
    v = np.concatenate(parts)
    v = v[np.isfinite(v) | np.isinf(v)]
    assert np.array_equal(orc.bf16_round(v.astype(np.float64)), _torch_bits(v))


def test_ties_go_to_even(orc):
    one = 1.0
    ulp = 2.0 ** -7  # spacing of bf16 in [1, 2)
    assert orc.bf16_from_double(one + ulp / 2) == 0x3F80  # 1.0 (even) wins
    assert orc.bf16_from_double(one + 3 * ulp / 2) == 0x3F82  # 1 + 2ulp (even) wins
    assert orc.bf16_from_double(-(one + ulp / 2)) == 0xBF80


def test_fp64_inputs_round_once(orc):
    # Just above a tie: a double that would first round to the tie in fp32
    # and then to even must round up when rounded once.
    v = 1.0 + 2.0 ** -8 + 2.0 ** -40
    assert orc.bf16_from_double(v) == 0x3F81
    assert orc.bf16_from_double(1.0 + 2.0 ** -8 - 2.0 ** -40) == 0x3F80


def test_special_values(orc):
    assert orc.bf16_from_double(0.0) == 0x0000
    assert orc.bf16_from_double(-0.0) == 0x8000
    assert orc.bf16_from_double(float("inf")) == 0x7F80
    assert orc.bf16_from_double(-float("inf")) == 0xFF80
    assert orc.bf16_from_double(1e39) == 0x7F80  # overflow
    assert orc.bf16_from_double(2.0 ** -133) == 0x0001  # smallest subnormal
    assert orc.bf16_from_double(2.0 ** -134) == 0x0000  # tie with 0 -> even (0)
    assert orc.bf16_from_double(3 * 2.0 ** -134) == 0x0002  # tie 1/2 -> even (2)
