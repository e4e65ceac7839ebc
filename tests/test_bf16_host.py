"""bf16 inputs on the CPU: the seeded generator's rounding to bf16 and the
promotion back to fp32 agree with torch's own bfloat16 conversions (a
library routine), and the bf16 entry point's argument check."""
import numpy as np
import pytest
import torch

import entropy_bounded_softmax_gb300 as cs
from entropy_bounded_softmax_gb300 import workloads as wl


def _edge_values():
    rng = np.random.default_rng(5)
    x = np.concatenate([
        rng.normal(0, 3, 20000), rng.normal(0, 1e30, 500),
        [0.0, -0.0, 1.0, -1.0, np.inf, -np.inf, 3.4e38, -3.4e38, 1e-40,
         1.00390625, 1.01171875, 1.0078125 + 2**-8]]).astype(np.float32)
    # values exactly halfway between two bf16 numbers (ties go to even)
    base = rng.integers(0, 2**15, 2000, dtype=np.uint32) << 16
    half = (base | 0x8000).view(np.float32)
    return np.concatenate([x, half])


def test_rounding_matches_torch():
    x = _edge_values()
    ours = wl.to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    nan = np.isnan(x)
    assert np.array_equal(ours[~nan], ref[~nan])
    # NaN payloads are not specified; NaN must stay NaN
    assert np.all(np.isnan(wl.bf16_to_f32(ours[nan])))


def test_promotion_matches_torch_and_is_exact():
    bits = np.arange(0, 2**16, dtype=np.uint32).astype(np.uint16)
    ours = wl.bf16_to_f32(bits)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).float().numpy()
    fin = np.isfinite(ref)
    assert np.array_equal(ours[fin], ref[fin])
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    # exact: rounding the promoted value gives the pattern back
    assert np.array_equal(wl.to_bf16_bits(ours)[fin], bits[fin])


def test_nan_stays_nan():
    x = np.array([np.nan, -np.nan], dtype=np.float32)
    assert np.all(np.isnan(wl.bf16_to_f32(wl.to_bf16_bits(x))))


A, B = 1 << 20, 1 << 30


@pytest.mark.parametrize("args,status", [
    ((A, B, 4, 10, 0.2, 0.01, 10.0, 20, None), 0),
    ((A + 2, B, 4, 10, 0.2, 0.01, 10.0, 20, None), 0),     # 2-byte aligned
    ((A + 1, B, 4, 10, 0.2, 0.01, 10.0, 20, None), 8),     # misaligned
    ((A, A + 80, 4, 10, 0.2, 0.01, 10.0, 20, None), 0),    # adjacent (80 B of bf16)
    ((A, A + 78, 4, 10, 0.2, 0.01, 10.0, 20, None), 8),    # overlap
    ((None, B, 4, 10, 0.2, 0.01, 10.0, 20, None), 8),
    ((A, B, 4, 10, 0.2, 0.01, 10.0, 20, A + 40), 8),       # t_out overlap
    ((A, B, 4, 0, 0.2, 0.01, 10.0, 20, None), 6),
])
def test_check_args_bf16(args, status):
    assert cs.cs_check_args_bf16(*args) == status
