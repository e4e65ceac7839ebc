"""The GPU tests' acceptance helpers, checked on the CPU against the oracle
itself: the per-row flags that launch_flags derives from H(1) and H(t_min)
alone equal the flags of the oracle's full search, and compare() rejects a
temperature two grid points off at max_iter <= 24."""
import numpy as np
import pytest

import oracle
from gpu_parity import compare, launch_flags


@pytest.mark.parametrize("kw", [
    dict(), dict(entropy_bound=0.05), dict(entropy_bound=1.0, max_iter=40),
    dict(t_min=0.05), dict(t_max=0.3), dict(t_min=1.5), dict(max_iter=0),
    dict(entropy_bound=-0.5), dict(entropy_bound=float("inf"))])
def test_launch_flags_match_the_oracle(kw):
    rng = np.random.default_rng(7)
    x = rng.normal(0.0, 2.0, (48, 37)).astype(np.float32)
    x[3] = 1.25                     # constant row
    x[5, 4] = np.nan
    x[6, 2] = np.inf
    x[7, 1] = -np.inf
    x[8, :2] = [9.0, 9.0 - 1e-3]    # near-tie at the top: unsatisfiable
    x[9, 0] += 40.0                 # no search
    flags, _ = launch_flags(x, **{k: v for k, v in kw.items()
                                  if k in ("entropy_bound", "t_min", "t_max")})
    ref = oracle.constrained_softmax(x, **kw)
    assert np.array_equal(flags, ref.flags)


def test_compare_rejects_a_temperature_two_grid_points_off():
    rng = np.random.default_rng(11)
    x = rng.normal(0.0, 2.0, (4, 200)).astype(np.float32)
    ref = oracle.constrained_softmax(x)
    T = ref.T.astype(np.float32)
    p = ref.p.astype(np.float32)
    mask = 0
    compare(x, p, T, mask, ref)                 # the oracle's own result
    w = oracle.final_interval(0.01, 10.0, 20)
    T_bad = T.copy()
    T_bad[0] = np.float32(ref.T[0] - 2.5 * w)
    p_bad = p.copy()
    p_bad[0] = oracle.softmax(x[0], float(T_bad[0])).astype(np.float32)
    with pytest.raises(AssertionError, match="one final interval"):
        compare(x, p_bad, T_bad, mask, ref)
