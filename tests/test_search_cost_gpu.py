"""The search's cost per row stays bounded on the workload shapes.

The temperature each row ends at is fixed by the bisection (parity is
tested elsewhere); how many temperatures the search evaluates to get there
is not, and a few rows whose fp32 entropy lands exactly on the bound, or
whose converged Newton points all fall on one side of the crossing, used
to take 20 to 49 evaluations where the others take 5 to 10, which set the
tail of every launch.  `cs_options.evals_out` reports, per row, the
temperatures its exponentials were evaluated at (the T = 1 pass, every
point of the search, the output pass); these tests hold the mean and the
slowest row to bounds a little above what the launches measure."""
import numpy as np
import pytest

from entropy_bounded_softmax_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _evals(w, rows=None):
    import torch
    import entropy_bounded_softmax_gb300 as cs
    x = wl.generate(w, rows)
    xin = torch.from_numpy(x).cuda()
    out = torch.empty_like(xin)
    ev = torch.zeros(x.shape[0], dtype=torch.int32, device="cuda")
    cs.constrained_softmax(xin, w.entropy_bound, w.t_min, w.t_max, w.max_iter,
                           out=out, evals_out=ev)
    return ev.cpu().numpy()


def _sweep(name):
    return [w for w in wl.sweep_workloads() if w.name == name][0]


# (workload, rows (None: all), mean bound, slowest-row bound); measured
# means 10.2, 6.5, 7.1, 7.6, 9.7 and slowest rows 14, 10, 10, 12, 25.  The
# 32 x 50000 launch evaluates a fan of three temperatures with T = 1 in
# every row (counted), which saves it search rounds.
CASES = [
    (wl.LATENCY, None, 11.0, 15),
    (wl.ROUTER, None, 7.0, 12),
    (wl.LONG, None, 7.6, 13),
    (_sweep("sweep_4096x32000_b0.05_it20"), 1024, 8.1, 16),
    (_sweep("sweep_4096x32000_b1.0_it40"), 1024, 10.3, 30),
]


@pytest.mark.parametrize("w,rows,mean_bound,max_bound", CASES,
                         ids=[c[0].name for c in CASES])
def test_evaluations_per_row(w, rows, mean_bound, max_bound):
    e = _evals(w, None if rows is None else np.arange(rows))
    # Every row evaluates at least T = 1 and its output.
    assert e.min() >= 2
    print(f"{w.name}: mean {e.mean():.2f}, slowest {e.max()}")
    assert e.mean() <= mean_bound
    assert e.max() <= max_bound
