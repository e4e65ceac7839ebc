"""GPU parity on the workload shapes: the CUDA path (through the C ABI)
against the fp64 oracle, element by element on the same seeded inputs.

Small shapes are compared in full; the full-size shapes are launched whole,
in the configuration the benchmark times, and compared on sampled rows the
oracle computes one by one."""
import numpy as np
import pytest

import oracle
from entropy_bounded_softmax_gb300 import workloads as wl
from gpu_parity import check_launch_status, compare, run_gpu

pytestmark = pytest.mark.gpu


def _params(w):
    return dict(entropy_bound=w.entropy_bound, t_min=w.t_min, t_max=w.t_max,
                max_iter=w.max_iter)


def _oracle(x, w):
    return oracle.constrained_softmax(x, **_params(w))


@pytest.mark.parametrize("variant,param", [("auto", 0), ("cluster", 1),
                                           ("cluster", 2), ("cluster", 4),
                                           ("rowgroup", 32)])
def test_small_4x1000(variant, param):
    w = wl.SMALL
    x = wl.generate(w)
    p, T, mask = run_gpu(x, variant=variant, param=param, **_params(w))
    compare(x, p, T, mask, _oracle(x, w), **_params(w))


@pytest.mark.parametrize("variant,param,threads,strict", [
    ("auto", 0, 0, False), ("cluster", 1, 0, True), ("cluster", 2, 0, False),
    ("cluster", 4, 0, False), ("cluster", 4, 256, False),
    ("cluster", 8, 0, False), ("cluster", 4, 0, True)])
def test_latency_32x50000(variant, param, threads, strict):
    w = wl.LATENCY
    x = wl.generate(w)
    p, T, mask = run_gpu(x, variant=variant, param=param, threads=threads,
                         strict=strict, **_params(w))
    stats = compare(x, p, T, mask, _oracle(x, w), **_params(w))
    assert stats["T_zone"] == 0


@pytest.mark.parametrize("C", [700, 1000, 1024, 1500, 2001, 4000])
def test_many_rows_of_middle_width(C):
    # Rows of up to 1024 classes run one warp each (row-group kernel, 32
    # classes a lane); wider ones in one-CTA clusters of 64 threads when
    # there are many rows.  Element by element against the oracle.
    import entropy_bounded_softmax_gb300 as cs
    w = wl.SMALL.with_(batch=1024, num_classes=C, sigma=2.0, seed=4000 + C)
    plan = cs.plan(w.batch, C)
    if C <= 1024:
        assert plan["variant"] == 1 and plan["lanes_per_row"] == 32
    elif C <= 4600:
        assert plan["cluster_size"] == 1 and plan["threads_per_cta"] == 64
    x = wl.generate(w)
    p, T, mask = run_gpu(x, **_params(w))
    stats = compare(x, p, T, mask, _oracle(x, w), **_params(w))
    assert stats["T_zone"] == 0


@pytest.mark.parametrize("seed", [7, 8, 9])
@pytest.mark.parametrize("bound", [0.05, 0.2, 1.0])
def test_few_row_launches_with_the_fan(seed, bound):
    # The 32 x 50000 shape takes the fan (temperatures evaluated with T = 1
    # that place the search's first point); other rows and bounds than the
    # workload's, element by element against the oracle.
    import entropy_bounded_softmax_gb300 as cs
    w = wl.LATENCY.with_(seed=seed, entropy_bound=bound)
    assert cs.plan(w.batch, w.num_classes)["fan_points"] == 3
    x = wl.generate(w)
    p, T, mask = run_gpu(x, **_params(w))
    stats = compare(x, p, T, mask, _oracle(x, w), **_params(w))
    assert stats["T_zone"] == 0


def test_moe_router_full():
    w = wl.ROUTER
    x = wl.generate(w)
    p, T, mask = run_gpu(x, **_params(w))
    stats = compare(x, p, T, mask, _oracle(x, w), **_params(w))
    assert stats["T_zone"] == 0


@pytest.mark.parametrize("lanes", [2, 4, 8, 16, 32])
def test_moe_router_lanes(lanes):
    w = wl.ROUTER
    rows = np.arange(2048)
    x = wl.generate(w, rows)
    p, T, mask = run_gpu(x, variant="rowgroup", param=lanes, **_params(w))
    compare(x, p, T, mask, _oracle(x, w), **_params(w))


def test_moe_router_cluster_variant():
    w = wl.ROUTER
    x = wl.generate(w, np.arange(512))
    p, T, mask = run_gpu(x, variant="cluster", param=1, **_params(w))
    compare(x, p, T, mask, _oracle(x, w), **_params(w))


@pytest.mark.parametrize("param,strict", [(0, False), (4, False),
                                             (8, False), (16, False),
                                             (4, True)])
def test_long_rows_sampled(param, strict):
    """256 x 131072 launched whole; rows sampled for the oracle, always
    including constant, spiked and normal rows."""
    w = wl.LONG
    x = wl.generate(w)
    p, T, mask = run_gpu(x, variant="cluster" if param else "auto",
                         param=param, strict=strict, **_params(w))
    kinds = wl.row_kinds(w)
    pick = sorted(set(wl.sample_rows(w, 10).tolist())
                  | set(np.flatnonzero(kinds == 2)[:3].tolist())
                  | set(np.flatnonzero(kinds == 1)[:3].tolist()))
    ref = _oracle(x[pick], w)
    compare(x[pick], p[pick], T[pick], mask, ref, check_mask=False,
            **_params(w))
    check_launch_status(x, T, mask, w.entropy_bound, w.t_min, w.t_max)
    # Constant rows: exactly uniform, T = t_min, overflow flagged.
    const = np.flatnonzero(kinds == 2)
    assert np.all(p[const] == p[const][:, :1])
    assert np.allclose(p[const], 1.0 / w.num_classes, rtol=1e-6, atol=0)
    assert np.all(T[const] == np.float32(w.t_min))
    assert mask & (1 << 3)


def test_long_rows_no_search_branch():
    """Rows spiked by +20 stay under the bound at T = 1 (no search)."""
    w = wl.LONG.with_(extra={"constant_frac": 0.0, "spike": 20.0}, batch=16)
    x = wl.generate(w)
    p, T, mask = run_gpu(x, **_params(w))
    ref = _oracle(x, w)
    assert np.sum(ref.T == 1.0) >= 6
    compare(x, p, T, mask, ref, **_params(w))


@pytest.mark.parametrize("bound,iters", wl.SWEEP_POINTS)
@pytest.mark.parametrize("param,threads", [(0, 0), (2, 512)])
def test_sweep_sampled(bound, iters, param, threads):
    w = wl.SWEEP.with_(entropy_bound=bound, max_iter=iters)
    x = wl.generate(w)
    p, T, mask = run_gpu(x, variant="cluster" if param else "auto",
                         param=param, threads=threads, **_params(w))
    pick = wl.sample_rows(w, 24)
    ref = _oracle(x[pick], w)
    compare(x[pick], p[pick], T[pick], mask, ref, check_mask=False,
            **_params(w))
    check_launch_status(x, T, mask, w.entropy_bound, w.t_min, w.t_max)


@pytest.mark.parametrize("name,rows", [("small_4x1000", None),
                                       ("latency_32x50000", None),
                                       ("moe_router_65536x64", 4096),
                                       ("sweep_4096x32000", 256)])
def test_settled_search_matches_strict_bisection(name, rows):
    """The default search (a bracket of grid points closed by Newton-placed
    evaluations) returns the temperature of the strict search (H evaluated
    at every midpoint) on every row, up to fp32 ties at the crossing, which
    the oracle then arbitrates."""
    w = wl.WORKLOADS[name]
    x = wl.generate(w, None if rows is None else np.arange(rows))
    p_s, T_s, m_s = run_gpu(x, strict=True, **_params(w))
    p_a, T_a, m_a = run_gpu(x, **_params(w))
    differ = np.flatnonzero(T_s != T_a)
    assert differ.size <= max(1, x.shape[0] // 1000), differ
    if differ.size:
        ref = _oracle(x[differ], w)
        compare(x[differ], p_a[differ], T_a[differ], m_a, ref,
                check_mask=False, **_params(w))
    check_launch_status(x, T_a, m_a, w.entropy_bound, w.t_min, w.t_max)
    same = np.flatnonzero(T_s == T_a)
    assert np.max(np.abs(p_s[same] - p_a[same])) <= 1e-6
    assert m_s == m_a
