"""GPU edge cases: ragged and unaligned rows, every variant, the NaN/Inf and
unsatisfiable-bound policy ("BURT-IMMA CUDA Kernel API Reference",
sections 5.3 and 5.4), parameter edges, argument errors, and the bounded
wait's timeout path."""
import math

import numpy as np
import pytest

import oracle
from gpu_parity import TIMEOUT_BIT, compare, run_gpu

pytestmark = pytest.mark.gpu

RAGGED = [1, 2, 3, 5, 31, 33, 63, 65, 255, 257, 511, 513, 1023, 4099, 50001]


def _x(B, C, seed, sigma=2.0):
    return np.random.default_rng(seed).normal(0, sigma, (B, C)).astype(np.float32)


@pytest.mark.parametrize("C", RAGGED)
@pytest.mark.parametrize("offsets", [(0, 0), (1, 3), (2, 2)])
def test_ragged_auto(C, offsets):
    x = _x(7, C, C)
    p, T, mask = run_gpu(x, in_offset=offsets[0], out_offset=offsets[1])
    compare(x, p, T, mask, oracle.constrained_softmax(x))


@pytest.mark.parametrize("C", [5, 63, 257, 1023])
@pytest.mark.parametrize("lanes", [1, 4, 32])
def test_ragged_rowgroup(C, lanes):
    if (C + 3) // 4 > 8 * lanes:
        pytest.skip("row too long for this many lanes")
    x = _x(9, C, 100 + C)
    p, T, mask = run_gpu(x, variant="rowgroup", param=lanes, in_offset=1,
                         out_offset=2)
    compare(x, p, T, mask, oracle.constrained_softmax(x))


@pytest.mark.parametrize("C", [3, 65, 4099, 50001])
@pytest.mark.parametrize("n", [1, 2, 3, 5, 16])
def test_ragged_cluster(C, n):
    x = _x(5, C, 200 + C)
    p, T, mask = run_gpu(x, variant="cluster", param=n, in_offset=3,
                         out_offset=1)
    compare(x, p, T, mask, oracle.constrained_softmax(x))


@pytest.mark.parametrize("variant,C", [("rowgroup", 64), ("cluster", 4096),
                                       ("cluster", 131072)])
def test_nan_inf_rows(variant, C):
    x = _x(6, C, 7)
    x[1, C // 2] = np.nan
    x[2, 0] = np.inf
    x[3, C - 1] = -np.inf
    x[4, 1 % C] = np.nan
    x[4, 0] = np.inf
    p, T, mask = run_gpu(x, variant=variant)
    ref = oracle.constrained_softmax(x)
    assert list(ref.flags[1:5]) == [1, 2, 2, 1]
    compare(x, p, T, mask, ref)


@pytest.mark.parametrize("C", [2, 64, 1000, 50000])
def test_constant_rows_uniform(C):
    x = np.full((3, C), 1.25, dtype=np.float32)
    p, T, mask = run_gpu(x)
    assert np.all(p == p[0, 0])
    assert abs(float(p[0, 0]) * C - 1.0) < 1e-6
    assert np.all(T == np.float32(0.01))
    assert mask == 1 << 3


@pytest.mark.parametrize("C", [64, 1000, 50000])
@pytest.mark.parametrize("kw", [
    dict(max_iter=0), dict(max_iter=1), dict(max_iter=40),
    dict(t_max=0.3), dict(t_min=1.5), dict(entropy_bound=-0.5),
    dict(entropy_bound=float("inf")), dict(entropy_bound=3.0),
    dict(entropy_bound=0.05, max_iter=40), dict(t_min=1e-6, max_iter=30),
])
def test_parameter_edges(C, kw):
    x = _x(6, C, 31 + C, sigma=3.0)
    p, T, mask = run_gpu(x, **kw)
    compare(x, p, T, mask, oracle.constrained_softmax(x, **kw), **kw)


def test_single_class():
    x = np.array([[3.0], [-1e30], [0.0]], dtype=np.float32)
    p, T, mask = run_gpu(x)
    assert np.all(p == 1.0) and np.all(T == 1.0) and mask == 0


def test_extreme_finite_logits():
    x = np.zeros((3, 300), dtype=np.float32)
    x[0, 5] = 3e38
    x[0, 6] = -3e38
    x[1] = np.linspace(-1e30, 1e30, 300, dtype=np.float32)
    x[2, :] = -3e38
    x[2, 7] = 3e38
    p, T, mask = run_gpu(x)
    compare(x, p, T, mask, oracle.constrained_softmax(x))


def test_batch_zero_and_argument_errors():
    import torch
    import entropy_bounded_softmax_gb300 as cs
    dev = torch.device("cuda", 0)
    x = torch.zeros((0, 10), device=dev)
    assert cs.constrained_softmax(x).shape == (0, 10)
    x = torch.randn(4, 10, device=dev)
    for kw, status in [(dict(t_min=0.0), 8), (dict(t_min=-1.0), 8),
                       (dict(t_max=0.001), 8),
                       (dict(entropy_bound=float("nan")), 8),
                       (dict(max_iter=-1), 8), (dict(max_iter=5000), 8)]:
        with pytest.raises(cs.CsError) as e:
            cs.constrained_softmax(x, **kw)
        assert e.value.status == status
    with pytest.raises(cs.CsError) as e:
        cs.constrained_softmax(x, out=x)
    assert e.value.status == 8
    assert cs.cs_constrained_softmax(x.data_ptr(), 0, 4, 10, 0.2, 0.01, 10.0,
                                     20, None, None) == 8
    assert cs.cs_constrained_softmax_ex(x.data_ptr(), x.data_ptr() + 4096, 4,
                                        10, 0.2, 0.01, 10.0, 20, None,
                                        cs.options(2, 0, 33, 0), None) == 8
    big = torch.zeros((1, 900000), device=dev)
    with pytest.raises(cs.CsError) as e:
        cs.constrained_softmax(big)
    assert e.value.status == 7
    with pytest.raises(cs.CsError) as e:
        cs.constrained_softmax(x, variant="rowgroup", param=3)
    assert e.value.status == 8


def test_wait_timeout_is_reported():
    """A barrier nothing completes: the bounded wait gives up after 1 ms and
    the kernel records CS_ERR_TIMEOUT; the context stays usable."""
    import torch
    import entropy_bounded_softmax_gb300 as cs
    cs.get_error()
    stream = torch.cuda.current_stream().cuda_stream
    assert cs.cs_test_wait_timeout(1_000_000, stream) == 0
    assert cs.get_error() == {"TIMEOUT"}
    x = _x(2, 100, 1)
    p, T, mask = run_gpu(x)
    compare(x, p, T, mask, oracle.constrained_softmax(x))


def test_probe_runs():
    import torch
    import entropy_bounded_softmax_gb300 as cs
    n = cs.cs_probe_ex2_sink_floats()
    sink = torch.empty(n, device="cuda")
    st, count = cs.cs_probe_ex2(sink.data_ptr(), 64,
                                torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert st == 0 and count == n * 64 * 8
    assert torch.isfinite(sink).all()


def test_plan_launch_matches_host_plan():
    import torch
    import entropy_bounded_softmax_gb300 as cs
    props = torch.cuda.get_device_properties(0)
    for shape in [(65536, 64), (32, 50000), (256, 131072), (4096, 32000)]:
        p = cs.plan(*shape)
        assert p["grid_ctas"] > 0
    assert props.multi_processor_count > 0
