"""GPU parity of the backward, grad = (1/T) p (g - <g, p>) per row
("BURT-IMMA CUDA Kernel API Reference", section 6.3, with the 1/T of
softmax(l / T) restored): the CUDA kernels through the C ABI against the
fp64 oracle on the same seeded inputs, on every workload shape (the two
largest compared on sampled rows), every variant, ragged and unaligned rows,
in place, the T = NaN rows, and the autograd wrapper end to end."""
import math

import numpy as np
import pytest

import oracle
from backward_parity import compare, probs_for, run_backward
from entropy_bounded_softmax_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _inputs(w, rows=None):
    x = wl.generate(w, rows)
    g, T = wl.backward_inputs(w, rows)
    return probs_for(x, T), g, T


@pytest.mark.parametrize("name", ["small_4x1000", "latency_32x50000",
                                  "moe_router_65536x64"])
def test_workloads_full(name):
    w = wl.WORKLOADS[name]
    p, g, T = _inputs(w)
    assert (T == 1.0).any() and (np.isnan(T).any() or w.batch <= 5)
    compare(run_backward(p, g, T), p, g, T)


@pytest.mark.parametrize("name", ["long_rows_256x131072", "sweep_4096x32000"])
def test_workloads_sampled(name):
    """Launched whole (the benchmark's configuration); rows sampled for the
    oracle, NaN-T and T = 1 rows included."""
    w = wl.WORKLOADS[name]
    p, g, T = _inputs(w)
    grad = run_backward(p, g, T)
    pick = sorted(set(wl.sample_rows(w, 48).tolist())
                  | set(np.flatnonzero(np.isnan(T))[:2].tolist())
                  | set(np.flatnonzero(T == 1.0)[:2].tolist()))
    compare(grad[pick], p[pick], g[pick], T[pick])


def _rand(B, C, seed, t_lo=0.05):
    rng = np.random.default_rng(seed)
    x = rng.normal(0.0, 2.0, (B, C)).astype(np.float32)
    g = rng.normal(0.0, 1.0, (B, C)).astype(np.float32)
    T = rng.uniform(t_lo, 1.0, B).astype(np.float32)
    T[0] = 1.0
    if B > 2:
        T[2] = np.nan
    return probs_for(x, T), g, T


RAGGED = [1, 2, 3, 5, 31, 33, 63, 64, 65, 255, 257, 511, 513, 1023, 4099,
          8191, 8193, 50001]


@pytest.mark.parametrize("C", RAGGED)
@pytest.mark.parametrize("offsets", [(0, 0, 0), (1, 3, 2), (2, 2, 2)])
def test_ragged_auto(C, offsets):
    p, g, T = _rand(7, C, C)
    compare(run_backward(p, g, T, offsets=offsets), p, g, T)


@pytest.mark.parametrize("C", [1, 5, 64, 127, 257, 1000])
@pytest.mark.parametrize("lanes", [1, 2, 4, 8, 16, 32])
def test_rowgroup_lanes(C, lanes):
    if (C + 6) // 4 > 8 * lanes:
        pytest.skip("row too long for this many lanes")
    p, g, T = _rand(9, C, 300 + C)
    compare(run_backward(p, g, T, variant="rowgroup", param=lanes,
                         offsets=(1, 2, 3)), p, g, T)


@pytest.mark.parametrize("C", [3, 65, 4099, 50001, 131072])
@pytest.mark.parametrize("n", [1, 2, 3, 5, 16])
def test_cluster_sizes(C, n):
    if -(-C // n) * 4 > 220000:
        pytest.skip("slice of p alone exceeds a CTA's shared memory")
    p, g, T = _rand(5, C, 400 + C)
    compare(run_backward(p, g, T, variant="cluster", param=n,
                         offsets=(3, 1, 2)), p, g, T)


@pytest.mark.parametrize("threads", [64, 96, 512])
def test_cluster_threads(threads):
    p, g, T = _rand(6, 20000, 77)
    compare(run_backward(p, g, T, variant="cluster", param=2,
                         threads=threads), p, g, T)


@pytest.mark.parametrize("C,n", [(50001, 1), (100003, 2), (850000, 16)])
def test_p_only_staging(C, n):
    """Slices too long to hold both p and g in shared memory keep p and read
    g again."""
    import entropy_bounded_softmax_gb300 as cs
    plan = cs.plan_backward(3, C, variant="cluster", param=n)
    assert plan["staged_tensors"] == 1
    p, g, T = _rand(3, C, 500 + n)
    compare(run_backward(p, g, T, variant="cluster", param=n,
                         offsets=(1, 1, 0)), p, g, T)


def test_auto_plan_for_largest_rows():
    import entropy_bounded_softmax_gb300 as cs
    plan = cs.plan_backward(2, 850000)
    assert plan["cluster_size"] == 16 and plan["staged_tensors"] == 1
    p, g, T = _rand(2, 850000, 9)
    compare(run_backward(p, g, T), p, g, T)


@pytest.mark.parametrize("inplace", ["probs", "grad_output"])
@pytest.mark.parametrize("variant,param,C", [("rowgroup", 0, 64),
                                             ("cluster", 1, 1000),
                                             ("cluster", 4, 32000),
                                             ("cluster", 1, 50001)])
def test_in_place(inplace, variant, param, C):
    p, g, T = _rand(6, C, 600 + C)
    compare(run_backward(p, g, T, variant=variant, param=param,
                         inplace=inplace), p, g, T)


@pytest.mark.parametrize("C", [64, 4096, 50000])
def test_invalid_temperatures_and_nan_gradients(C):
    """T NaN, +-0, negative or +inf: zero rows.  A NaN or Inf in g spreads
    through the row's dot product exactly as in fp64."""
    p, g, T = _rand(8, C, 700 + C)
    T[1] = np.inf
    T[3] = 0.0
    T[4] = -0.5
    T[5] = -0.0
    g[6, C // 3] = np.nan
    g[7, C // 2] = np.inf
    grad = run_backward(p, g, T)
    assert np.all(grad[[1, 2, 3, 4, 5]] == 0.0)
    assert np.all(np.isnan(grad[6]))
    compare(grad, p, g, T)


def test_batch_zero_and_argument_errors():
    import torch
    import entropy_bounded_softmax_gb300 as cs
    dev = torch.device("cuda", 0)
    z = torch.zeros((0, 10), device=dev)
    t0 = torch.zeros(0, device=dev)
    assert cs.constrained_softmax_backward(z, z, t0).shape == (0, 10)
    p = torch.rand(4, 10, device=dev)
    t = torch.ones(4, device=dev)
    with pytest.raises(cs.CsError) as e:
        cs.constrained_softmax_backward(p, p, t, variant="rowgroup", param=3)
    assert e.value.status == 8
    with pytest.raises(cs.CsError) as e:
        cs.constrained_softmax_backward(p, p, t, variant="cluster", param=17)
    assert e.value.status == 8
    buf = torch.zeros(50, device=dev)
    with pytest.raises(cs.CsError) as e:   # grad overlaps p, not equal
        cs.constrained_softmax_backward(buf[:40].view(4, 10), p, t,
                                        out=buf[5:45].view(4, 10))
    assert e.value.status == 8
    assert cs.cs_constrained_softmax_backward(
        p.data_ptr(), p.data_ptr(), None, p.data_ptr(), 4, 10, None) == 8
    with pytest.raises(cs.CsError) as e:
        big = torch.zeros((1, 900000), device=dev)
        cs.constrained_softmax_backward(big, big, t[:1])
    assert e.value.status == 7


def test_autograd_end_to_end():
    """ConstrainedSoftmaxFunction: forward and backward on the GPU against
    the oracle's forward and backward on the same logits.  Rows where the
    two forwards settle on the same T are compared; the bound allows for the
    forward's |dp| <= 2e-5 on both p and <g, p>."""
    import torch
    import entropy_bounded_softmax_gb300 as cs
    rng = np.random.default_rng(81)
    x = rng.normal(0.0, 3.0, (64, 700)).astype(np.float32)
    x[9, 3] = np.nan
    w = rng.normal(0.0, 1.0, (64, 700)).astype(np.float32)
    ref = oracle.constrained_softmax(x)
    dev = torch.device("cuda", 0)
    l = torch.tensor(x, device=dev, requires_grad=True)
    out = cs.ConstrainedSoftmaxFunction.apply(l, 0.2, 0.01, 10.0, 20)
    (out * torch.tensor(w, device=dev)).sum().backward()
    grad = l.grad.cpu().numpy().astype(np.float64)
    _, T_gpu = cs.constrained_softmax(l.detach(), return_t=True)
    T_gpu = T_gpu.cpu().numpy()
    ref_grad = oracle.constrained_softmax_backward(ref.p, w, ref.T)
    same = np.flatnonzero((T_gpu == ref.T.astype(np.float32))
                          | (np.isnan(T_gpu) & np.isnan(ref.T)))
    assert same.size >= 60
    w64 = w.astype(np.float64)
    dot = np.sum(ref.p * w64, axis=1, keepdims=True)
    bound = (2e-5 * np.abs(w64 - dot)
             + (ref.p + 2e-5) * 2e-5 * np.sum(np.abs(w64), axis=1,
                                               keepdims=True)) / \
        np.where(np.isnan(ref.T), 1.0, ref.T)[:, None] + 1e-6
    assert np.all(np.abs(grad[same] - ref_grad[same]) <= bound[same])
    assert np.all(grad[9] == 0.0) and math.isnan(ref.T[9])
