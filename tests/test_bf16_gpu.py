"""bf16 logits (cs_constrained_softmax_bf16) on the GPU.

The bf16 entry point promotes each logit to fp32 on load (exact) and then
runs the fp32 operation, so on the same logits it must reproduce the fp32
entry point bit for bit: probabilities, temperatures and the error mask.
That is checked on every workload shape, kernel variant and row alignment;
the results are also compared with the oracle on the promoted logits with
the forward's acceptance (tests/gpu_parity.py)."""
import numpy as np
import pytest

import oracle
from entropy_bounded_softmax_gb300 import workloads as wl
from gpu_parity import check_launch_status, compare, run_gpu, run_gpu_bf16

pytestmark = pytest.mark.gpu


def _params(w):
    return dict(entropy_bound=w.entropy_bound, t_min=w.t_min, t_max=w.t_max,
                max_iter=w.max_iter)


def _bf16(x):
    bits = wl.to_bf16_bits(x)
    return bits, wl.bf16_to_f32(bits)


def _same(a, b):
    pa, Ta, ma = a
    pb, Tb, mb = b
    assert np.array_equal(pa.view(np.uint32), pb.view(np.uint32))
    assert np.array_equal(np.asarray(Ta).view(np.uint32),
                          np.asarray(Tb).view(np.uint32))
    assert ma == mb


@pytest.mark.parametrize("name,rows", [("small_4x1000", None),
                                       ("latency_32x50000", None),
                                       ("moe_router_65536x64", 4096)])
def test_workloads_against_oracle(name, rows):
    w = wl.WORKLOADS[name]
    bits, x = _bf16(wl.generate(w, None if rows is None else np.arange(rows)))
    got = run_gpu_bf16(bits, **_params(w))
    _same(got, run_gpu(x, **_params(w)))
    stats = compare(x, *got, oracle.constrained_softmax(x, **_params(w)),
                    **_params(w))
    assert stats["T_zone"] == 0


@pytest.mark.parametrize("name", ["long_rows_256x131072",
                                  "sweep_4096x32000_b0.2_it20"])
def test_full_size_matches_fp32(name):
    w = wl.WORKLOADS.get(name) or next(v for v in wl.sweep_workloads()
                                       if v.name == name)
    bits, x = _bf16(wl.generate(w))
    got = run_gpu_bf16(bits, **_params(w))
    _same(got, run_gpu(x, **_params(w)))
    pick = wl.sample_rows(w, 8)
    compare(x[pick], got[0][pick], got[1][pick], got[2],
            oracle.constrained_softmax(x[pick], **_params(w)),
            check_mask=False, **_params(w))
    check_launch_status(x, got[1], got[2], w.entropy_bound, w.t_min, w.t_max)


@pytest.mark.parametrize("C", [1, 3, 5, 33, 64, 257, 513, 4099, 50001])
@pytest.mark.parametrize("variant,param", [("auto", 0), ("rowgroup", 32),
                                           ("cluster", 1), ("cluster", 3)])
@pytest.mark.parametrize("offsets", [(0, 0), (1, 0), (2, 3), (3, 1)])
def test_shapes_variants_alignments(C, variant, param, offsets):
    if variant == "rowgroup" and C > 1024:
        pytest.skip("row longer than 32 lanes x 32 classes")
    rng = np.random.default_rng([C, param, *offsets])
    x = (rng.normal(0, 2.5, (6, C)) + rng.normal(0, 3, (6, 1))).astype(np.float32)
    bits, xf = _bf16(x)
    kw = dict(variant=variant, param=param, in_offset=offsets[0],
              out_offset=offsets[1])
    got = run_gpu_bf16(bits, **kw)
    _same(got, run_gpu(xf, **kw))
    compare(xf, *got, oracle.constrained_softmax(xf))


def test_nan_inf_patterns():
    x = np.random.default_rng(3).normal(0, 2, (6, 700)).astype(np.float32)
    bits = wl.to_bf16_bits(x)
    bits[1, 5] = 0x7FC0      # NaN
    bits[2, 9] = 0x7F80      # +inf
    bits[3, 0] = 0xFF80      # -inf
    bits[4, 1] = 0xFFC1      # NaN with payload
    xf = wl.bf16_to_f32(bits)
    got = run_gpu_bf16(bits)
    ref = oracle.constrained_softmax(xf)
    assert list(ref.flags[1:5]) == [1, 2, 2, 1]
    compare(xf, *got, ref)


@pytest.mark.parametrize("strict", [False, True])
def test_strict_and_forty_steps(strict):
    w = wl.SWEEP.with_(batch=64, max_iter=40, entropy_bound=0.05)
    bits, x = _bf16(wl.generate(w))
    got = run_gpu_bf16(bits, strict=strict, **_params(w))
    _same(got, run_gpu(x, strict=strict, **_params(w)))
    compare(x, *got, oracle.constrained_softmax(x, **_params(w)), **_params(w))
