"""GPU parity of biencoder_attention ("BURT-IMMA CUDA Kernel API
Reference", section 2.5), fused: the CUDA kernel through the C ABI against
the oracle on the same seeded inputs: the page's shape and a 256-item
context in full, ragged context lengths, head sizes and query counts,
every lane count, the NaN/Inf and unsatisfiable-bound policy, argument
errors."""
import numpy as np
import pytest

from biencoder_parity import (compare_biencoder,
                              compare_biencoder_fp64_scores, run_biencoder)
from entropy_bounded_softmax_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", list(wl.BIENCODER_WORKLOADS))
def test_workloads_full(name):
    w = wl.BIENCODER_WORKLOADS[name]
    q, k, v = wl.generate_biencoder(w)
    scale = 1.0 / np.sqrt(w.d_head)
    out, attn, T, mask = run_biencoder(q, k, v, scale, w.entropy_bound)
    stats = compare_biencoder(q, k, v, scale, out, attn, T, mask,
                              w.entropy_bound)
    assert stats["T_zone"] == 0


@pytest.mark.parametrize("name", list(wl.BIENCODER_WORKLOADS))
def test_against_scores_from_an_fp64_matmul(name):
    """Parity does not rest on the kernel and the oracle sharing the fp32
    order of step 1: with the oracle's search run on fp64-matmul scores, the
    GPU's weights, temperatures and output still pass the acceptance."""
    w = wl.BIENCODER_WORKLOADS[name]
    q, k, v = wl.generate_biencoder(w)
    scale = 1.0 / np.sqrt(w.d_head)
    out, attn, T, mask = run_biencoder(q, k, v, scale, w.entropy_bound)
    stats = compare_biencoder_fp64_scores(q, k, v, scale, out, attn, T, mask,
                                          w.entropy_bound)
    assert stats["T_zone"] == 0
    assert stats["rows_with_other_scores"] > 0   # the scores do differ


def _rand(B, H, Q, K, D, seed, sigma=1.0):
    rng = np.random.default_rng(seed)
    q = rng.normal(0.0, sigma, (B, H, Q, D)).astype(np.float32)
    k = rng.normal(0.0, sigma, (B, H, K, D)).astype(np.float32)
    v = rng.normal(0.0, 1.0, (B, H, K, D)).astype(np.float32)
    return q, k, v


@pytest.mark.parametrize("K", [1, 3, 5, 8, 9, 33, 64, 100, 255, 256])
@pytest.mark.parametrize("D", [4, 12, 64])
def test_ragged_shapes(K, D):
    q, k, v = _rand(2, 3, 37, K, D, 7 * K + D, sigma=1.5)
    scale = 1.0 / np.sqrt(D)
    out, attn, T, mask = run_biencoder(q, k, v, scale)
    compare_biencoder(q, k, v, scale, out, attn, T, mask)


@pytest.mark.parametrize("Q", [1, 31, 32, 33, 300])
def test_query_tiles(Q):
    q, k, v = _rand(1, 2, Q, 64, 64, Q)
    out, attn, T, mask = run_biencoder(q, k, v, 0.125)
    compare_biencoder(q, k, v, 0.125, out, attn, T, mask)


@pytest.mark.parametrize("lanes", [1, 2, 4, 8, 16, 32])
@pytest.mark.parametrize("per_lane", [8, 16])
def test_lane_counts(lanes, per_lane):
    """A forced lane count holds eight items a lane when that covers the
    context, else sixteen."""
    K = min(per_lane * lanes, 40)
    if per_lane == 16 and K <= 8 * lanes:
        pytest.skip("eight items a lane already hold this context")
    q, k, v = _rand(2, 2, 50, K, 16, lanes + per_lane)
    out, attn, T, mask = run_biencoder(q, k, v, 0.25, lanes=lanes)
    compare_biencoder(q, k, v, 0.25, out, attn, T, mask)


@pytest.mark.parametrize("kw", [dict(entropy_bound=-1.0),
                                dict(entropy_bound=1e30),
                                dict(entropy_bound=0.05, max_iter=40),
                                dict(t_max=0.3)])
def test_search_parameters(kw):
    q, k, v = _rand(1, 2, 40, 24, 8, 11)
    out, attn, T, mask = run_biencoder(q, k, v, 0.5, **kw)
    compare_biencoder(q, k, v, 0.5, out, attn, T, mask, **kw)


def test_nan_inf_inputs():
    """A NaN query zeroes its row (NAN_INPUT); an infinite key makes every
    row of its (batch, head) pair non-finite (INF_INPUT); a NaN value leaves
    the weights alone and spreads into the outputs that use it."""
    q, k, v = _rand(2, 2, 16, 12, 8, 21)
    q[0, 0, 3, 2] = np.nan
    k[1, 1, 5, 0] = np.inf
    out, attn, T, mask = run_biencoder(q, k, v, 0.3)
    compare_biencoder(q, k, v, 0.3, out, attn, T, mask)
    assert np.all(out[0, 0, 3] == 0.0) and np.isnan(T[0, 0, 3])
    assert np.all(np.isnan(T[1, 1]))
    v2 = v.copy()
    v2[0, 1, 4, 6] = np.nan
    out2, attn2, T2, mask2 = run_biencoder(q[:1], k[:1], v2[:1], 0.3)
    assert np.all(np.isnan(out2[0, 1, :, 6]))
    assert np.all(np.isfinite(out2[0, 1, :, :6]))


def test_argument_errors_and_empty():
    import torch
    import entropy_bounded_softmax_gb300 as cs
    dev = torch.device("cuda", 0)
    q = torch.zeros((0, 2, 4, 8), device=dev)
    k = torch.zeros((0, 2, 3, 8), device=dev)
    assert cs.biencoder_attention(q, k, k).shape == (0, 2, 4, 8)
    q = torch.randn(1, 1, 4, 6, device=dev)
    k = torch.randn(1, 1, 3, 6, device=dev)
    with pytest.raises(cs.CsError) as e:          # d_head not a multiple of 4
        cs.biencoder_attention(q, k, k)
    assert e.value.status == 8
    q = torch.randn(1, 1, 4, 8, device=dev)
    k = torch.randn(1, 1, 300, 8, device=dev)
    with pytest.raises(cs.CsError) as e:          # context too long
        cs.biencoder_attention(q, k, k)
    assert e.value.status == 7
    k = torch.randn(1, 1, 40, 8, device=dev)
    with pytest.raises(cs.CsError) as e:          # 2 lanes hold 32 items
        cs.biencoder_attention(q, k, k, lanes=2)
    assert e.value.status == 7
    with pytest.raises(cs.CsError) as e:          # output overlaps query
        cs.biencoder_attention(q, k, k, out=q)
    assert e.value.status == 8


@pytest.mark.parametrize("K,D", [(64, 64), (1, 4), (5, 12), (12, 12),
                                 (33, 48), (16, 64)])
@pytest.mark.parametrize("Q", [1, 127, 128, 300])
def test_tensor_core_step3_matches_fused(K, D, Q):
    """Step 3 on the tensor cores (three TF32 products, fp32 accumulation)
    against the oracle, with and without attn_out (the weights then pass
    through the output buffer), and against the fused fp32 kernel: same
    weights and temperatures bit for bit (steps 1-2 are the same code), the
    outputs within the fp32 accumulation's bound."""
    import entropy_bounded_softmax_gb300 as cs
    st, plan = cs.cs_plan_biencoder_host(2, Q, K, D, 3, None, 232448)
    assert st == 0 and plan.tensor_cores == 1
    q, k, v = _rand(2, 3, Q, K, D, 97 * K + D + Q, sigma=1.5)
    scale = 1.0 / np.sqrt(D)
    out_tc, attn_tc, T_tc, m_tc = run_biencoder(q, k, v, scale)
    compare_biencoder(q, k, v, scale, out_tc, attn_tc, T_tc, m_tc)
    out_nb, _, T_nb, m_nb = run_biencoder(q, k, v, scale, return_attn=False)
    compare_biencoder(q, k, v, scale, out_nb, attn_tc, T_nb, m_nb)
    out_f, attn_f, T_f, m_f = run_biencoder(q, k, v, scale, fused=True)
    assert np.array_equal(attn_f, attn_tc) and np.array_equal(T_f, T_tc)
    assert m_f == m_tc == m_nb
    assert np.array_equal(T_nb, T_tc)
    v64 = np.abs(v.astype(np.float64))
    bound = 1e-5 * np.einsum("bhqk,bhkd->bhqd", attn_f.astype(np.float64), v64) + 1e-30
    assert np.all(np.abs(out_tc.astype(np.float64) - out_f) <= 2 * bound)
    assert np.array_equal(out_nb, out_tc)
