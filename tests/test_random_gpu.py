"""Seeded random cases for every operation, drawn from wide ranges of
shapes and parameters, each checked against the oracle with the same
acceptance as the dedicated tests (tests/gpu_parity.py,
tests/backward_parity.py, tests/attention_parity.py,
tests/biencoder_parity.py)."""
import numpy as np
import pytest

import oracle
from attention_parity import compare_full, run_attention
from backward_parity import compare as compare_backward
from backward_parity import probs_for, run_backward
from biencoder_parity import compare_biencoder, run_biencoder
from gpu_parity import compare, run_gpu

pytestmark = pytest.mark.gpu


def _case_rng(kind, seed):
    return np.random.default_rng([ord(c) for c in kind] + [seed])


@pytest.mark.parametrize("seed", range(12))
def test_forward_random(seed):
    rng = _case_rng("forward", seed)
    B = int(rng.integers(1, 40))
    C = int(rng.choice([int(rng.integers(1, 600)), int(rng.integers(600, 70000))]))
    sigma = float(rng.uniform(0.2, 5.0))
    kw = dict(entropy_bound=float(rng.choice([0.05, 0.2, 0.7, 2.0])),
              t_min=float(rng.choice([0.01, 0.05, 0.2])),
              t_max=float(rng.choice([0.5, 1.0, 10.0])),
              max_iter=int(rng.choice([0, 5, 20, 33])))
    x = (rng.normal(0.0, sigma, (B, C)) + rng.normal(0.0, 3.0, (B, 1))).astype(np.float32)
    p, T, mask = run_gpu(x, in_offset=int(rng.integers(0, 4)),
                         out_offset=int(rng.integers(0, 4)), **kw)
    compare(x, p, T, mask, oracle.constrained_softmax(x, **kw), **kw)


@pytest.mark.parametrize("seed", range(8))
def test_backward_random(seed):
    rng = _case_rng("backward", seed)
    B = int(rng.integers(1, 30))
    C = int(rng.choice([int(rng.integers(1, 600)), int(rng.integers(600, 200000))]))
    x = rng.normal(0.0, 2.0, (B, C)).astype(np.float32)
    g = rng.normal(0.0, 1.0, (B, C)).astype(np.float32)
    T = rng.uniform(0.01, 1.0, B).astype(np.float32)
    T[rng.random(B) < 0.1] = np.nan
    p = probs_for(x, T)
    grad = run_backward(p, g, T, offsets=tuple(int(v) for v in rng.integers(0, 4, 3)))
    compare_backward(grad, p, g, T)


@pytest.mark.parametrize("seed", range(8))
def test_attention_random(seed):
    rng = _case_rng("attention", seed)
    S = int(rng.choice([int(rng.integers(1, 200)), int(rng.integers(200, 3000))]))
    B, H = int(rng.integers(1, 3)), int(rng.integers(1, 3))
    x = rng.normal(0.0, float(rng.uniform(0.5, 4.0)), (B, H, S, S)).astype(np.float32)
    mask = None
    if rng.random() < 0.7:
        mask = np.zeros((B, S), dtype=np.float32)
        val = np.float32(-1e9) if rng.random() < 0.5 else np.float32(-np.inf)
        mask[rng.random((B, S)) < 0.3] = val
    causal = bool(rng.random() < 0.5)
    out, em = run_attention(x, mask, causal,
                            offsets=tuple(int(v) for v in rng.integers(0, 4, 3)))
    compare_full(x, mask, causal, out, em)


@pytest.mark.parametrize("seed", range(6))
def test_biencoder_random(seed):
    rng = _case_rng("biencoder", seed)
    K = int(rng.integers(1, 257))
    D = 4 * int(rng.integers(1, 33))
    if K * D > 20000:
        D = 4 * max(1, 20000 // (4 * K))
    B, H, Q = int(rng.integers(1, 3)), int(rng.integers(1, 4)), int(rng.integers(1, 300))
    q = rng.normal(0.0, 1.0, (B, H, Q, D)).astype(np.float32)
    k = rng.normal(0.0, 1.0, (B, H, K, D)).astype(np.float32)
    v = rng.normal(0.0, 1.0, (B, H, K, D)).astype(np.float32)
    scale = float(rng.uniform(0.05, 1.0))
    bound = float(rng.choice([0.05, 0.2, 1.0]))
    out, attn, T, mask = run_biencoder(q, k, v, scale, bound)
    compare_biencoder(q, k, v, scale, out, attn, T, mask, bound)


@pytest.mark.parametrize("seed", range(8))
def test_biencoder_tensor_core_random(seed):
    """Shapes that take the tensor-core attn . V kernel (context_len <=
    d_head <= 64): many (batch, head) pairs per persistent CTA, ragged
    query tiles, contexts that are not a multiple of 4 or 32.  Against the
    oracle with the weights returned (attn_out; element loads when its rows
    are not 16-byte aligned), and the same output bit for bit with the
    weights passing through the output buffer (tensor copies)."""
    rng = _case_rng("biencoder_tc", seed)
    D = 4 * int(rng.integers(1, 17))
    K = int(rng.integers(1, D + 1))
    B, H, Q = (int(rng.integers(1, 4)), int(rng.integers(1, 9)),
               int(rng.integers(1, 600)))
    q = rng.normal(0.0, 1.0, (B, H, Q, D)).astype(np.float32)
    k = rng.normal(0.0, 1.0, (B, H, K, D)).astype(np.float32)
    v = rng.normal(0.0, 1.0, (B, H, K, D)).astype(np.float32)
    scale = float(rng.uniform(0.05, 1.0))
    bound = float(rng.choice([0.05, 0.2, 1.0]))
    out, attn, T, mask = run_biencoder(q, k, v, scale, bound)
    compare_biencoder(q, k, v, scale, out, attn, T, mask, bound)
    out2, _, T2, mask2 = run_biencoder(q, k, v, scale, bound, return_attn=False)
    assert np.array_equal(T2, T) and mask2 == mask
    assert np.array_equal(out2, out)
