"""GPU parity of attention_softmax ("BURT-IMMA CUDA Kernel API Reference",
section 2.6): the CUDA kernels through the C ABI against the fp64 oracle on
the same seeded inputs.  The page's workload (32 x 8 x 512, with and
without causal) is compared in full, the long causal case on sampled rows;
ragged and unaligned rows, every variant, in place, masks of -1e9 and -inf,
and the NaN/Inf policy."""
import numpy as np
import pytest

import oracle
from attention_parity import (compare_full, compare_rows, expected_mask,
                              run_attention)
from entropy_bounded_softmax_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _workload(w):
    x = wl.generate_attention(w).reshape(w.batch, w.heads, w.seq_len,
                                         w.seq_len)
    return x, wl.attention_mask(w)


@pytest.mark.parametrize("name", ["attention_32x8x512",
                                  "attention_32x8x512_causal"])
def test_page_workload_full(name):
    w = wl.ATTENTION_WORKLOADS[name]
    x, mask = _workload(w)
    p, em = run_attention(x, mask, w.causal)
    compare_full(x, mask, w.causal, p, em)


def test_long_causal_sampled():
    """2 x 8 x 4096, causal, -inf padding: the row-CTA kernel, launched
    whole, compared on sampled rows (first, last, fully padded queries)."""
    w = wl.ATTN_LONG
    x, mask = _workload(w)
    p, em = run_attention(x, mask, True)
    assert em == 0
    S = w.seq_len
    rng = np.random.default_rng(5)
    picks = sorted(set(rng.choice(w.rows, 40, replace=False).tolist())
                   | {0, S - 1, w.rows - 1, S * 8 - 1})
    pf = p.reshape(w.rows, S)
    xf = x.reshape(w.rows, S)
    for r in picks:
        b, i = r // (w.heads * S), r % S
        ref, flag = oracle.attention_softmax_row(xf[r], i, mask[b], True)
        compare_rows(pf[r:r + 1], xf[r:r + 1], np.array([i]),
                     mask[b:b + 1], True, ref[None], np.array([flag]))


def _rand(B, H, S, seed, kind):
    rng = np.random.default_rng(seed)
    x = rng.normal(0.0, 2.0, (B, H, S, S)).astype(np.float32)
    if kind == "none":
        return x, None
    mask = np.zeros((B, S), dtype=np.float32)
    val = np.float32(-1e9) if kind == "neg_1e9" else np.float32(-np.inf)
    for b in range(B):
        mask[b, rng.random(S) < 0.25] = val
        mask[b, 0] = 0.0
    return x, mask


SEQ = [1, 2, 3, 5, 31, 33, 64, 100, 257, 512, 513, 1000, 1024, 1025, 2048,
       3001]


@pytest.mark.parametrize("S", SEQ)
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("kind", ["none", "neg_1e9", "neg_inf"])
def test_ragged(S, causal, kind):
    x, mask = _rand(2, 2, S, S + 7, kind)
    p, em = run_attention(x, mask, causal, offsets=(1, 3, 2))
    compare_full(x, mask, causal, p, em)


@pytest.mark.parametrize("S", [5, 64, 127, 512, 1000])
@pytest.mark.parametrize("lanes", [1, 2, 4, 8, 16, 32])
def test_rowgroup_lanes(S, lanes):
    if (S + 6) // 4 > 8 * lanes:
        pytest.skip("row too long for this many lanes")
    x, mask = _rand(1, 3, S, 11 * S + lanes, "neg_1e9")
    p, em = run_attention(x, mask, True, variant="rowgroup", param=lanes,
                          offsets=(2, 1, 3))
    compare_full(x, mask, True, p, em)


@pytest.mark.parametrize("S", [3, 64, 513, 2048, 8192])
@pytest.mark.parametrize("threads", [0, 64, 512])
def test_row_cta(S, threads):
    B, H = (1, 1) if S >= 8192 else (2, 2)
    x, mask = _rand(B, H, S, 13 * S + threads, "neg_inf")
    p, em = run_attention(x, mask, S % 2 == 0, variant="cluster",
                          threads=threads)
    if S >= 8192:
        pf, xf = p.reshape(-1, S), x.reshape(-1, S)
        for r in (0, 1, S // 2, S - 1):
            ref, flag = oracle.attention_softmax_row(xf[r], r, mask[0], True)
            compare_rows(pf[r:r + 1], xf[r:r + 1], np.array([r]),
                         mask[0:1], True, ref[None], np.array([flag]))
    else:
        compare_full(x, mask, S % 2 == 0, p, em)


@pytest.mark.parametrize("variant,S", [("rowgroup", 64), ("rowgroup", 512),
                                       ("cluster", 512), ("cluster", 3001)])
def test_in_place(variant, S):
    x, mask = _rand(2, 2, S, 3 * S, "neg_1e9")
    p, em = run_attention(x, mask, True, variant=variant, inplace=True)
    compare_full(x, mask, True, p, em)


@pytest.mark.parametrize("variant,S", [("rowgroup", 64), ("cluster", 64),
                                       ("cluster", 2048)])
def test_nan_inf_and_fully_masked(variant, S):
    """NaN (flag 1) and +-Inf (flag 2) in used scores or mask values zero
    their rows; a NaN under the causal mask is never read; a batch whose
    mask removes every key gives zero rows without a flag."""
    x, mask = _rand(3, 2, S, 17 * S, "neg_1e9")
    x[0, 0, 5, 3] = np.nan
    x[0, 1, 2, 9] = np.nan          # key 9 > query 2
    x[1, 0, 7, 0] = np.inf
    x[1, 1, 4, 4] = -np.inf
    mask[2, :] = -np.inf
    p, em = run_attention(x, mask, True, variant=variant)
    compare_full(x, mask, True, p, em)
    assert em == (1 << 1) | (1 << 2)
    assert np.all(p[2] == 0.0) and np.all(p[0, 0, 5] == 0.0)
    assert abs(p[0, 1, 2].sum() - 1.0) < 1e-5
    m2 = mask.copy()
    m2[1, 3] = np.nan
    p2, em2 = run_attention(x[:2], m2[:2], False, variant=variant)
    compare_full(x[:2], m2[:2], False, p2, em2)
    assert np.all(p2[1] == 0.0)


def test_argument_errors_and_empty():
    import torch
    import entropy_bounded_softmax_gb300 as cs
    dev = torch.device("cuda", 0)
    z = torch.zeros((0, 2, 4, 4), device=dev)
    assert cs.attention_softmax(z).shape == (0, 2, 4, 4)
    x = torch.randn(2, 2, 8, 8, device=dev)
    with pytest.raises(cs.CsError) as e:
        cs.attention_softmax(x, variant="rowgroup", param=3)
    assert e.value.status == 8
    with pytest.raises(cs.CsError) as e:
        cs.attention_softmax(x, variant="cluster", param=2)
    assert e.value.status == 8
    buf = torch.zeros(300, device=dev)
    with pytest.raises(cs.CsError) as e:
        cs.attention_softmax(buf[:256].view(2, 2, 8, 8),
                             out=buf[4:260].view(2, 2, 8, 8))
    assert e.value.status == 8
    assert cs.cs_attention_softmax(x.data_ptr(), x.data_ptr(), None, 2, 2, 8,
                                   2, None) == 8
    assert cs.cs_attention_softmax(x.data_ptr(), x.data_ptr(), None, 1, 1,
                                   60000, 0, None) == 7
