"""Helpers for the biencoder_attention GPU-vs-oracle parity tests.

Step 1's fp32 scores are fixed by the reading both sides follow (one fused
multiply-add per d in order, then * scale), so the GPU's logits equal the
oracle's bit for bit and steps 2-3 reuse the constrained softmax's
acceptance (tests/gpu_parity.py): the weights and temperatures row by row,
with the oracle's softmax at the GPU's temperature where the two settle on
different grid points.  The output is then compared with those reference
weights times the values in fp64:

    |out_gpu - out_ref| <= 2e-5 sum_j |v_jd| + 1e-5 sum_j p_j |v_jd| + 1e-30

(the weights' own tolerance, 2e-5 each, carried through the sum, plus the
fp32 accumulation of K <= 256 products, below 1e-5 of sum p |v|).
"""
from __future__ import annotations

import numpy as np

import oracle
from gpu_parity import compare


def run_biencoder(q, k, v, scale, entropy_bound=0.2, t_min=0.01, t_max=10.0,
                  max_iter=20, lanes=0):
    """The CUDA path through the C ABI; returns (out, attn, T, error mask)."""
    import torch
    import entropy_bounded_softmax_gb300 as cs
    dev = torch.device("cuda", 0)
    qd, kd, vd = (torch.from_numpy(np.ascontiguousarray(a)).to(dev)
                  for a in (q, k, v))
    cs.get_error()
    out, attn, T = cs.biencoder_attention(qd, kd, vd, scale, entropy_bound,
                                          t_min, t_max, max_iter,
                                          return_attn=True, return_t=True,
                                          lanes=lanes)
    bits = cs.get_error()
    mask = 0
    for name, bit in cs.ERROR_BITS.items():
        if name in bits:
            mask |= bit
    return out.cpu().numpy(), attn.cpu().numpy(), T.cpu().numpy(), mask


def compare_biencoder(q, k, v, scale, out, attn, T, mask, entropy_bound=0.2,
                      t_min=0.01, t_max=10.0, max_iter=20) -> dict:
    ref = oracle.biencoder_attention(q, k, v, scale, entropy_bound, t_min,
                                     t_max, max_iter)
    B, H, Q, K = ref.scores.shape
    D = q.shape[3]
    x = ref.scores.reshape(-1, K)
    Tg = T.reshape(-1)
    stats = compare(x, attn.reshape(-1, K), Tg, mask, ref.attn,
                    entropy_bound, t_min, t_max, max_iter)
    p = ref.attn.p.copy()
    for r in np.flatnonzero(ref.attn.flags == 0):
        if float(Tg[r]) != float(np.float32(ref.attn.T[r])):
            p[r] = oracle.softmax(x[r], float(Tg[r]))
    p = p.reshape(B, H, Q, K)
    v64 = v.astype(np.float64)
    o_ref = np.einsum("bhqk,bhkd->bhqd", p, v64)
    tol = (2e-5 * np.abs(v64).sum(axis=2)[:, :, None, :]
           + 1e-5 * np.einsum("bhqk,bhkd->bhqd", p, np.abs(v64)) + 1e-30)
    err = np.abs(out.astype(np.float64) - o_ref)
    worst = float(np.max(err / tol)) if err.size else 0.0
    if worst > 1.0:
        i = np.unravel_index(np.argmax(err / tol), err.shape)
        raise AssertionError(f"out {out[i]} vs {o_ref[i]} at {i}: error "
                             f"{err[i]:.3e} > bound {tol[i]:.3e}")
    stats["out_worst_fraction_of_bound"] = worst
    return stats
