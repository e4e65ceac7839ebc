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
                  max_iter=20, lanes=0, fused=False, return_attn=True):
    """The CUDA path through the C ABI; returns (out, attn, T, error mask)
    (attn None when not requested: then the weights pass through the
    output buffer on the tensor-core path)."""
    import torch
    import entropy_bounded_softmax_gb300 as cs
    dev = torch.device("cuda", 0)
    qd, kd, vd = (torch.from_numpy(np.ascontiguousarray(a)).to(dev)
                  for a in (q, k, v))
    cs.get_error()
    res = cs.biencoder_attention(qd, kd, vd, scale, entropy_bound,
                                 t_min, t_max, max_iter,
                                 return_attn=return_attn, return_t=True,
                                 lanes=lanes, fused=fused)
    if return_attn:
        out, attn, T = res
    else:
        (out, T), attn = res, None
    bits = cs.get_error()
    mask = 0
    for name, bit in cs.ERROR_BITS.items():
        if name in bits:
            mask |= bit
    return (out.cpu().numpy(), None if attn is None else attn.cpu().numpy(),
            T.cpu().numpy(), mask)


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


def compare_biencoder_fp64_scores(q, k, v, scale, out, attn, T, mask,
                                  entropy_bound=0.2, t_min=0.01, t_max=10.0,
                                  max_iter=20) -> dict:
    """The same acceptance with the oracle's search run on scores from an
    fp64 matmul rounded once to fp32 (independent of the fixed fp32
    evaluation order the kernel and the oracle's own scores share).  The
    temperatures must pass the forward's acceptance unchanged.  The
    kernel's scores differ from these by at most
    ds = (D + 2) u sum_d |q_d k_d| scale (u = 2^-24; the error of an
    in-order fma chain plus the scale and the final rounding), which moves
    each x_j = s_j / T by beta ds and each weight by at most
    p_i (|dx_i| + sum_j p_j |dx_j|) <= 2 p_i beta max_j ds_j; the weights
    are accepted within 2e-5 plus that.  Returns the statistics plus the
    number of rows whose scores differ."""
    B, H, Q, D = q.shape
    K = k.shape[2]
    q64, k64 = q.astype(np.float64), k.astype(np.float64)
    s64 = np.einsum("bhqd,bhkd->bhqk", q64, k64) * float(np.float32(scale))
    x = s64.astype(np.float32).reshape(-1, K)
    ref = oracle.constrained_softmax(x, entropy_bound, t_min, t_max, max_iter)
    Tg = T.reshape(-1)
    mag = np.einsum("bhqd,bhkd->bhqk", np.abs(q64), np.abs(k64)).reshape(-1, K)
    ds = (D + 2) * 2.0 ** -24 * mag.max(axis=1) * abs(float(np.float32(scale)))
    beta = np.where(np.isfinite(Tg) & (Tg > 0), 1.0 / np.where(Tg > 0, Tg, 1.0), 0.0)
    stats = compare(x, attn.reshape(-1, K), Tg, mask, ref, entropy_bound,
                    t_min, t_max, max_iter, p_slack=2.0 * beta * ds)
    fixed = oracle.biencoder_scores(q, k, scale).reshape(-1, K)
    stats["rows_with_other_scores"] = int(np.sum(np.any(fixed != x, axis=1)))
    p = ref.p.copy()
    for r in np.flatnonzero(ref.flags == 0):
        if float(Tg[r]) != float(np.float32(ref.T[r])):
            p[r] = oracle.softmax(x[r], float(Tg[r]))
    p = p.reshape(B, H, Q, K)
    v64 = v.astype(np.float64)
    o_ref = np.einsum("bhqk,bhkd->bhqd", p, v64)
    pv = np.einsum("bhqk,bhkd->bhqd", p, np.abs(v64))
    slack = (2.0 * beta * ds).reshape(B, H, Q)[..., None]
    tol = (2e-5 * np.abs(v64).sum(axis=2)[:, :, None, :]
           + (1e-5 + slack) * pv + 1e-30)
    err = np.abs(out.astype(np.float64) - o_ref)
    worst = float(np.max(err / tol)) if err.size else 0.0
    assert worst <= 1.0, f"output error {worst:.3f} of the bound"
    stats["out_worst_fraction_of_bound"] = worst
    return stats
