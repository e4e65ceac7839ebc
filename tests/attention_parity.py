"""Helpers for the attention_softmax GPU-vs-oracle parity tests.

Both sides take the same fp32 scores and mask.  Acceptance, element by
element, with v = fl32(s + m) the masked score, m* the row's max and
y = (v - m*) log2 e from the oracle's values:

    |p_gpu - p_oracle| <= p_oracle (2e-6 + 1.3e-7 |y|) + 2^-125

The GPU forms y as fl(fl(v - m*) log2e) (two roundings, plus log2 e
rounded to fp32: about 3u|y| in the exponent, 3u ln2 |y| = 1.24e-7 |y|
relative in 2^y), takes 2^y on the ex2 unit (2 ulp, 2.4e-7), sums in fp32
(chains of at most 64 terms plus a 5-level butterfly or a 16-slot sum:
below 1e-6 relative) and scales by the correctly rounded reciprocal (2
roundings).  2^-125 covers results the ex2 unit flushes to zero (2^y below
2^-126).  Removed keys must be exactly 0, NaN/Inf rows all zero, and the
launch's error bits the OR of the oracle's row flags.
"""
from __future__ import annotations

import numpy as np

import oracle

LOG2E = 1.4426950408889634
ATOL = 2.0 ** -125


def tolerance(x: np.ndarray, mask, causal: bool, ref_p: np.ndarray,
              rows_i: np.ndarray, mask_rows) -> np.ndarray:
    """x [n, S] scores rows, rows_i [n] their query indices, mask_rows
    [n, S] or None."""
    v = x if mask_rows is None else (x + mask_rows)          # fp32 addition
    v = v.astype(np.float64)
    S = x.shape[1]
    if causal:
        keep = np.arange(S)[None, :] <= rows_i[:, None]
        v = np.where(keep, v, -np.inf)
    with np.errstate(invalid="ignore"):
        vmax = np.max(np.where(np.isfinite(v), v, -np.inf), axis=1,
                      keepdims=True)
        y = np.abs((v - vmax) * LOG2E)
    y[~np.isfinite(y)] = 0.0
    return ref_p * (2e-6 + 1.3e-7 * y) + ATOL


def compare_rows(p_gpu: np.ndarray, x: np.ndarray, rows_i: np.ndarray,
                 mask_rows, causal: bool, ref_p: np.ndarray,
                 ref_flags: np.ndarray) -> float:
    """Asserts parity of rows; returns the worst error over its bound."""
    bad = ref_flags != 0
    assert np.all(p_gpu[bad] == 0.0), "NaN/Inf rows not zero"
    assert np.all(p_gpu[ref_p == 0.0] == 0.0), "removed keys not zero"
    tol = tolerance(x, mask_rows is not None, causal, ref_p, rows_i,
                    mask_rows)
    err = np.abs(p_gpu.astype(np.float64) - ref_p)
    worst = float(np.max(err / tol)) if err.size else 0.0
    if worst > 1.0:
        k = np.unravel_index(np.argmax(err / tol), err.shape)
        raise AssertionError(f"p {p_gpu[k]} vs {ref_p[k]} at {k}: error "
                             f"{err[k]:.3e} > bound {tol[k]:.3e}")
    return worst


def run_attention(x: np.ndarray, mask, causal: bool, variant="auto",
                  param=0, threads=0, offsets=(0, 0, 0), inplace=False):
    """The CUDA path through the C ABI on scores x [B, H, S, S]; returns
    (p [B, H, S, S], error mask).  offsets shift (scores, out, mask) by
    that many floats inside their allocations; guard words around the
    output must survive."""
    import torch
    import entropy_bounded_softmax_gb300 as cs
    B, H, S, _ = x.shape
    n = x.size
    dev = torch.device("cuda", 0)
    bs = torch.full((n + offsets[0] + 4,), -7.0, dtype=torch.float32,
                    device=dev)
    xs = bs[offsets[0]:offsets[0] + n].view(B, H, S, S)
    xs.copy_(torch.from_numpy(np.ascontiguousarray(x)))
    if inplace:
        bo, out, oo = bs, xs, offsets[0]
    else:
        bo = torch.full((n + offsets[1] + 4,), -7.0, dtype=torch.float32,
                        device=dev)
        out = bo[offsets[1]:offsets[1] + n].view(B, H, S, S)
        oo = offsets[1]
    md = None
    if mask is not None:
        bm = torch.zeros(B * S + offsets[2] + 4, dtype=torch.float32,
                         device=dev)
        md = bm[offsets[2]:offsets[2] + B * S].view(B, S)
        md.copy_(torch.from_numpy(np.ascontiguousarray(mask)))
    cs.get_error()
    cs.attention_softmax(xs, md, causal, out=out, variant=variant,
                         param=param, threads=threads)
    bits = cs.get_error()
    em = 0
    for name, bit in cs.ERROR_BITS.items():
        if name in bits:
            em |= bit
    assert torch.all(bo[:oo] == -7.0) and torch.all(bo[oo + n:] == -7.0)
    return out.cpu().numpy(), em


def expected_mask(flags: np.ndarray) -> int:
    em = 0
    if np.any(flags == 1):
        em |= 1 << 1
    if np.any(flags == 2):
        em |= 1 << 2
    return em


def compare_full(x: np.ndarray, mask, causal: bool, p_gpu: np.ndarray,
                 err_mask: int) -> float:
    """Whole-tensor parity, one batch at a time."""
    B, H, S, _ = x.shape
    worst = 0.0
    flags_all = []
    for b in range(B):
        mb = None if mask is None else mask[b:b + 1]
        ref = oracle.attention_softmax(x[b:b + 1], mb, causal)
        flags_all.append(ref.flags)
        rows_i = np.tile(np.arange(S), H)
        mrows = None if mask is None else np.repeat(mask[b:b + 1], H * S, 0)
        worst = max(worst, compare_rows(
            p_gpu[b].reshape(H * S, S), x[b].reshape(H * S, S), rows_i,
            mrows, causal, ref.p[0].reshape(H * S, S),
            ref.flags[0].reshape(H * S)))
    assert err_mask == expected_mask(np.concatenate([f.reshape(-1) for f in flags_all]))
    return worst
