"""Helpers for the backward's GPU-vs-oracle parity tests.

Inputs: the workload's logits l, its seeded (g, T) and p = softmax(l / T)
from the oracle (rows with T NaN get p = 0, as the forward writes them).
The same fp32 p, g and T go to the kernel and, promoted exactly to fp64,
to the oracle.

Acceptance, element by element:
    |grad_gpu - grad_oracle| <= (p / T) (EPS_DOT sum_j |p_j g_j|
                                         + 4 u |g - <g, p>|) + 2^-126
with u = 2^-24.  The kernel sums the row's dot product in fp32; a sum of n
terms carries at most gamma_n = n u / (1 - n u) of sum |p_j g_j| in error,
and EPS_DOT = 1e-5 is gamma_n for n = 167, well above the longest chain of
additions in any plan (a thread's float4s, then shuffle, warp and rank
sums: under 70 at 850000 classes).  4 u covers the three roundings of
(p * (1/T)) * (g - dot) and the reciprocal.  Rows with T NaN must be exactly
zero; a NaN in the oracle's output must be NaN on the GPU too, and an
infinity the same infinity.
"""
from __future__ import annotations

from concurrent.futures import ThreadPoolExecutor

import numpy as np

import oracle

EPS_DOT = 1e-5
U = 2.0 ** -24
ATOL = 2.0 ** -126


def probs_for(x: np.ndarray, T: np.ndarray) -> np.ndarray:
    """fp32 p = softmax(l / T) by the oracle, zeros where T is not a
    positive finite number."""
    p = np.zeros(x.shape, dtype=np.float32)

    def row(r):
        t = float(T[r])
        if t > 0.0 and np.isfinite(t):
            p[r] = oracle.softmax(x[r], t).astype(np.float32)

    with ThreadPoolExecutor(max_workers=oracle.default_threads()) as pool:
        list(pool.map(row, range(x.shape[0])))
    return p


def tolerance(p: np.ndarray, g: np.ndarray, T: np.ndarray) -> np.ndarray:
    p64 = p.astype(np.float64)
    g64 = g.astype(np.float64)
    T64 = T.astype(np.float64)
    dot = np.sum(p64 * g64, axis=1, keepdims=True)
    absdot = np.sum(np.abs(p64 * g64), axis=1, keepdims=True)
    with np.errstate(invalid="ignore", divide="ignore"):
        tol = (p64 / T64[:, None]) * (EPS_DOT * absdot
                                      + 4 * U * np.abs(g64 - dot))
    ok = (T64 > 0) & np.isfinite(T64)
    tol[~ok] = 0.0
    return tol + ATOL


def compare(grad_gpu: np.ndarray, p: np.ndarray, g: np.ndarray,
            T: np.ndarray) -> dict:
    """Asserts parity; returns the largest error relative to its bound."""
    ref = oracle.constrained_softmax_backward(p, g, T)
    bad_T = ~((T > 0) & np.isfinite(T))
    assert np.all(grad_gpu[bad_T] == 0.0), "rows without a valid T not zero"
    nan_ref = np.isnan(ref)
    assert np.array_equal(np.isnan(grad_gpu), nan_ref), "NaN pattern differs"
    inf_ref = np.isinf(ref)
    assert np.array_equal(grad_gpu[inf_ref], ref[inf_ref]), "Inf differs"
    tol = tolerance(p, g, T)
    with np.errstate(invalid="ignore"):
        err = np.abs(grad_gpu.astype(np.float64) - ref)
    err[nan_ref | inf_ref] = 0.0
    assert np.all(np.isfinite(err))
    worst = float(np.max(err / tol)) if err.size else 0.0
    if worst > 1.0:
        i = np.unravel_index(np.argmax(err / tol), err.shape)
        raise AssertionError(f"grad {grad_gpu[i]} vs {ref[i]} at {i}: error "
                             f"{err[i]:.3e} > bound {tol[i]:.3e}")
    return {"worst_fraction_of_bound": worst}


def run_backward(p: np.ndarray, g: np.ndarray, T: np.ndarray,
                 variant="auto", param=0, threads=0, offsets=(0, 0, 0),
                 inplace=None) -> np.ndarray:
    """The CUDA backward through the C ABI.  offsets shift (p, g, grad) by
    that many floats inside their allocations; inplace = "probs" or
    "grad_output" writes the gradient over that input."""
    import torch
    import entropy_bounded_softmax_gb300 as cs
    B, C = p.shape
    n = B * C
    dev = torch.device("cuda", 0)

    def place(a, off, fill=None):
        buf = torch.full((n + off + 4,), -7.0, dtype=torch.float32,
                         device=dev)
        view = buf[off:off + n].view(B, C)
        if a is not None:
            view.copy_(torch.from_numpy(np.ascontiguousarray(a)))
        return buf, view

    bp, tp = place(p, offsets[0])
    bg, tg = place(g, offsets[1])
    if inplace == "probs":
        bo, to, off_o = bp, tp, offsets[0]
    elif inplace == "grad_output":
        bo, to, off_o = bg, tg, offsets[1]
    else:
        bo, to = place(None, offsets[2])
        off_o = offsets[2]
    tt = torch.from_numpy(np.ascontiguousarray(T)).to(dev)
    cs.constrained_softmax_backward(tp, tg, tt, out=to, variant=variant,
                                    param=param, threads=threads)
    torch.cuda.synchronize()
    assert torch.all(bo[:off_o] == -7.0)
    assert torch.all(bo[off_o + n:] == -7.0)
    return to.cpu().numpy()
