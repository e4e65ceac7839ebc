"""Helpers for the GPU-vs-oracle parity tests.

Acceptance (per row, on the same seeded inputs):
  * the temperature: equal to the oracle's (as fp32), or within one final
    bisection interval plus 4 fp32 ulps of it.  Only for max_iter > 24,
    where the final interval is finer than fp32 resolves over most of
    [t_min, 1] and the GPU's grid is the fp32 numbers themselves, a third
    case is accepted: an endpoint that a bisection whose H is exact to
    EPS_H would also return, H(T_gpu) <= bound + EPS_H and
    H(T_gpu + interval + 4 ulps) >= bound - EPS_H, with H the oracle's fp64
    entropy.  When T differs, the GPU's probabilities are compared with
    the oracle's fp64 softmax(l / T_gpu);
  * the row's status: the oracle flags the bound unsatisfiable (section
    5.4) exactly when the GPU's T is t_min and the fp64 H there exceeds the
    bound;
  * probabilities: elementwise |dp| <= 2e-5;
  * entropy of the output (fp64, scipy.special.entr): |dH| <= 1e-4, and
    H(out) <= bound + 1e-4 whenever the oracle found the bound achievable;
  * the error mask of the launch equals the OR of the oracle's row flags
    (for launches compared on sampled rows, the flags of every row follow
    from H(1) and H(t_min) alone: see launch_flags);
  * NaN/Inf rows: all zeros and T = NaN.
"""
from __future__ import annotations

import math

import numpy as np
import scipy.special

import oracle

P_TOL = 2e-5
H_TOL = 1e-4
T_ULPS = 4
EPS_H = 1e-6
# Above this many halvings the grid is the fp32 numbers of the interval.
FINE_GRID_ITERS = 24

ERR_BIT = {1: 1 << 1, 2: 1 << 2, 3: 1 << 3}
TIMEOUT_BIT = 1 << 10


def run_gpu(x: np.ndarray, entropy_bound=0.2, t_min=0.01, t_max=10.0,
            max_iter=20, variant="auto", param=0, in_offset=0, out_offset=0,
            threads=0, strict=False):
    """Runs the CUDA path through the C ABI; returns (p, T, error_mask).
    in_offset/out_offset shift the tensors by that many floats inside their
    allocations (to exercise unaligned rows)."""
    import torch
    import entropy_bounded_softmax_gb300 as cs
    B, C = x.shape
    n = B * C
    dev = torch.device("cuda", 0)
    buf_in = torch.empty(n + in_offset + 4, dtype=torch.float32, device=dev)
    xin = buf_in[in_offset:in_offset + n].view(B, C)
    xin.copy_(torch.from_numpy(np.ascontiguousarray(x)))
    buf_out = torch.full((n + out_offset + 4,), -7.0, dtype=torch.float32,
                         device=dev)
    out = buf_out[out_offset:out_offset + n].view(B, C)
    t_out = torch.full((B,), -3.0, dtype=torch.float32, device=dev)
    cs.get_error()  # clear
    cs.constrained_softmax(xin, entropy_bound, t_min, t_max, max_iter,
                           out=out, t_out=t_out, variant=variant,
                           param=param, threads=threads, strict=strict)
    bits = cs.get_error()
    mask = 0
    for name, bit in cs.ERROR_BITS.items():
        if name in bits:
            mask |= bit
    # Guard words around the output must be untouched.
    assert torch.all(buf_out[:out_offset] == -7.0)
    assert torch.all(buf_out[out_offset + n:] == -7.0)
    return out.cpu().numpy(), t_out.cpu().numpy(), mask


def run_gpu_bf16(bits: np.ndarray, entropy_bound=0.2, t_min=0.01,
                 t_max=10.0, max_iter=20, variant="auto", param=0,
                 in_offset=0, out_offset=0, threads=0, strict=False):
    """run_gpu for bf16 logits given as uint16 patterns (in_offset in bf16
    elements); returns (p, T, error_mask)."""
    import torch
    import entropy_bounded_softmax_gb300 as cs
    B, C = bits.shape
    n = B * C
    dev = torch.device("cuda", 0)
    buf_in = torch.empty(n + in_offset + 8, dtype=torch.bfloat16, device=dev)
    xin = buf_in[in_offset:in_offset + n].view(B, C)
    xin.copy_(torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
              .view(torch.bfloat16))
    buf_out = torch.full((n + out_offset + 4,), -7.0, dtype=torch.float32,
                         device=dev)
    out = buf_out[out_offset:out_offset + n].view(B, C)
    t_out = torch.full((B,), -3.0, dtype=torch.float32, device=dev)
    cs.get_error()  # clear
    cs.constrained_softmax(xin, entropy_bound, t_min, t_max, max_iter,
                           out=out, t_out=t_out, variant=variant,
                           param=param, threads=threads, strict=strict)
    bits_err = cs.get_error()
    mask = 0
    for name, bit in cs.ERROR_BITS.items():
        if name in bits_err:
            mask |= bit
    assert torch.all(buf_out[:out_offset] == -7.0)
    assert torch.all(buf_out[out_offset + n:] == -7.0)
    return out.cpu().numpy(), t_out.cpu().numpy(), mask


def entropy64(p: np.ndarray) -> np.ndarray:
    return scipy.special.entr(p.astype(np.float64)).sum(axis=-1)


def t_tolerance(T: float, t_min: float, t_max: float, max_iter: int) -> float:
    w = oracle.final_interval(t_min, t_max, max_iter)
    return w + T_ULPS * float(np.spacing(np.float32(T)))


def compare(x: np.ndarray, p_gpu: np.ndarray, T_gpu: np.ndarray, mask: int,
            ref: oracle.Result, entropy_bound=0.2, t_min=0.01, t_max=10.0,
            max_iter=20, check_mask=True, p_slack=None) -> dict:
    """Asserts parity row by row; returns summary statistics (the
    T_zone count, rows accepted by the third temperature case, is always
    0 for max_iter <= FINE_GRID_ITERS).  p_slack (per row, optional) widens
    the probability tolerance to P_TOL + p_slack[b] * p element by element,
    for callers whose GPU logits differ from the oracle's by a known
    rounding."""
    B = x.shape[0]
    bound32 = float(np.float32(entropy_bound))
    tmin32 = float(np.float32(t_min))
    fine = int(max_iter) > FINE_GRID_ITERS
    stats = {"rows": B, "T_equal": 0, "T_within": 0, "T_zone": 0,
             "max_dp": 0.0,
             "max_dH": 0.0}
    want_mask = 0
    for b in range(B):
        f = int(ref.flags[b])
        if f:
            want_mask |= ERR_BIT[f]
        if f in (1, 2):
            assert math.isnan(T_gpu[b]), (b, T_gpu[b])
            assert np.all(p_gpu[b] == 0.0), b
            continue
        To = ref.T[b]
        Tg = float(T_gpu[b])
        # Section 5.4 status of the row: unsatisfiable in the oracle exactly
        # when the GPU settled on t_min and fp64 H there exceeds the bound.
        gpu_overflow = Tg == tmin32 and oracle.entropy(x[b], Tg) > bound32
        assert (f == 3) == gpu_overflow, (
            f"row {b}: oracle flag {f}, T_gpu={Tg!r}, t_min={tmin32!r}")
        if Tg == float(np.float32(To)):
            stats["T_equal"] += 1
            p_ref = ref.p[b]
        else:
            tol = t_tolerance(To, t_min, t_max, max_iter)
            if abs(Tg - To) <= tol:
                stats["T_within"] += 1
            else:
                assert fine, (
                    f"row {b}: T_gpu={Tg!r} T_oracle={To!r} differ by "
                    f"{abs(Tg - To):.3g} > one final interval + "
                    f"{T_ULPS} ulps ({tol:.3g}) at max_iter={max_iter}")
                H_at = oracle.entropy(x[b], Tg)
                H_up = oracle.entropy(x[b], Tg + t_tolerance(Tg, t_min, t_max,
                                                             max_iter))
                assert H_at <= bound32 + EPS_H and H_up >= bound32 - EPS_H, (
                    f"row {b}: T_gpu={Tg!r} T_oracle={To!r} tol={tol:.3g} "
                    f"H(T_gpu)-bound={H_at - bound32:.3g} "
                    f"H(T_gpu+w)-bound={H_up - bound32:.3g}")
                stats["T_zone"] += 1
            p_ref = oracle.softmax(x[b], Tg)
        err = np.abs(p_gpu[b].astype(np.float64) - p_ref)
        dp = float(np.max(err))
        if p_slack is None:
            assert dp <= P_TOL, f"row {b}: max |dp| = {dp:.3g}"
        else:
            lim = P_TOL + float(p_slack[b]) * p_ref
            assert np.all(err <= lim), (
                f"row {b}: |dp| {dp:.3g} above {P_TOL} + {float(p_slack[b]):.3g} p")
        Hg = float(entropy64(p_gpu[b]))
        Hr = float(entropy64(p_ref))
        dH = abs(Hg - Hr)
        assert dH <= H_TOL, f"row {b}: |dH| = {dH:.3g}"
        if f == 0:
            assert Hg <= bound32 + H_TOL or ref.T[b] == 1.0, \
                f"row {b}: H(out)={Hg} above bound"
        s = float(np.sum(p_gpu[b], dtype=np.float64))
        assert abs(s - 1.0) <= 1e-5, f"row {b}: sum p = {s}"
        stats["max_dp"] = max(stats["max_dp"], dp)
        stats["max_dH"] = max(stats["max_dH"], dH)
    if check_mask:
        assert mask == want_mask, f"error mask {mask:#x} != oracle {want_mask:#x}"
    print(f"parity: {stats}")
    return stats


def launch_flags(x: np.ndarray, entropy_bound=0.2, t_min=0.01,
                 t_max=10.0) -> tuple[np.ndarray, np.ndarray]:
    """The oracle's section 5.1 flag of every row without running its
    search, plus each row's margin |H(t_min) - bound| (nats; inf where the
    flag does not depend on it).  NaN rows flag 1, other non-finite rows 2;
    otherwise the bisection ends unsatisfiable (flag 3) exactly when H(1)
    and H(t_min) both exceed the bound: H is nondecreasing in T, so every
    midpoint is then infeasible and lo stays at t_min, while H(t_min) within
    the bound keeps lo feasible."""
    bound32 = float(np.float32(entropy_bound))
    tmin32 = float(np.float32(t_min))
    flags = np.zeros(x.shape[0], dtype=np.int32)
    margin = np.full(x.shape[0], np.inf)

    def one(b: int) -> None:
        row = x[b]
        if np.isnan(row).any():
            flags[b] = 1
            return
        if not np.isfinite(row).all():
            flags[b] = 2
            return
        if oracle.entropy(row, 1.0) <= bound32:
            return
        h = oracle.entropy(row, tmin32)
        margin[b] = abs(h - bound32)
        if h > bound32:
            flags[b] = 3

    from concurrent.futures import ThreadPoolExecutor
    oracle.load()
    with ThreadPoolExecutor(max_workers=oracle.default_threads()) as pool:
        list(pool.map(one, range(x.shape[0])))
    return flags, margin


def check_launch_status(x: np.ndarray, T_gpu: np.ndarray, mask: int,
                        entropy_bound=0.2, t_min=0.01, t_max=10.0) -> dict:
    """Per-row status over a whole launch compared on sampled rows: every
    row the oracle would flag unsatisfiable has T_gpu = t_min, every
    NaN/Inf row T_gpu = NaN, and the launch's error mask is the OR of the
    rows' flags.  Rows whose H(t_min) lies within EPS_H of the bound could
    go either way in fp32; the overflow bit is then not checked."""
    flags, margin = launch_flags(x, entropy_bound, t_min, t_max)
    tmin32 = np.float32(t_min)
    clear = margin > EPS_H
    over = flags == 3
    bad = np.flatnonzero(over & clear & (T_gpu != tmin32))
    assert bad.size == 0, f"rows {bad[:8]} unsatisfiable but T_gpu != t_min"
    nonfin = (flags == 1) | (flags == 2)
    assert np.all(np.isnan(T_gpu[nonfin]))
    want = 0
    for f in (1, 2, 3):
        if np.any(flags == f):
            want |= ERR_BIT[f]
    if np.all(clear):
        assert mask == want, f"error mask {mask:#x} != rows' flags {want:#x}"
    else:
        keep = ~ERR_BIT[3]
        assert mask & keep == want & keep, \
            f"error mask {mask:#x} != rows' flags {want:#x}"
    return {"flagged_overflow": int(over.sum()), "ambiguous": int((~clear).sum())}
