"""Pins for the CPU oracle: facts fixed by the mathematics, not by the oracle.

Each ``check_*`` function takes a loaded oracle library and raises
AssertionError when the oracle disagrees with:
  * closed forms of H(T) and of the optimal temperature for 2-class rows and
    for "spike" rows (C-1 equal logits, one larger),
  * a library softmax (scipy) in the case where no search is needed,
  * a brute-force scan of a dense temperature grid on tiny rows, using
    scipy's softmax and entropy routines,
  * invariants (probabilities sum to 1, argmax kept, constant rows uniform,
    shift invariance, H monotone along the search path, C = 1),
  * the NaN/Inf and unsatisfiable-bound policy of "BURT-IMMA CUDA Kernel API
    Reference", sections 5.1, 5.3 and 5.4,
  * for the backward (section 6.3 with the temperature restored): central
    finite differences through the whole forward, search included; the
    vector-Jacobian product of a library softmax (torch autograd, fp64) at
    the forward's temperature; the explicit Jacobian diag(p) - p p^T at
    T = 1; and invariants (gradients sum to 0, shift invariance in the
    upstream gradient, zero rows where T is NaN),
  * for attention_softmax (section 2.6): scipy's softmax of each row, of
    each causal prefix and of the unmasked subset (scores plus mask added
    in numpy fp32); the fp32 addition of a -1e9 mask; invariants and the
    NaN/Inf policy,
  * for biencoder_attention (section 2.5): the fp32 scores against fp64
    matmul within the dot product's rounding bound, one-hot queries, the
    fp32 accumulation order, scipy's softmax and a matmul when no row
    searches, convex combinations of the value rows, a single context item.

The same checks run against deliberately broken copies of the oracle in
``test_oracle_mutants.py``: every plausible mistake must fail at least one.
"""
from __future__ import annotations

import math

import numpy as np
import scipy.optimize
import scipy.special
import scipy.stats

import oracle

T_MIN, T_MAX, ITERS, BOUND = 0.01, 10.0, 20, 0.20


# ---------------------------------------------------------------- closed forms
def h_two_class(delta: float, T: float) -> float:
    """Entropy (nats) of softmax([0, delta] / T): the binary entropy of
    q = sigmoid(delta / T), written with log1p so that it stays accurate when
    q is close to 1."""
    z = abs(delta) / T
    ez = math.exp(-z)
    q = 1.0 / (1.0 + ez)
    one_minus_q = ez / (1.0 + ez)
    lp = math.log1p(ez)              # -ln q
    return q * lp + one_minus_q * (z + lp)


def h_spike(C: int, delta: float, T: float) -> float:
    """Entropy of softmax(l / T) where C-1 logits are equal and one is larger
    by delta > 0: p_top = 1 / (1 + (C-1) e^{-z}), every other p = e^{-z} p_top,
    z = delta / T."""
    z = delta / T
    a = (C - 1) * math.exp(-z)
    p_top = 1.0 / (1.0 + a)
    r = math.exp(-z) / (1.0 + a)
    lp = math.log1p(a)               # -ln p_top
    return p_top * lp + (C - 1) * r * (z + lp)


def t_star(h_of_T, bound: float, lo: float, hi: float) -> float | None:
    """Temperature where the (increasing) closed-form H crosses the bound,
    or None if it does not cross inside (lo, hi)."""
    f = lambda T: h_of_T(T) - bound
    if f(lo) > 0 or f(hi) <= 0:
        return None
    return scipy.optimize.brentq(f, lo, hi, xtol=1e-16, rtol=1e-15,
                                 maxiter=500)


def _f32(x) -> float:
    return float(np.float32(x))


# --------------------------------------------------------------------- checks
def check_two_class_entropy(lib) -> None:
    for delta in (0.125, 0.5, 1.5, 3.0, 7.25):
        for T in (0.01, 0.05, 0.1, 0.37, 1.0, 2.0):
            row = np.array([0.25, 0.25 + delta], dtype=np.float32)
            d = float(row[1]) - float(row[0])
            got = oracle.entropy(row, T, lib=lib)
            want = h_two_class(d, T)
            assert abs(got - want) <= 1e-13 + 1e-12 * want, (delta, T, got, want)


def check_spike_entropy(lib) -> None:
    for C in (3, 10, 1000):
        for delta in (0.5, 2.0, 9.0):
            for T in (0.02, 0.2, 1.0):
                row = np.full(C, -1.5, dtype=np.float32)
                row[C // 3] += np.float32(delta)
                d = float(row[C // 3]) - float(row[0])
                got = oracle.entropy(row, T, lib=lib)
                want = h_spike(C, d, T)
                assert abs(got - want) <= 1e-12 * max(1.0, want), \
                    (C, delta, T, got, want)


def check_large_logits(lib) -> None:
    """Rows of large logits: exp() of them overflows unless the row maximum
    is subtracted first, so this fixes that subtraction."""
    row = np.array([1000.0, 1001.5], dtype=np.float32)
    for T in (0.05, 1.0):
        got = oracle.entropy(row, T, lib=lib)
        assert math.isfinite(got)
        assert abs(got - h_two_class(1.5, T)) < 1e-13
    p = oracle.softmax(row, 1.0, lib=lib)
    assert np.all(np.isfinite(p))
    q = 1.0 / (1.0 + math.exp(-1.5))
    assert abs(p[1] - q) < 1e-15 and abs(p[0] - (1 - q)) < 1e-15
    # A gap of 40 at T = 0.05 puts exp(800) in reach of a wrong shift.
    row = np.array([1000.0, 1040.0], dtype=np.float32)
    for T in (0.05, 1.0):
        got = oracle.entropy(row, T, lib=lib)
        assert math.isfinite(got) and abs(got - h_two_class(40.0, T)) < 1e-13
        p = oracle.softmax(row, T, lib=lib)
        assert np.all(np.isfinite(p)) and abs(p.sum() - 1.0) < 1e-15


def _check_T_against(res_T, Tstar, w, flag, row_desc):
    # The search keeps lo feasible and hi infeasible, so lo lies in
    # (T* - w, T*]; allow relative 1e-11 for fp64 rounding of H near T*.
    slack = 1e-11 * Tstar
    assert flag == 0, row_desc
    assert Tstar - w - slack <= res_T <= Tstar + slack, \
        (row_desc, res_T, Tstar, w)


def check_two_class_temperature(lib) -> None:
    for max_iter in (20, 40, 7):
        w = oracle.final_interval(T_MIN, T_MAX, max_iter)
        lo0, hi0 = oracle.search_interval(T_MIN, T_MAX)
        for delta in (0.05, 0.1, 0.3, 0.9, 2.7):
            row = np.array([0.0, delta], dtype=np.float32)
            d = float(row[1])
            Ts = t_star(lambda T: h_two_class(d, T), _f32(BOUND), lo0, hi0)
            assert Ts is not None
            r = oracle.constrained_softmax(row[None, :], BOUND, T_MIN, T_MAX,
                                           max_iter, threads=1, lib=lib)
            _check_T_against(r.T[0], Ts, w, r.flags[0], (delta, max_iter))
            assert r.iters[0] == max_iter
            q = 1.0 / (1.0 + math.exp(-d / r.T[0]))
            assert abs(r.p[0, 1] - q) < 1e-14 and abs(r.p[0, 0] - (1 - q)) < 1e-14
    # delta = 0.02: even T = t_min leaves H above 0.2 (z = 2 gives
    # h_b(sigmoid(2)) = 0.36), so the bound is unsatisfiable.
    row = np.array([[0.0, 0.02]], dtype=np.float32)
    assert h_two_class(float(row[0, 1]), _f32(T_MIN)) > _f32(BOUND)
    r = oracle.constrained_softmax(row, BOUND, T_MIN, T_MAX, ITERS, threads=1,
                                   lib=lib)
    assert r.flags[0] == oracle.FLAG_ENTROPY_OVERFLOW and r.T[0] == _f32(T_MIN)


def check_spike_temperature(lib) -> None:
    w = oracle.final_interval(T_MIN, T_MAX, ITERS)
    lo0, hi0 = oracle.search_interval(T_MIN, T_MAX)
    for C, delta, bound in ((5, 1.0, 0.2), (64, 3.0, 0.2), (1000, 4.0, 0.5),
                            (50000, 6.0, 0.2), (7, 0.7, 1.0)):
        row = np.zeros(C, dtype=np.float32)
        row[C - 2] = delta
        d = float(row[C - 2])
        Ts = t_star(lambda T: h_spike(C, d, T), _f32(bound), lo0, hi0)
        assert Ts is not None, (C, delta, bound)
        r = oracle.constrained_softmax(row[None, :], bound, T_MIN, T_MAX,
                                       ITERS, threads=1, lib=lib)
        _check_T_against(r.T[0], Ts, w, r.flags[0], (C, delta, bound))


def check_softmax_special_case(lib) -> None:
    """A bound at or above H(1) needs no search: the output is the plain
    softmax, which scipy computes independently."""
    rng = np.random.default_rng(11)
    for C in (1, 2, 17, 1000):
        x = rng.normal(0.0, 2.0, size=(3, C)).astype(np.float32)
        for bound in (math.log(C) + 0.5, 1e30):
            r = oracle.constrained_softmax(x, bound, T_MIN, T_MAX, ITERS,
                                           threads=1, lib=lib)
            ref = scipy.special.softmax(x.astype(np.float64), axis=1)
            assert np.all(r.T == 1.0) and np.all(r.flags == 0)
            assert np.all(r.iters == 0)
            assert np.max(np.abs(r.p - ref)) < 1e-15
    # Bounds a hair above and below H(1) of a 2-class row: the first must
    # give T = 1 exactly, the second must search (T < 1).
    for delta in (1.0, 3.0, 5.0):
        row = np.array([[0.0, delta]], dtype=np.float32)
        H1 = h_two_class(delta, 1.0)
        above = np.nextafter(np.float32(H1), np.float32(1.0))
        below = np.nextafter(np.float32(H1), np.float32(0.0))
        if float(above) < H1:
            above = np.nextafter(above, np.float32(1.0))
        if float(below) >= H1:
            below = np.nextafter(below, np.float32(0.0))
        r = oracle.constrained_softmax(row, float(above), T_MIN, T_MAX, ITERS,
                                       threads=1, lib=lib)
        assert r.T[0] == 1.0 and r.iters[0] == 0
        r = oracle.constrained_softmax(row, float(below), T_MIN, T_MAX, ITERS,
                                       threads=1, lib=lib)
        assert r.T[0] < 1.0 and r.iters[0] == ITERS


def _grid_largest_feasible(row: np.ndarray, bound: float, lo: float,
                           hi: float, n: int):
    T = np.linspace(lo, hi, n)
    p = scipy.special.softmax(row.astype(np.float64)[None, :] / T[:, None],
                              axis=1)
    H = scipy.stats.entropy(p, axis=1)
    ok = np.flatnonzero(H <= bound)
    return (T[ok[-1]] if ok.size else None), T[1] - T[0]


def check_brute_force(lib) -> None:
    rng = np.random.default_rng(5)
    lo0, hi0 = oracle.search_interval(T_MIN, T_MAX)
    w = oracle.final_interval(T_MIN, T_MAX, ITERS)
    n = 1_000_000
    seen_search = seen_overflow = 0
    for trial in range(8):
        C = int(rng.integers(2, 9))
        row = rng.normal(0.0, 0.4 + 0.3 * trial, size=C).astype(np.float32)
        bound = _f32([0.2, 0.35, 0.6, 0.1][trial % 4])
        r = oracle.constrained_softmax(row[None, :], bound, T_MIN, T_MAX,
                                       ITERS, threads=1, lib=lib)
        H1 = scipy.stats.entropy(scipy.special.softmax(row.astype(np.float64)))
        if H1 <= bound:
            assert r.T[0] == 1.0 and r.flags[0] == 0
            continue
        Tg, dT = _grid_largest_feasible(row, bound, lo0, hi0, n)
        if Tg is None:
            seen_overflow += 1
            assert r.flags[0] == oracle.FLAG_ENTROPY_OVERFLOW
            assert r.T[0] == lo0
        else:
            seen_search += 1
            assert r.flags[0] == 0
            assert abs(r.T[0] - Tg) <= dT + w + 1e-12, (trial, r.T[0], Tg)
    assert seen_search >= 4


def check_invariants(lib) -> None:
    rng = np.random.default_rng(3)
    x = rng.normal(0.0, 2.0, size=(16, 300)).astype(np.float32)
    r = oracle.constrained_softmax(x, BOUND, T_MIN, T_MAX, ITERS, threads=1,
                                   lib=lib)
    assert np.max(np.abs(r.p.sum(axis=1) - 1.0)) < 1e-12
    assert np.all(np.argmax(r.p, axis=1) == np.argmax(x, axis=1))
    for b in range(x.shape[0]):
        Hout = scipy.stats.entropy(r.p[b])
        H_tmin = oracle.entropy(x[b], _f32(T_MIN), lib=lib)
        if H_tmin <= _f32(BOUND):
            assert r.flags[b] == 0
            assert Hout <= _f32(BOUND) + 1e-9
        else:
            assert r.flags[b] == oracle.FLAG_ENTROPY_OVERFLOW
            assert r.T[b] == _f32(T_MIN)

    # Shift invariance (the shift by 8 is exact in fp32 for these values).
    xs = (np.round(x * 64) / 64).astype(np.float32)
    r1 = oracle.constrained_softmax(xs, BOUND, T_MIN, T_MAX, ITERS, threads=1,
                                    lib=lib)
    r2 = oracle.constrained_softmax(xs + np.float32(8.0), BOUND, T_MIN, T_MAX,
                                    ITERS, threads=1, lib=lib)
    assert np.array_equal(r1.T, r2.T) and np.array_equal(r1.flags, r2.flags)
    assert np.max(np.abs(r1.p - r2.p)) < 1e-12

    # Constant rows: H = ln C at every T, so any bound below ln C is
    # unsatisfiable and the output stays exactly uniform.
    for C in (2, 5, 1000):
        row = np.full((1, C), 0.7, dtype=np.float32)
        r = oracle.constrained_softmax(row, BOUND, T_MIN, T_MAX, ITERS,
                                       threads=1, lib=lib)
        assert np.all(r.p == r.p[0, 0]) and abs(r.p[0, 0] * C - 1) < 1e-15
        assert r.flags[0] == oracle.FLAG_ENTROPY_OVERFLOW
        assert r.T[0] == _f32(T_MIN)
        assert abs(oracle.entropy(row[0], 0.3, lib=lib) - math.log(C)) < 1e-12

    # C = 1: the only probability is 1 and H = 0 <= bound.
    r = oracle.constrained_softmax(np.array([[3.5]], np.float32), BOUND,
                                   T_MIN, T_MAX, ITERS, threads=1, lib=lib)
    assert r.p[0, 0] == 1.0 and r.T[0] == 1.0 and r.flags[0] == 0


def check_search_path(lib) -> None:
    """H is nondecreasing in T (section 2.1 step 4), each step keeps the
    feasible half, and the bracket halves every step."""
    rng = np.random.default_rng(9)
    lo0, hi0 = oracle.search_interval(T_MIN, T_MAX)
    for trial in range(6):
        row = rng.normal(0.0, 1.0 + trial, size=200).astype(np.float32)
        path = oracle.constrained_softmax_path(row, BOUND, T_MIN, T_MAX,
                                               ITERS, lib=lib)
        assert path.iters == ITERS
        order = np.argsort(path.mids)
        assert np.all(np.diff(path.H[order]) >= -1e-12)
        lo, hi = lo0, hi0
        for mid, H in zip(path.mids, path.H):
            assert abs(mid - (lo + hi) / 2) <= 1e-15
            assert abs(H - oracle.entropy(row, mid, lib=lib)) <= 1e-12
            if H > _f32(BOUND):
                hi = mid
            else:
                lo = mid
        assert path.T == lo
        assert abs((hi - lo) - (hi0 - lo0) / 2 ** ITERS) < 1e-15


def check_fault_policy(lib) -> None:
    """Section 5.3: a NaN/Inf in the input zeroes the row and sets its flag;
    section 5.4: an unsatisfiable bound gives T = temperature_min and flag 3."""
    x = np.random.default_rng(1).normal(size=(6, 40)).astype(np.float32)
    x[1, 7] = np.nan
    x[2, 0] = np.inf
    x[3, 39] = -np.inf
    x[4, 3] = np.nan
    x[4, 5] = np.inf
    r = oracle.constrained_softmax(x, BOUND, T_MIN, T_MAX, ITERS, threads=1,
                                   lib=lib)
    assert list(r.flags[1:5]) == [1, 2, 2, 1]
    for b in (1, 2, 3, 4):
        assert np.all(r.p[b] == 0.0) and math.isnan(r.T[b])
        assert r.iters[b] == 0
    clean = oracle.constrained_softmax(x[[0, 5]], BOUND, T_MIN, T_MAX, ITERS,
                                       threads=1, lib=lib)
    assert np.array_equal(clean.p, r.p[[0, 5]])

    # Negative bound: no distribution has H < 0.
    r = oracle.constrained_softmax(x[[0]], -0.5, T_MIN, T_MAX, ITERS,
                                   threads=1, lib=lib)
    assert r.flags[0] == 3 and r.T[0] == _f32(T_MIN)
    np.testing.assert_allclose(r.p[0], oracle.softmax(x[0], _f32(T_MIN),
                                                      lib=lib), rtol=0,
                               atol=1e-15)


def check_parameter_edges(lib) -> None:
    rng = np.random.default_rng(21)
    x = rng.normal(0.0, 3.0, size=(4, 50)).astype(np.float32)
    # max_iter = 0: no halving, T = temperature_min.
    r = oracle.constrained_softmax(x, BOUND, T_MIN, T_MAX, 0, threads=1,
                                   lib=lib)
    for b in range(4):
        assert r.T[b] == _f32(T_MIN) and r.iters[b] == 0
        H_tmin = oracle.entropy(x[b], _f32(T_MIN), lib=lib)
        assert r.flags[b] == (3 if H_tmin > _f32(BOUND) else 0)
    # temperature_max < 1: the search runs on [t_min, t_max].
    row = np.array([0.0, 0.3], dtype=np.float32)
    t_max = 0.2
    Ts = t_star(lambda T: h_two_class(float(row[1]), T), _f32(0.6),
                _f32(T_MIN), _f32(t_max))
    assert Ts is None   # whole interval feasible: lo -> t_max
    r = oracle.constrained_softmax(row[None], 0.6, T_MIN, t_max, ITERS,
                                   threads=1, lib=lib)
    w = oracle.final_interval(T_MIN, t_max, ITERS)
    assert _f32(t_max) - w - 1e-15 <= r.T[0] < _f32(t_max)
    # temperature_min >= 1: nothing to halve, T = temperature_min.
    r = oracle.constrained_softmax(row[None], 0.01, 1.5, 10.0, ITERS,
                                   threads=1, lib=lib)
    assert r.T[0] == 1.5 and r.iters[0] == 0 and r.flags[0] == 3


# ------------------------------------------------------------------- backward
def _pow2_floor(x: float) -> float:
    return 2.0 ** math.floor(math.log2(x))


def check_backward_finite_difference(lib) -> None:
    """d(g . p)/dl_k by central differences through the whole forward (the
    search runs again at l +- h e_k) against the backward at the forward's
    T.  Agreement needs both the 1/T factor and T's zero derivative away
    from the points where a bisection comparison flips; perturbations that
    move T are skipped (they straddle such a point)."""
    rng = np.random.default_rng(61)
    cases = [(2, 1.0, BOUND), (5, 3.0, BOUND), (17, 2.0, 0.5),
             (64, 3.0, BOUND), (9, 2.0, 1e30), (12, 2.0, -1.0)]
    checked = 0
    for C, sigma, bound in cases:
        x = rng.normal(0.0, sigma, size=(2, C)).astype(np.float32)
        g = rng.normal(0.0, 1.0, size=(2, C))
        r0 = oracle.constrained_softmax(x, bound, T_MIN, T_MAX, ITERS,
                                        threads=1, lib=lib)
        grad = oracle.constrained_softmax_backward(r0.p, g, r0.T, lib=lib)
        for b in range(2):
            T0 = r0.T[b]
            h = _pow2_floor(T0 * 2.0 ** -12)
            ks = range(C) if C <= 17 else rng.choice(C, 12, replace=False)
            for k in ks:
                xp = x[b:b + 1].copy()
                xm = x[b:b + 1].copy()
                xp[0, k] = np.float32(float(x[b, k]) + h)
                xm[0, k] = np.float32(float(x[b, k]) - h)
                assert float(xp[0, k]) - float(x[b, k]) == h
                assert float(x[b, k]) - float(xm[0, k]) == h
                rp = oracle.constrained_softmax(xp, bound, T_MIN, T_MAX,
                                                ITERS, threads=1, lib=lib)
                rm = oracle.constrained_softmax(xm, bound, T_MIN, T_MAX,
                                                ITERS, threads=1, lib=lib)
                if not (rp.T[0] == T0 and rm.T[0] == T0):
                    continue
                fd = float(g[b] @ (rp.p[0] - rm.p[0])) / (2.0 * h)
                scale = np.max(np.abs(g[b])) / T0
                assert abs(fd - grad[b, k]) <= 1e-6 * scale, (C, b, k, fd,
                                                              grad[b, k])
                checked += 1
    assert checked >= 90


def check_backward_library_vjp(lib) -> None:
    """At the forward's T, the backward is the vector-Jacobian product of
    softmax(l / T) with T held fixed, which torch's autograd computes in
    fp64 by its own softmax backward."""
    import torch
    rng = np.random.default_rng(67)
    for C, bound in ((3, BOUND), (40, BOUND), (1000, 0.5), (257, -1.0),
                     (33, 1e30)):
        x = rng.normal(0.0, 2.5, size=(4, C)).astype(np.float32)
        g = rng.normal(0.0, 1.0, size=(4, C))
        r = oracle.constrained_softmax(x, bound, T_MIN, T_MAX, ITERS,
                                       threads=1, lib=lib)
        grad = oracle.constrained_softmax_backward(r.p, g, r.T, lib=lib)
        l = torch.tensor(x, dtype=torch.float64, requires_grad=True)
        T = torch.tensor(r.T, dtype=torch.float64)[:, None]
        out = torch.softmax(l / T, dim=1)
        out.backward(torch.tensor(g))
        ref = l.grad.numpy()
        scale = np.max(np.abs(g), axis=1, keepdims=True) / r.T[:, None]
        assert np.all(np.abs(grad - ref) <= 1e-12 * scale), C


def check_backward_jacobian_t1(lib) -> None:
    """Where no search is needed (T = 1) the backward is J^T g with the
    textbook softmax Jacobian J = diag(p) - p p^T, formed explicitly."""
    rng = np.random.default_rng(71)
    for C in (1, 2, 6, 50):
        x = rng.normal(0.0, 1.0, size=(3, C)).astype(np.float32)
        g = rng.normal(0.0, 1.0, size=(3, C))
        r = oracle.constrained_softmax(x, 1e30, T_MIN, T_MAX, ITERS,
                                       threads=1, lib=lib)
        assert np.all(r.T == 1.0)
        grad = oracle.constrained_softmax_backward(r.p, g, r.T, lib=lib)
        for b in range(3):
            p = scipy.special.softmax(x[b].astype(np.float64))
            J = np.diag(p) - np.outer(p, p)
            assert np.max(np.abs(grad[b] - J.T @ g[b])) < 1e-14


def check_backward_invariants(lib) -> None:
    """Gradients of a row sum to zero (the probabilities sum to 1), adding a
    constant to the upstream gradient changes nothing, the map is linear in
    the upstream gradient, a one-hot row has zero gradient, and rows whose T
    is not a positive finite number (NaN: the forward zeroed them) get
    zeros."""
    rng = np.random.default_rng(73)
    x = rng.normal(0.0, 3.0, size=(6, 300)).astype(np.float32)
    r = oracle.constrained_softmax(x, BOUND, T_MIN, T_MAX, ITERS, threads=1,
                                   lib=lib)
    assert np.all(r.T < 1.0)
    g = rng.normal(0.0, 1.0, size=x.shape)
    grad = oracle.constrained_softmax_backward(r.p, g, r.T, lib=lib)
    scale = np.max(np.abs(g)) / np.min(r.T)
    assert np.max(np.abs(grad.sum(axis=1))) <= 1e-13 * scale
    shifted = oracle.constrained_softmax_backward(r.p, g + 3.5, r.T, lib=lib)
    assert np.max(np.abs(shifted - grad)) <= 1e-13 * scale
    doubled = oracle.constrained_softmax_backward(r.p, 2.0 * g, r.T, lib=lib)
    assert np.array_equal(doubled, 2.0 * grad)
    onehot = np.zeros((1, 5))
    onehot[0, 2] = 1.0
    z = oracle.constrained_softmax_backward(onehot, g[:1, :5], [0.3], lib=lib)
    assert np.all(z == 0.0)
    T_bad = np.array([np.nan, -1.0, 0.0, np.inf, 0.5, 1.0])
    xb = x.copy()
    xb[0, 7] = np.nan
    rb = oracle.constrained_softmax(xb, BOUND, T_MIN, T_MAX, ITERS, threads=1,
                                    lib=lib)
    assert math.isnan(rb.T[0])
    T_bad[0] = rb.T[0]
    gb = oracle.constrained_softmax_backward(rb.p, g, T_bad, lib=lib)
    assert np.all(gb[:4] == 0.0)
    assert np.all(np.isfinite(gb[4:])) and np.any(gb[4:] != 0.0)


# ---------------------------------------------------------- attention_softmax
def _scipy_rows(v: np.ndarray) -> np.ndarray:
    return scipy.special.softmax(v.astype(np.float64), axis=-1)


def check_attention_plain_softmax(lib) -> None:
    """No mask, not causal: every row is the library softmax."""
    rng = np.random.default_rng(91)
    for B, H, S in ((1, 1, 1), (2, 3, 5), (1, 2, 64), (2, 1, 300)):
        x = rng.normal(0.0, 3.0, (B, H, S, S)).astype(np.float32)
        r = oracle.attention_softmax(x, threads=1, lib=lib)
        assert np.all(r.flags == 0)
        assert np.max(np.abs(r.p - _scipy_rows(x))) < 1e-13


def check_attention_causal_prefix(lib) -> None:
    """Causal row i is the library softmax of keys 0..i, zero after."""
    rng = np.random.default_rng(92)
    B, H, S = 2, 2, 37
    x = rng.normal(0.0, 2.0, (B, H, S, S)).astype(np.float32)
    r = oracle.attention_softmax(x, causal=True, threads=1, lib=lib)
    for b in range(B):
        for h in range(H):
            for i in range(S):
                ref = _scipy_rows(x[b, h, i, :i + 1])
                assert np.max(np.abs(r.p[b, h, i, :i + 1] - ref)) < 1e-13
                assert np.all(r.p[b, h, i, i + 1:] == 0.0)


def check_attention_mask_subset(lib) -> None:
    """An additive mask with -inf holes: on the kept keys the library
    softmax of scores + mask (added in numpy fp32), zeros on the holes;
    each batch uses its own mask row, with and without causal."""
    rng = np.random.default_rng(93)
    B, H, S = 3, 2, 40
    x = rng.normal(0.0, 2.0, (B, H, S, S)).astype(np.float32)
    mask = rng.normal(0.0, 1.0, (B, S)).astype(np.float32)
    mask[rng.random((B, S)) < 0.3] = -np.inf
    mask[:, 0] = 0.0
    for causal in (False, True):
        r = oracle.attention_softmax(x, mask, causal=causal, threads=1,
                                     lib=lib)
        assert np.all(r.flags == 0)
        for b in range(B):
            v = x[b] + mask[b][None, None, :]          # fp32 addition
            for h in range(H):
                for i in range(S):
                    end = i + 1 if causal else S
                    keep = np.flatnonzero(np.isfinite(v[h, i, :end]))
                    ref = np.zeros(S)
                    ref[keep] = _scipy_rows(v[h, i, keep])
                    assert np.max(np.abs(r.p[b, h, i] - ref)) < 1e-13
                    if (i + h) % 7 == 0:
                        one, flag = oracle.attention_softmax_row(
                            x[b, h, i], i, mask[b], causal, lib=lib)
                        assert flag == 0
                        assert np.max(np.abs(one - ref)) < 1e-13


def check_attention_fp32_mask_addition(lib) -> None:
    """The page's -1e9 mask is added in fp32: near 1e9 fp32 steps by 64, so
    every score of magnitude below 32 vanishes into -1e9 and a fully
    masked row becomes uniform; a partly masked row puts exactly 0 on its
    masked keys."""
    rng = np.random.default_rng(94)
    B, H, S = 2, 2, 24
    x = rng.uniform(-30.0, 30.0, (B, H, S, S)).astype(np.float32)
    mask = np.zeros((B, S), dtype=np.float32)
    mask[0, :] = -1e9
    mask[1, S // 2:] = -1e9
    r = oracle.attention_softmax(x, mask, threads=1, lib=lib)
    assert np.all(r.p[0] == 1.0 / S)
    assert np.all(r.p[1, :, :, S // 2:] == 0.0)
    ref = _scipy_rows(x[1, :, :, :S // 2])
    assert np.max(np.abs(r.p[1, :, :, :S // 2] - ref)) < 1e-13


def check_attention_invariants_and_faults(lib) -> None:
    """Rows sum to 1; an exactly representable shift of the scores changes
    nothing; logits near 1000 do not overflow; NaN (flag 1) and +-Inf
    (flag 2) in a used score or mask value zero the row (a NaN key that a
    causal row never uses does not); a row with every key masked by -inf
    is zeros with flag 0."""
    rng = np.random.default_rng(95)
    B, H, S = 2, 2, 16
    x = (np.round(rng.normal(0.0, 2.0, (B, H, S, S)) * 1024) / 1024).astype(np.float32)
    r = oracle.attention_softmax(x, causal=True, threads=1, lib=lib)
    assert np.max(np.abs(r.p.sum(axis=-1) - 1.0)) < 1e-14
    r8 = oracle.attention_softmax(x + np.float32(8.0), causal=True, threads=1,
                                  lib=lib)
    assert np.max(np.abs(r8.p - r.p)) < 1e-13
    big = oracle.attention_softmax(x + np.float32(1000.0), threads=1, lib=lib)
    assert np.all(np.isfinite(big.p))
    assert np.max(np.abs(big.p.sum(axis=-1) - 1.0)) < 1e-14
    y = x.copy()
    y[0, 0, 5, 3] = np.nan          # used by row 5
    y[0, 1, 2, 9] = np.nan          # key 9 > 2: a causal row 2 never uses it
    y[1, 0, 7, 0] = np.inf
    y[1, 1, 4, 4] = -np.inf
    mask = np.zeros((B, S), dtype=np.float32)
    rc = oracle.attention_softmax(y, causal=True, threads=1, lib=lib)
    assert rc.flags[0, 0, 5] == 1 and np.all(rc.p[0, 0, 5] == 0.0)
    assert rc.flags[0, 1, 2] == 0 and abs(rc.p[0, 1, 2].sum() - 1.0) < 1e-14
    assert rc.flags[1, 0, 7] == 2 and rc.flags[1, 1, 4] == 2
    assert np.all(rc.p[1, 1, 4] == 0.0)
    rn = oracle.attention_softmax(y, causal=False, threads=1, lib=lib)
    assert rn.flags[0, 1, 2] == 1
    mask[1, 3] = np.nan
    mask[0, 6] = np.inf
    rm = oracle.attention_softmax(x, mask, threads=1, lib=lib)
    assert np.all(rm.flags[1] == 1) and np.all(rm.flags[0] == 2)
    assert np.all(rm.p == 0.0)
    mask = np.zeros((B, S), dtype=np.float32)
    mask[0, :] = -np.inf
    ra = oracle.attention_softmax(x, mask, threads=1, lib=lib)
    assert np.all(ra.flags == 0) and np.all(ra.p[0] == 0.0)
    assert np.max(np.abs(ra.p[1].sum(axis=-1) - 1.0)) < 1e-14


# -------------------------------------------------------- biencoder_attention
def _bienc_inputs(seed, B=2, H=2, Q=6, K=5, D=16, sigma=1.0):
    rng = np.random.default_rng(seed)
    q = rng.normal(0.0, sigma, (B, H, Q, D)).astype(np.float32)
    k = rng.normal(0.0, sigma, (B, H, K, D)).astype(np.float32)
    v = rng.normal(0.0, 1.0, (B, H, K, D)).astype(np.float32)
    return q, k, v


def check_biencoder_scores(lib) -> None:
    """Step 1 against fp64 matmul (numpy): each fp32 score is within the
    rounding bound of a D-term dot product, (D + 1) u sum |q_d k_d| scale,
    of the exact q . k scale; and a query equal to a one-hot e_d picks
    k_d exactly."""
    u = 2.0 ** -24
    for seed, D in ((101, 16), (102, 64), (103, 3)):
        q, k, _ = _bienc_inputs(seed, D=D)
        scale = np.float32(1.0 / np.sqrt(D))
        s = oracle.biencoder_scores(q, k, scale, lib=lib)
        exact = np.einsum("bhqd,bhkd->bhqk", q.astype(np.float64),
                          k.astype(np.float64)) * float(scale)
        absd = np.einsum("bhqd,bhkd->bhqk", np.abs(q.astype(np.float64)),
                         np.abs(k.astype(np.float64))) * float(scale)
        assert np.all(np.abs(s - exact) <= (D + 2) * u * absd + 1e-30)
    q, k, _ = _bienc_inputs(104, Q=4, K=3, D=4)
    q[:] = 0.0
    for i in range(4):
        q[:, :, i, i] = 1.0
    s = oracle.biencoder_scores(q, k, 1.0, lib=lib)
    assert np.array_equal(s[:, :, :, :], np.swapaxes(k, 2, 3)[:, :, :4, :])
    # The fp32 order of the reading: 2^24 + 1 + 1 + 1 accumulated term by
    # term in fp32 stays at 2^24 (each +1 is a tie rounded to even), where
    # the exact sum 2^24 + 3 rounds to 2^24 + 4.
    q = np.ones((1, 1, 1, 4), dtype=np.float32)
    k = np.array([[[[2.0 ** 24, 1.0, 1.0, 1.0]]]], dtype=np.float32)
    s = oracle.biencoder_scores(q, k, 1.0, lib=lib)
    assert s[0, 0, 0, 0] == np.float32(2.0 ** 24)


def check_biencoder_composition(lib) -> None:
    """Steps 2-3: the attention rows are the oracle constrained softmax of
    the step-1 scores (pinned above); with a bound no row exceeds the
    attention is scipy's softmax, and every output row is attn @ values,
    a convex combination of value rows (inside their per-column range); a
    single context item returns its value row exactly."""
    q, k, v = _bienc_inputs(111, Q=7, K=9, D=12, sigma=2.0)
    r = oracle.biencoder_attention(q, k, v, 0.5, 1e30, lib=lib)
    ref = _scipy_rows(r.scores)
    assert np.max(np.abs(r.attn.p.reshape(ref.shape) - ref)) < 1e-13
    out = np.einsum("bhqk,bhkd->bhqd", ref, v.astype(np.float64))
    assert np.max(np.abs(r.out - out)) < 1e-12
    r = oracle.biencoder_attention(q, k, v, 0.5, 0.2, lib=lib)
    assert np.sum(r.attn.T < 1.0) >= 10
    lo = v.min(axis=2, keepdims=True).astype(np.float64)
    hi = v.max(axis=2, keepdims=True).astype(np.float64)
    assert np.all(r.out >= lo - 1e-12) and np.all(r.out <= hi + 1e-12)
    q1, k1, v1 = _bienc_inputs(112, K=1)
    r1 = oracle.biencoder_attention(q1, k1, v1, 0.25, 0.2, lib=lib)
    assert np.array_equal(r1.out, np.broadcast_to(v1.astype(np.float64),
                                                  r1.out.shape))


ALL_CHECKS = [
    check_two_class_entropy,
    check_spike_entropy,
    check_large_logits,
    check_two_class_temperature,
    check_spike_temperature,
    check_softmax_special_case,
    check_brute_force,
    check_invariants,
    check_search_path,
    check_fault_policy,
    check_parameter_edges,
    check_backward_finite_difference,
    check_backward_library_vjp,
    check_backward_jacobian_t1,
    check_backward_invariants,
    check_attention_plain_softmax,
    check_attention_causal_prefix,
    check_attention_mask_subset,
    check_attention_fp32_mask_addition,
    check_attention_invariants_and_faults,
    check_biencoder_scores,
    check_biencoder_composition,
]
