"""CPU oracle for the entropy-bounded softmax (``constrained_softmax``).

TEST INFRASTRUCTURE ONLY.  The test suite, the smoke check and the CPU-baseline
leg of ``bench.py`` are the only callers.  The product path (the CUDA library
and its Python binding) never imports this package, and this package imports
nothing from the product.

The arithmetic lives in ``constrained_softmax_oracle.c`` (plain fp64 C, libm
``exp``/``log``), which follows "BURT-IMMA CUDA Kernel API Reference",
section 2.1 ``constrained_softmax`` and section 5 (error codes, NaN/Inf policy,
graceful degradation), the backward of section 6.3 with the temperature
restored, attention_softmax (section 2.6) and biencoder_attention (section
2.5).  This module only compiles it with gcc, marshals numpy
arrays in and out through ctypes, and splits a batch over threads (rows are
independent, so the split changes no arithmetic).

Every function here is pinned by ``tests/test_oracle_pins.py`` against closed
forms, a library softmax, brute-force temperature scans and invariants.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "constrained_softmax_oracle.c")
LIBRARY = os.path.join(_HERE, "liboracle.so")

# gcc flags: IEEE double semantics, no contraction into FMA, so the x86 host
# and the Arm GPU host compute the same thing (up to libm's own rounding).
GCC_FLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
             "-fno-fast-math"]

_lock = threading.Lock()
_lib = None

FLAG_NONE = 0
FLAG_NAN_INPUT = 1
FLAG_INF_INPUT = 2
FLAG_ENTROPY_OVERFLOW = 3


def build_command(source: str = SOURCE, library: str = LIBRARY) -> list[str]:
    return ["gcc", *GCC_FLAGS, "-o", library, source, "-lm"]


def build(force: bool = False, source: str = SOURCE,
          library: str = LIBRARY) -> str:
    """Compile the oracle into a shared library (gcc, a second or so)."""
    if (not force and os.path.exists(library)
            and os.path.getmtime(library) >= os.path.getmtime(source)):
        return library
    tmp = f"{library}.{os.getpid()}.tmp"
    subprocess.run(build_command(source, tmp), check=True)
    os.replace(tmp, library)
    return library


def _bind(lib: ctypes.CDLL) -> ctypes.CDLL:
    f32p = ctypes.POINTER(ctypes.c_float)
    f64p = ctypes.POINTER(ctypes.c_double)
    i32p = ctypes.POINTER(ctypes.c_int32)
    lib.oracle_entropy.restype = ctypes.c_double
    lib.oracle_entropy.argtypes = [f32p, ctypes.c_int64, ctypes.c_double]
    lib.oracle_softmax.restype = None
    lib.oracle_softmax.argtypes = [f32p, ctypes.c_int64, ctypes.c_double, f64p]
    lib.oracle_constrained_softmax_rows.restype = None
    lib.oracle_constrained_softmax_rows.argtypes = [
        f32p, f64p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
        ctypes.c_float, ctypes.c_float, ctypes.c_float, ctypes.c_int32,
        f64p, i32p, i32p]
    lib.oracle_constrained_softmax_path.restype = ctypes.c_int32
    lib.oracle_constrained_softmax_path.argtypes = [
        f32p, f64p, ctypes.c_int64, ctypes.c_float, ctypes.c_float,
        ctypes.c_float, ctypes.c_int32, f64p, i32p, f64p, f64p]
    lib.oracle_attention_softmax_rows.restype = None
    lib.oracle_attention_softmax_rows.argtypes = [
        f32p, f32p, f64p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
        ctypes.c_int64, ctypes.c_int32, i32p]
    lib.oracle_attention_softmax_row.restype = ctypes.c_int32
    lib.oracle_attention_softmax_row.argtypes = [
        f32p, f32p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int32, f64p]
    lib.oracle_biencoder_scores.restype = None
    lib.oracle_biencoder_scores.argtypes = [
        f32p, f32p, f32p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
        ctypes.c_int64, ctypes.c_float]
    lib.oracle_constrained_softmax_backward_rows.restype = None
    lib.oracle_constrained_softmax_backward_rows.argtypes = [
        f64p, f64p, f64p, f64p, ctypes.c_int64, ctypes.c_int64,
        ctypes.c_int64]
    return lib


def load(path: str | None = None) -> ctypes.CDLL:
    """Load (building first if needed) the oracle library."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            _lib = _bind(ctypes.CDLL(build()))
        return _lib


def _ptr(a: np.ndarray, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _as_row(l) -> np.ndarray:
    row = np.ascontiguousarray(np.asarray(l, dtype=np.float32).reshape(-1))
    if row.size == 0:
        raise ValueError("a row needs at least one class")
    return row


def entropy(l, T: float, lib: ctypes.CDLL | None = None) -> float:
    """H(T) in nats of softmax(l / T) for one fp32 row (section 2.1 step 2)."""
    lib = lib or load()
    row = _as_row(l)
    return float(lib.oracle_entropy(_ptr(row, ctypes.c_float), row.size,
                                    float(T)))


def softmax(l, T: float, lib: ctypes.CDLL | None = None) -> np.ndarray:
    """softmax(l / T) in fp64 for one fp32 row (section 2.1 step 1)."""
    lib = lib or load()
    row = _as_row(l)
    p = np.empty(row.size, dtype=np.float64)
    lib.oracle_softmax(_ptr(row, ctypes.c_float), row.size, float(T),
                       _ptr(p, ctypes.c_double))
    return p


@dataclass
class Result:
    """Per-row results: probabilities, temperature, flag, bisection steps."""
    p: np.ndarray        # [batch, C] float64
    T: np.ndarray        # [batch] float64 (NaN for non-finite rows)
    flags: np.ndarray    # [batch] int32, section 5.1 codes 0..3
    iters: np.ndarray    # [batch] int32, H evaluations in the search


def default_threads() -> int:
    return len(os.sched_getaffinity(0))


def constrained_softmax(logits, entropy_bound: float = 0.20,
                        t_min: float = 0.01, t_max: float = 10.0,
                        max_iter: int = 20, threads: int | None = None,
                        lib: ctypes.CDLL | None = None) -> Result:
    """Oracle constrained_softmax over a [batch, C] fp32 matrix.

    Parameters and defaults follow section 2.1's signature (entropy_bound
    0.20, temperature_min 0.01, temperature_max 10.0, max_iterations 20).
    Rows are split over ``threads`` worker threads (default: every core this
    process may run on); each row is computed by the same C code regardless.
    """
    lib = lib or load()
    x = np.ascontiguousarray(np.asarray(logits, dtype=np.float32))
    if x.ndim != 2:
        raise ValueError("logits must be [batch, num_classes]")
    batch, C = x.shape
    if C < 1:
        raise ValueError("num_classes must be >= 1")
    p = np.empty((batch, C), dtype=np.float64)
    T = np.empty(batch, dtype=np.float64)
    flags = np.empty(batch, dtype=np.int32)
    iters = np.empty(batch, dtype=np.int32)
    if batch == 0:
        return Result(p, T, flags, iters)

    bound = np.float32(entropy_bound)
    lo_t = np.float32(t_min)
    hi_t = np.float32(t_max)

    def run(b0: int, b1: int) -> None:
        lib.oracle_constrained_softmax_rows(
            _ptr(x, ctypes.c_float), _ptr(p, ctypes.c_double), b0, b1, C,
            float(bound), float(lo_t), float(hi_t), int(max_iter),
            _ptr(T, ctypes.c_double), _ptr(flags, ctypes.c_int32),
            _ptr(iters, ctypes.c_int32))

    n = threads or default_threads()
    n = max(1, min(n, batch))
    if n == 1:
        run(0, batch)
    else:
        edges = np.linspace(0, batch, n + 1).astype(np.int64)
        with ThreadPoolExecutor(max_workers=n) as pool:
            futs = [pool.submit(run, int(edges[i]), int(edges[i + 1]))
                    for i in range(n) if edges[i + 1] > edges[i]]
            for f in futs:
                f.result()
    return Result(p, T, flags, iters)


@dataclass
class Path:
    """One row's result with its bisection path."""
    p: np.ndarray
    T: float
    flag: int
    iters: int
    mids: np.ndarray     # [iters] midpoints in order
    H: np.ndarray        # [iters] H(mid)


def constrained_softmax_path(l, entropy_bound: float = 0.20,
                             t_min: float = 0.01, t_max: float = 10.0,
                             max_iter: int = 20,
                             lib: ctypes.CDLL | None = None) -> Path:
    """One row, recording every bisection midpoint and H(midpoint)."""
    lib = lib or load()
    row = _as_row(l)
    C = row.size
    p = np.empty(C, dtype=np.float64)
    T = np.zeros(1, dtype=np.float64)
    it = np.zeros(1, dtype=np.int32)
    n = max(int(max_iter), 1)
    mids = np.full(n, np.nan)
    Hs = np.full(n, np.nan)
    flag = lib.oracle_constrained_softmax_path(
        _ptr(row, ctypes.c_float), _ptr(p, ctypes.c_double), C,
        float(np.float32(entropy_bound)), float(np.float32(t_min)),
        float(np.float32(t_max)), int(max_iter), _ptr(T, ctypes.c_double),
        _ptr(it, ctypes.c_int32), _ptr(mids, ctypes.c_double),
        _ptr(Hs, ctypes.c_double))
    k = int(it[0])
    return Path(p, float(T[0]), int(flag), k, mids[:k].copy(), Hs[:k].copy())


def constrained_softmax_backward(p, grad_output, T,
                                 lib: ctypes.CDLL | None = None) -> np.ndarray:
    """Gradient of the loss with respect to the logits, in fp64.

    ``p`` is the forward's output [batch, C], ``grad_output`` the upstream
    gradient of the same shape and ``T`` the forward's per-row temperature
    [batch].  Each row gets (1/T) p (g - <g, p>): section 6.3's
    ConstrainedSoftmaxFunction.backward with the 1/T of softmax(l / T)
    restored (T is piecewise constant in the logits, so it contributes no
    term of its own); rows with T NaN (or not positive and finite) get
    zeros.  Inputs of any float dtype are promoted exactly to fp64.
    """
    lib = lib or load()
    pp = np.ascontiguousarray(np.asarray(p, dtype=np.float64))
    gg = np.ascontiguousarray(np.asarray(grad_output, dtype=np.float64))
    tt = np.ascontiguousarray(np.asarray(T, dtype=np.float64).reshape(-1))
    if pp.ndim != 2 or gg.shape != pp.shape or tt.size != pp.shape[0]:
        raise ValueError("p, grad_output: [batch, C]; T: [batch]")
    batch, C = pp.shape
    grad = np.empty((batch, C), dtype=np.float64)
    if batch and C:
        lib.oracle_constrained_softmax_backward_rows(
            _ptr(pp, ctypes.c_double), _ptr(gg, ctypes.c_double),
            _ptr(tt, ctypes.c_double), _ptr(grad, ctypes.c_double), 0, batch,
            C)
    return grad


@dataclass
class AttentionResult:
    p: np.ndarray        # [B, H, S, S] float64
    flags: np.ndarray    # [B, H, S] int32, section 5.1 codes 0..2


def attention_softmax(scores, mask=None, causal: bool = False,
                      threads: int | None = None,
                      lib: ctypes.CDLL | None = None) -> AttentionResult:
    """Oracle attention_softmax (section 2.6) of fp32 scores [B, H, S, S]
    with an optional additive fp32 mask [B, S] (the page's [B, 1, 1, S]).
    Rows are split over threads; each row is the same C code."""
    lib = lib or load()
    x = np.ascontiguousarray(np.asarray(scores, dtype=np.float32))
    if x.ndim != 4 or x.shape[2] != x.shape[3]:
        raise ValueError("scores must be [B, H, S, S]")
    B, H, S, _ = x.shape
    m = None
    if mask is not None:
        m = np.ascontiguousarray(np.asarray(mask, dtype=np.float32))
        m = m.reshape(B, S)
    p = np.empty(x.shape, dtype=np.float64)
    flags = np.empty((B, H, S), dtype=np.int32)
    rows = B * H * S
    if rows == 0:
        return AttentionResult(p, flags)
    mp = _ptr(m, ctypes.c_float) if m is not None else None

    def run(r0: int, r1: int) -> None:
        lib.oracle_attention_softmax_rows(
            _ptr(x, ctypes.c_float), mp, _ptr(p, ctypes.c_double), r0, r1, H,
            S, int(bool(causal)), _ptr(flags, ctypes.c_int32))

    n = max(1, min(threads or default_threads(), rows))
    if n == 1:
        run(0, rows)
    else:
        edges = np.linspace(0, rows, n + 1).astype(np.int64)
        with ThreadPoolExecutor(max_workers=n) as pool:
            for f in [pool.submit(run, int(edges[i]), int(edges[i + 1]))
                      for i in range(n) if edges[i + 1] > edges[i]]:
                f.result()
    return AttentionResult(p, flags)


def attention_softmax_row(s, i: int, mask_row=None, causal: bool = False,
                          lib: ctypes.CDLL | None = None):
    """One row of attention_softmax: fp32 scores s [S] of query i, the
    batch's mask row [S] or None.  Returns (p [S] float64, flag)."""
    lib = lib or load()
    row = _as_row(s)
    m = None
    if mask_row is not None:
        m = np.ascontiguousarray(np.asarray(mask_row, dtype=np.float32).reshape(-1))
        if m.size != row.size:
            raise ValueError("mask row must match the scores row")
    p = np.empty(row.size, dtype=np.float64)
    flag = lib.oracle_attention_softmax_row(
        _ptr(row, ctypes.c_float), _ptr(m, ctypes.c_float) if m is not None
        else None, row.size, int(i), int(bool(causal)),
        _ptr(p, ctypes.c_double))
    return p, int(flag)


@dataclass
class BiencoderResult:
    out: np.ndarray      # [B, H, Q, D] float64
    scores: np.ndarray   # [B, H, Q, K] float32 (step 1)
    attn: Result         # step 2 on the [B H Q, K] score rows


def biencoder_scores(query, keys, scale: float,
                     lib: ctypes.CDLL | None = None) -> np.ndarray:
    """Step 1 of section 2.5 in fp32 as fixed by the oracle's reading:
    per score one fused multiply-add per d in order, then * scale."""
    lib = lib or load()
    q = np.ascontiguousarray(np.asarray(query, dtype=np.float32))
    k = np.ascontiguousarray(np.asarray(keys, dtype=np.float32))
    if q.ndim != 4 or k.ndim != 4 or q.shape[:2] != k.shape[:2] \
            or q.shape[3] != k.shape[3]:
        raise ValueError("query [B, H, Q, D] and keys [B, H, K, D]")
    B, H, Q, D = q.shape
    K = k.shape[2]
    s = np.empty((B, H, Q, K), dtype=np.float32)
    if s.size:
        lib.oracle_biencoder_scores(_ptr(q, ctypes.c_float),
                                    _ptr(k, ctypes.c_float),
                                    _ptr(s, ctypes.c_float), B * H, Q, K, D,
                                    float(np.float32(scale)))
    return s


def biencoder_attention(query, keys, values, scale: float,
                        entropy_bound: float = 0.20, t_min: float = 0.01,
                        t_max: float = 10.0, max_iter: int = 20,
                        lib: ctypes.CDLL | None = None) -> BiencoderResult:
    """Section 2.5 biencoder_attention: scores (step 1, fp32 as above), the
    oracle constrained softmax of every score row (step 2, fp64), then
    attn @ values in fp64 (step 3, a library matmul)."""
    lib = lib or load()
    s = biencoder_scores(query, keys, scale, lib=lib)
    B, H, Q, K = s.shape
    v = np.asarray(values, dtype=np.float32)
    if v.shape[:3] != (B, H, K):
        raise ValueError("values must be [B, H, K, D]")
    attn = constrained_softmax(s.reshape(B * H * Q, K), entropy_bound, t_min,
                               t_max, max_iter, lib=lib)
    p = attn.p.reshape(B, H, Q, K)
    out = np.einsum("bhqk,bhkd->bhqd", p, v.astype(np.float64))
    return BiencoderResult(out, s, attn)


def search_interval(t_min: float, t_max: float) -> tuple[float, float]:
    """(lo0, hi0) of the bisection, with the fp32 parameters as doubles."""
    lo = float(np.float32(t_min))
    hi = min(1.0, float(np.float32(t_max)))
    return lo, hi


def final_interval(t_min: float, t_max: float, max_iter: int) -> float:
    """Width of the bracket after max_iter halvings of [lo0, hi0]."""
    lo, hi = search_interval(t_min, t_max)
    if hi <= lo:
        return 0.0
    return (hi - lo) / 2.0 ** int(max_iter)
