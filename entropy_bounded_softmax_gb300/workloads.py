"""Seeded synthetic inputs for the constrained-softmax workloads.

This module only draws random numbers; it holds none of the method's
arithmetic.  Both the CUDA path's tests/benchmark and the CPU oracle take
their inputs from here, so the two always see the same logits.

Recipe (numpy ``Generator(PCG64)``): rows are drawn in blocks of
``BLOCK_ROWS``; block ``k`` of a workload with seed ``s`` uses
``Generator(PCG64([s, k]))``, so any subset of rows can be regenerated
without drawing the whole matrix.  Within a block the draws are, in order:
the block's normals (``standard_normal`` in fp32, times sigma), then the
workload-specific extras described on each workload.

The workloads are the shapes the page quotes or the ones a user of the op
meets: a small case, the page's latency case (batch 32 x 50000 classes,
"BURT-IMMA CUDA Kernel API Reference", section 2.1 Performance Notes and
section 7.1), a mixture-of-experts router (64 experts; the Parameters table
names "number of experts" as a use of num_classes), rows too long for one
CTA's shared memory, and a throughput sweep over the bound and the iteration
count.  The page measures on no dataset; every input is synthetic.
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace

import numpy as np

BLOCK_ROWS = 64


@dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    num_classes: int
    kind: str                 # "normal" | "router" | "long_mixed"
    sigma: float = 1.0
    seed: int = 1000
    entropy_bound: float = 0.20
    t_min: float = 0.01
    t_max: float = 10.0
    max_iter: int = 20
    note: str = ""
    extra: dict = field(default_factory=dict)

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)

    @property
    def elements(self) -> int:
        return self.batch * self.num_classes


# The five workloads (sizes and distributions as stated on each line).
SMALL = Workload("small_4x1000", 4, 1000, "normal", 1.0, 1001,
                 note="batch 4, 1000 classes, N(0,1)")
LATENCY = Workload("latency_32x50000", 32, 50000, "normal", 2.0, 1002,
                   note="batch 32, 50000 classes, N(0,2^2)")
ROUTER = Workload("moe_router_65536x64", 65536, 64, "router", 1.0, 1003,
                  note="65536 tokens, 64 experts, N(0,1) plus one expert per "
                       "row boosted by U(0,3)")
LONG = Workload("long_rows_256x131072", 256, 131072, "long_mixed", 1.0, 1004,
                note="256 rows of 131072 classes: 13 constant rows, the rest "
                     "alternate N(0,1) and N(0,1) with one index +15",
                extra={"constant_frac": 0.05, "spike": 15.0})
SWEEP = Workload("sweep_4096x32000", 4096, 32000, "normal", 3.0, 1005,
                 note="batch 4096, 32000 classes, N(0,3^2); bound in "
                      "{0.05,0.2,1.0} x max_iter in {20,40}")

WORKLOADS = {w.name: w for w in (SMALL, LATENCY, ROUTER, LONG, SWEEP)}
SWEEP_POINTS = [(b, it) for b in (0.05, 0.20, 1.0) for it in (20, 40)]


def sweep_workloads() -> list[Workload]:
    return [SWEEP.with_(name=f"{SWEEP.name}_b{b}_it{it}", entropy_bound=b,
                        max_iter=it) for b, it in SWEEP_POINTS]


def _block_rng(seed: int, block: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64([seed, block]))


def _constant_rows(w: Workload) -> np.ndarray:
    """Indices of the constant rows of a long_mixed workload (seeded)."""
    n_const = int(round(w.extra.get("constant_frac", 0.05) * w.batch))
    rng = np.random.Generator(np.random.PCG64([w.seed, 1 << 30]))
    return np.sort(rng.choice(w.batch, size=n_const, replace=False))


def row_kinds(w: Workload) -> np.ndarray:
    """Per-row label for long_mixed: 0 normal, 1 spiked, 2 constant."""
    kinds = np.zeros(w.batch, dtype=np.int8)
    if w.kind != "long_mixed":
        return kinds
    const = np.zeros(w.batch, dtype=bool)
    const[_constant_rows(w)] = True
    rest = np.flatnonzero(~const)
    kinds[rest[1::2]] = 1
    kinds[const] = 2
    return kinds


def _gen_block(w: Workload, block: int, kinds: np.ndarray) -> np.ndarray:
    r0 = block * BLOCK_ROWS
    r1 = min(w.batch, r0 + BLOCK_ROWS)
    n = r1 - r0
    C = w.num_classes
    rng = _block_rng(w.seed, block)
    x = rng.standard_normal((n, C), dtype=np.float32)
    x *= np.float32(w.sigma)
    if w.kind == "router":
        idx = rng.integers(0, C, size=n)
        boost = rng.uniform(0.0, 3.0, size=n).astype(np.float32)
        x[np.arange(n), idx] += boost
    elif w.kind == "long_mixed":
        idx = rng.integers(0, C, size=n)
        const_val = rng.standard_normal(n, dtype=np.float32)
        spike = np.float32(w.extra.get("spike", 15.0))
        k = kinds[r0:r1]
        for j in range(n):
            if k[j] == 1:
                x[j, idx[j]] += spike
            elif k[j] == 2:
                x[j, :] = const_val[j]
    elif w.kind != "normal":
        raise ValueError(f"unknown workload kind {w.kind!r}")
    return x


def generate(w: Workload, rows=None) -> np.ndarray:
    """The workload's fp32 logits, or only ``rows`` (indices) of them."""
    kinds = row_kinds(w)
    if rows is None:
        rows_arr = np.arange(w.batch)
    else:
        rows_arr = np.asarray(rows, dtype=np.int64).reshape(-1)
        if rows_arr.size and (rows_arr.min() < 0 or rows_arr.max() >= w.batch):
            raise IndexError("row index out of range")
    out = np.empty((rows_arr.size, w.num_classes), dtype=np.float32)
    if rows_arr.size == 0:
        return out
    blocks = np.unique(rows_arr // BLOCK_ROWS)
    for blk in blocks:
        xb = _gen_block(w, int(blk), kinds)
        sel = np.flatnonzero(rows_arr // BLOCK_ROWS == blk)
        out[sel] = xb[rows_arr[sel] - blk * BLOCK_ROWS]
    return out


# bf16 inputs.  The bf16 workloads are the fp32 workloads' logits rounded
# to the nearest bf16 (ties to even), stored as 16-bit patterns; both sides
# then see the same values: the CUDA path reads the patterns, the oracle the
# fp32 numbers they stand for (a bf16 pattern is the top half of that fp32).
def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 array -> uint16 bf16 patterns, rounded to nearest even (NaN
    stays a quiet NaN, infinities stay infinite)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
    nan = np.isnan(np.asarray(x, dtype=np.float32))
    r[nan] = ((u[nan] >> 16) | 0x40).astype(np.uint16)
    return r


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """uint16 bf16 patterns -> the fp32 values they stand for."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def sample_rows(w: Workload, n: int, seed: int = 7) -> np.ndarray:
    """A seeded, sorted sample of n distinct row indices (always includes
    the first and last row)."""
    n = min(n, w.batch)
    rng = np.random.Generator(np.random.PCG64([w.seed, seed, 99]))
    picks = set(rng.choice(w.batch, size=n, replace=False).tolist())
    picks.update({0, w.batch - 1})
    return np.array(sorted(picks), dtype=np.int64)


# Backward inputs.  The backward takes the forward's output p, its per-row
# temperature T and an upstream gradient g.  g and T are drawn here; p is
# then softmax(l / T) of the workload's logits, computed by whichever side
# needs it (the oracle in the tests, the forward kernel in the benchmark).
BACKWARD_T1_EVERY = 16      # rows r with r % 16 == 3 have T = 1 (no search)
BACKWARD_NAN_EVERY = 64     # rows r with r % 64 == 5 have T = NaN (a row the
                            # forward zeroed)


def backward_inputs(w: Workload, rows=None) -> tuple[np.ndarray, np.ndarray]:
    """(g, T) for the workload's rows (or ``rows``): g ~ N(0, 1) fp32 of the
    logits' shape; T ~ U(t_min, 1) fp32 per row, except T = 1 on every 16th
    row and NaN on every 64th.  Block k of seed s draws from
    ``Generator(PCG64([s, k, 2]))``: g's normals, then the block's T."""
    rows_arr = (np.arange(w.batch) if rows is None
                else np.asarray(rows, dtype=np.int64).reshape(-1))
    if rows_arr.size and (rows_arr.min() < 0 or rows_arr.max() >= w.batch):
        raise IndexError("row index out of range")
    C = w.num_classes
    g = np.empty((rows_arr.size, C), dtype=np.float32)
    T = np.empty(rows_arr.size, dtype=np.float32)
    for blk in np.unique(rows_arr // BLOCK_ROWS):
        r0 = int(blk) * BLOCK_ROWS
        n = min(w.batch, r0 + BLOCK_ROWS) - r0
        rng = np.random.Generator(np.random.PCG64([w.seed, int(blk), 2]))
        gb = rng.standard_normal((n, C), dtype=np.float32)
        tb = rng.uniform(w.t_min, 1.0, size=n).astype(np.float32)
        r = np.arange(r0, r0 + n)
        tb[r % BACKWARD_T1_EVERY == 3] = 1.0
        tb[r % BACKWARD_NAN_EVERY == 5] = np.nan
        sel = np.flatnonzero(rows_arr // BLOCK_ROWS == blk)
        g[sel] = gb[rows_arr[sel] - r0]
        T[sel] = tb[rows_arr[sel] - r0]
    return g, T


# attention_softmax workloads ("BURT-IMMA CUDA Kernel API Reference",
# section 2.6 Performance Notes and section 7.1: batch 32, 8 heads, seq_len
# 512), plus a causal variant and a long-row case past the page's 2048-key
# two-pass threshold.  Scores ~ N(0, 1) fp32 (scaled dot products).  Mask:
# each batch keeps its first L_b keys, L_b ~ U{S/2, ..., S}, and masks the
# rest with the page's -1e9 (or -inf for mask="neg_inf").
@dataclass(frozen=True)
class AttentionWorkload:
    name: str
    batch: int
    heads: int
    seq_len: int
    causal: bool
    mask: str = "neg_1e9"      # "none" | "neg_1e9" | "neg_inf"
    seed: int = 2000
    note: str = ""

    @property
    def rows(self) -> int:
        return self.batch * self.heads * self.seq_len

    @property
    def elements(self) -> int:
        return self.rows * self.seq_len


ATTN_PAGE = AttentionWorkload(
    "attention_32x8x512", 32, 8, 512, False, "neg_1e9", 2001,
    note="batch 32, 8 heads, seq_len 512, N(0,1) scores, -1e9 padding mask")
ATTN_PAGE_CAUSAL = AttentionWorkload(
    "attention_32x8x512_causal", 32, 8, 512, True, "neg_1e9", 2002,
    note="as attention_32x8x512, causal")
ATTN_LONG = AttentionWorkload(
    "attention_2x8x4096_causal", 2, 8, 4096, True, "neg_inf", 2003,
    note="batch 2, 8 heads, seq_len 4096, causal, -inf padding mask")
ATTENTION_WORKLOADS = {w.name: w for w in (ATTN_PAGE, ATTN_PAGE_CAUSAL,
                                           ATTN_LONG)}


def attention_mask(w: AttentionWorkload) -> np.ndarray | None:
    """The [B, S] fp32 additive mask (None for mask="none")."""
    if w.mask == "none":
        return None
    rng = np.random.Generator(np.random.PCG64([w.seed, 1 << 30]))
    S = w.seq_len
    lengths = rng.integers(S // 2, S + 1, size=w.batch)
    value = np.float32(-1e9) if w.mask == "neg_1e9" else np.float32(-np.inf)
    m = np.zeros((w.batch, S), dtype=np.float32)
    for b in range(w.batch):
        m[b, lengths[b]:] = value
    return m


def generate_attention(w: AttentionWorkload, rows=None) -> np.ndarray:
    """Scores of the workload's rows (flattened row index r = (b H + h) S +
    i), shape [n, S]; all rows when ``rows`` is None.  Rows are drawn in
    blocks of BLOCK_ROWS from Generator(PCG64([seed, block]))."""
    S = w.seq_len
    rows_arr = (np.arange(w.rows) if rows is None
                else np.asarray(rows, dtype=np.int64).reshape(-1))
    if rows_arr.size and (rows_arr.min() < 0 or rows_arr.max() >= w.rows):
        raise IndexError("row index out of range")
    out = np.empty((rows_arr.size, S), dtype=np.float32)
    for blk in np.unique(rows_arr // BLOCK_ROWS):
        r0 = int(blk) * BLOCK_ROWS
        n = min(w.rows, r0 + BLOCK_ROWS) - r0
        rng = _block_rng(w.seed, int(blk))
        xb = rng.standard_normal((n, S), dtype=np.float32)
        sel = np.flatnonzero(rows_arr // BLOCK_ROWS == blk)
        out[sel] = xb[rows_arr[sel] - r0]
    return out


# biencoder_attention workloads ("BURT-IMMA CUDA Kernel API Reference",
# section 2.5 Performance Notes and section 7.1: batch 32, query_len 512,
# context_len 64, d_head 64, 8 heads).  query, keys, values ~ N(0, 1) fp32;
# with scale 1/sqrt(d_head) the scores are about N(0, 1).
@dataclass(frozen=True)
class BiencoderWorkload:
    name: str
    batch: int
    heads: int
    query_len: int
    context_len: int
    d_head: int
    seed: int = 3000
    entropy_bound: float = 0.20
    note: str = ""

    @property
    def rows(self) -> int:
        return self.batch * self.heads * self.query_len


BIENC_PAGE = BiencoderWorkload(
    "biencoder_32x8x512x64x64", 32, 8, 512, 64, 64, 3001,
    note="batch 32, 8 heads, 512 queries, 64 context items, d_head 64, "
         "N(0,1) inputs")
BIENC_WIDE = BiencoderWorkload(
    "biencoder_4x8x1024x256x64", 4, 8, 1024, 256, 64, 3002,
    note="batch 4, 8 heads, 1024 queries, 256 context items, d_head 64")
BIENCODER_WORKLOADS = {w.name: w for w in (BIENC_PAGE, BIENC_WIDE)}


def generate_biencoder(w: BiencoderWorkload):
    """(query [B, H, Q, D], keys [B, H, K, D], values [B, H, K, D]) fp32,
    drawn in that order from Generator(PCG64([seed, 0]))."""
    rng = np.random.Generator(np.random.PCG64([w.seed, 0]))
    B, H, Q, K, D = w.batch, w.heads, w.query_len, w.context_len, w.d_head
    q = rng.standard_normal((B, H, Q, D), dtype=np.float32)
    k = rng.standard_normal((B, H, K, D), dtype=np.float32)
    v = rng.standard_normal((B, H, K, D), dtype=np.float32)
    return q, k, v
