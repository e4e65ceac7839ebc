// Cluster kernel: one thread-block cluster of n CTAs per row (n = 1: one CTA
// per row).  Each CTA holds its slice of the row in shared memory for the
// whole search, so the row is read from HBM once and written once.
//
// Method: "BURT-IMMA CUDA Kernel API Reference", section 2.1
// `constrained_softmax`, Description steps 1-4, with the error policy of
// sections 5.3 and 5.4.  Per row:
//   stage   every thread brings its part of the slice into shared memory
//           (16-byte asynchronous copies, all in flight at once, in
//           launches with several CTAs per SM; 128-bit loads eight at a
//           time otherwise) and folds it into its own max m_t and a
//           finiteness check;
//   T = 1   one pass turns the thread's classes into y_i = (l_i - m_t)
//           log2(e) in place and sums S = sum 2^y_i, V = sum y_i 2^y_i,
//           W = sum y_i^2 2^y_i; a single reduction then forms the row's max
//           m = max_i l_i (T-independent, computed once) and S, V, W
//           rescaled to it, and H(1) = ln2 (log2 S - V/S) decides whether a
//           search is needed.  Each thread keeps its offset d = (m_t - m)
//           log2 e and every later pass uses beta (y + d);
//   search  rounds of the temperature search of cs_search.cuh: each round
//           evaluates (S, V) at 1-3 temperatures in one pass over the slice
//           (plus W at the first one when a Newton step follows) and
//           reduces them; the search returns the bisection's final lo and
//           S(lo);
//   output  p_i = 2^(beta_lo y_i) / S(lo), written with 128-bit streaming
//           stores.
//
// Reduction.  Every warp reduces its partial sums with a shuffle tree, then
// pushes them into its own slot of every CTA of the cluster (st.async,
// counted on that CTA's mbarrier; in a launch without clusters, a plain
// store and an arrival).  Every warp waits for the mbarrier and reduces all
// n x warps slots in one fixed order (each lane folds slots lane, lane + 32,
// ..., then a butterfly), so every thread of the cluster holds bit-identical
// sums and takes the same decisions, with no CTA-wide barrier in the
// search.  The T = 1 statistics, whose partials are relative to different
// maxima, take the max first at the warp and at the cluster stage and move
// every partial to it once before summing.  Slots and mbarriers are
// double-buffered, which is safe because no warp can push for exchange k+2
// before every warp of the cluster has pushed for exchange k+1, which each
// does only after reading exchange k.
//
// Every wait is bounded (cs::kWaitLimitCycles by default).  A thread whose
// wait times out records CS_ERR_TIMEOUT and from then on neither waits nor
// pushes; the search then ends within its round limit on whatever the slots
// hold, and before exiting such a CTA sleeps for a bounded while, so that
// pushes peers had already issued into it land first.
#include <math.h>

#include "cs_search.cuh"

namespace cs {
namespace {

using namespace csd;

// Geometry of one CTA's slice in shared memory.  Element j of the slice
// lives at row[pad + j], so groups of four elements that are aligned in
// global memory (16 bytes of fp32, 8 of bf16) land on 16-byte aligned
// shared addresses.  Float4 q in [qb0, qb1) comes in by vector loads; the
// head (q = 0 when pad > 0) and tail float4s element by element.
struct Slice {
    int pad;
    int len;
    int q4;       // float4s of the slice in shared memory
    int qb0, qb1; // 16-byte aligned body
    int head_q;   // -1 if none
    int tail_q;   // -1 if none
};

template <class In>
__device__ __forceinline__ Slice make_slice(const typename In::T* src, int len) {
    Slice s;
    s.pad = static_cast<int>((reinterpret_cast<uintptr_t>(src) / In::kBytes) & 3);
    s.len = len;
    if (len <= 0) {
        s.len = 0;
        s.q4 = s.qb0 = s.qb1 = 0;
        s.head_q = s.tail_q = -1;
        return s;
    }
    const int end = s.pad + len;
    s.q4 = (end + 3) >> 2;
    s.qb0 = s.pad > 0 ? 1 : 0;
    s.qb1 = end >> 2;
    if (s.qb1 < s.qb0) s.qb1 = s.qb0;
    s.head_q = s.pad > 0 ? 0 : -1;
    s.tail_q = (end & 3) ? (end >> 2) : -1;
    if (s.tail_q == s.head_q) s.tail_q = -1;
    return s;
}

// Shared-memory objects of one CTA (cs::cluster_smem_layout places them).
struct Smem {
    float* cslot;     // [2][n * warps][kSlotVals] exchange slots
    uint64_t* cbar;   // [2] exchange mbarriers
    float4* row4;     // the slice
};

// Exchange state of one thread (every thread runs every exchange).
struct Exch {
    int warps;
    int n;
    uint32_t rank;
    uint32_t xk;      // exchanges so far (slot buffer, mbarrier phase)
    uint64_t limit;
    bool dead;
};

// Reduction operators.  combine(a, b) must give the same bits as
// combine(b, a), so that both lanes of every shuffle-tree exchange agree and
// every lane ends with the same result.
struct OpSum {
    template <int NV>
    static __device__ __forceinline__ void identity(float (&a)[NV]) {
#pragma unroll
        for (int i = 0; i < NV; ++i) a[i] = 0.0f;
    }
    template <int NV>
    static __device__ __forceinline__ void combine(float (&a)[NV],
                                                   const float (&b)[NV]) {
#pragma unroll
        for (int i = 0; i < NV; ++i) a[i] = a[i] + b[i];
    }
};

// Partial softmax statistics of a set of classes: {m, S, V, W, code} with
// m the set's max, y = (l - m) log2 e, S = sum 2^y, V = sum y 2^y,
// W = sum y^2 2^y, and code the set's NaN/Inf code, then, for each of NF
// fan points at inverse temperature b_k = fb0 4^k, S_k = sum 2^(b_k y) and
// V_k = sum y 2^(b_k y).  Combining rescales both sides to the larger max:
// with d = (m_i - m) log2 e <= 0, a side contributes 2^d S_i,
// 2^d (V_i + d S_i) and 2^d (W_i + 2 d V_i + d^2 S_i), and at fan point k
// f_k S_k,i and f_k (V_k,i + d S_k,i) with f_k = 2^(b_k d) (f_0 from the
// ex2 unit, each next one the previous squared twice).  An empty side
// (S = 0) contributes nothing.  Explicit roundings keep the compiler from
// contracting the two sides differently.
template <int NF>
struct OpSoftmaxT {
    // Value layout: {m, S, V, W, code} without a fan; with one W (not
    // needed: the first Newton step starts from the fan's point) is left
    // out, {m, S, V, code, S_0, V_0, ...}.
    static constexpr int kCode = NF == 0 ? 4 : 3;
    static constexpr int kFan = kCode + 1;
    static constexpr int kN = kFan + 2 * NF;
    float fb0;  // the fan's first inverse temperature

    __device__ __forceinline__ void identity(float (&a)[kN]) const {
        a[0] = -INFINITY;
#pragma unroll
        for (int i = 1; i < kN; ++i) a[i] = 0.0f;
    }
    __device__ __forceinline__ void combine(float (&a)[kN],
                                            const float (&b)[kN]) const {
        const float m = fmaxf(a[0], b[0]);
        const float da = __fmul_rn(__fsub_rn(a[0], m), kLog2e);
        const float db = __fmul_rn(__fsub_rn(b[0], m), kLog2e);
        const float fa = ex2(da), fb = ex2(db);
        const bool la = a[1] > 0.0f, lb = b[1] > 0.0f;
        const float aS = la ? __fmul_rn(fa, a[1]) : 0.0f;
        const float bS = lb ? __fmul_rn(fb, b[1]) : 0.0f;
        const float aV = la ? __fmul_rn(fa, __fmaf_rn(da, a[1], a[2])) : 0.0f;
        const float bV = lb ? __fmul_rn(fb, __fmaf_rn(db, b[1], b[2])) : 0.0f;
        if (NF == 0) {
            const int iW = NF == 0 ? 3 : 0;
            const float aW = la ? __fmul_rn(fa, __fmaf_rn(da, __fmaf_rn(da, a[1], __fmul_rn(2.0f, a[2])), a[iW]))
                                : 0.0f;
            const float bW = lb ? __fmul_rn(fb, __fmaf_rn(db, __fmaf_rn(db, b[1], __fmul_rn(2.0f, b[2])), b[iW]))
                                : 0.0f;
            a[iW] = __fadd_rn(aW, bW);
        } else {
            float ga = ex2(__fmul_rn(fb0, da));
            float gb = ex2(__fmul_rn(fb0, db));
#pragma unroll
            for (int k = 0; k < NF; ++k) {
                if (k > 0) {
                    ga = __fmul_rn(ga, ga);
                    ga = __fmul_rn(ga, ga);
                    gb = __fmul_rn(gb, gb);
                    gb = __fmul_rn(gb, gb);
                }
                const int iS = kFan + 2 * k, iV = kFan + 1 + 2 * k;
                const bool lka = a[iS] > 0.0f, lkb = b[iS] > 0.0f;
                const float sa = lka ? __fmul_rn(ga, a[iS]) : 0.0f;
                const float va = lka ? __fmul_rn(ga, __fmaf_rn(da, a[iS], a[iV])) : 0.0f;
                const float sb = lkb ? __fmul_rn(gb, b[iS]) : 0.0f;
                const float vb = lkb ? __fmul_rn(gb, __fmaf_rn(db, b[iS], b[iV])) : 0.0f;
                a[iS] = __fadd_rn(sa, sb);
                a[iV] = __fadd_rn(va, vb);
            }
        }
        a[0] = m;
        a[1] = __fadd_rn(aS, bS);
        a[2] = __fadd_rn(aV, bV);
        a[kCode] = fmaxf(a[kCode], b[kCode]);
    }
    // Moves a's sums from its own max a[0] to m >= a[0]: one side of
    // combine, the same scalings.  An empty a (S = 0) becomes zeros.
    __device__ __forceinline__ void rescale(float (&a)[kN], float m) const {
        const float da = __fmul_rn(__fsub_rn(a[0], m), kLog2e);
        const float fa = ex2(da);
        const bool la = a[1] > 0.0f;
        const float S = a[1], V = a[2];
        a[0] = m;
        a[1] = la ? __fmul_rn(fa, S) : 0.0f;
        a[2] = la ? __fmul_rn(fa, __fmaf_rn(da, S, V)) : 0.0f;
        if (NF == 0) {
            const int iW = NF == 0 ? 3 : 0;
            a[iW] = la ? __fmul_rn(fa, __fmaf_rn(da, __fmaf_rn(da, S, __fmul_rn(2.0f, V)), a[iW]))
                       : 0.0f;
        } else {
            float ga = ex2(__fmul_rn(fb0, da));
#pragma unroll
            for (int k = 0; k < NF; ++k) {
                if (k > 0) {
                    ga = __fmul_rn(ga, ga);
                    ga = __fmul_rn(ga, ga);
                }
                const int iS = kFan + 2 * k, iV = kFan + 1 + 2 * k;
                const bool lka = a[iS] > 0.0f;
                const float Sk = a[iS];
                a[iS] = lka ? __fmul_rn(ga, Sk) : 0.0f;
                a[iV] = lka ? __fmul_rn(ga, __fmaf_rn(da, Sk, a[iV])) : 0.0f;
            }
        }
    }
};
using OpSoftmax = OpSoftmaxT<0>;

// Shuffle-tree all-reduce over the warp; every lane ends with the same
// (bit-identical) values.
template <class Op, int NV>
__device__ __forceinline__ void warp_reduce(float (&a)[NV], const Op& op) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        float b[NV];
#pragma unroll
        for (int i = 0; i < NV; ++i) b[i] = __shfl_xor_sync(0xffffffffu, a[i], o);
        op.combine(a, b);
    }
}

// The cluster step of a reduction: pushes this warp's a[0..NV) (the same
// in every lane) into slot (rank, warp) of every CTA of the cluster, waits
// until all the cluster's slots of this exchange have landed, and leaves in
// each lane the Op fold of slots lane, lane + 32, ... (Op's identity in a
// lane without one).
template <bool CLUSTER, class Op, int NV>
__device__ __forceinline__ void push_fold(float (&a)[NV], const Smem& sm,
                                          Exch& x, const Op& op) {
    static_assert(NV <= kSlotVals, "payload");
    constexpr int NE = NV + (NV & 1);   // pushed as pairs
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t buf = x.xk & 1u;
    const uint32_t parity = (x.xk >> 1) & 1u;
    ++x.xk;
    const int nslot = x.n * x.warps;
    float* cs = sm.cslot + buf * nslot * kSlotVals;
    const int mine = static_cast<int>(x.rank) * x.warps + warp;
    if (!x.dead) {
        if (CLUSTER) {
            if (threadIdx.x == 0)
                mbar_arrive_expect_tx(&sm.cbar[buf], nslot * NE * 4);
            if (lane < x.n) {
                const uint32_t bar = map_to_rank(smem_addr(&sm.cbar[buf]), lane);
                const uint32_t dst = map_to_rank(smem_addr(&cs[mine * kSlotVals]), lane);
#pragma unroll
                for (int i = 0; i < NE; i += 2) {
                    const float hi_half = (i + 1 < NV) ? a[(i + 1 < NV) ? i + 1 : 0] : 0.0f;
                    push_pair(dst + 4 * i, a[i], hi_half, bar);
                }
            }
        } else if (lane == 0) {
#pragma unroll
            for (int i = 0; i < NV; ++i) cs[mine * kSlotVals + i] = a[i];
            mbar_arrive(&sm.cbar[buf]);
        }
        if (!mbar_wait<CLUSTER>(&sm.cbar[buf], parity, x.limit)) x.dead = true;
    }
    // A slot is kSlotVals floats, 16-byte aligned: NV values in
    // (NV + 3) / 4 128-bit loads.
    auto load_slot = [&](int k, float (&b)[NV]) {
        constexpr int NQ = (NV + 3) / 4;
        float v[4 * NQ];
        const float4* s4 = reinterpret_cast<const float4*>(&cs[k * kSlotVals]);
#pragma unroll
        for (int c = 0; c < NQ; ++c) {
            const float4 q = s4[c];
            v[4 * c] = q.x;
            v[4 * c + 1] = q.y;
            v[4 * c + 2] = q.z;
            v[4 * c + 3] = q.w;
        }
#pragma unroll
        for (int i = 0; i < NV; ++i) b[i] = v[i];
    };
    // The lane's first slot is taken as it is (combining it with the
    // identity would give the same values).
    int k = lane;
    if (k < nslot) {
        load_slot(k, a);
        k += 32;
    } else {
        op.identity(a);
    }
    for (; k < nslot; k += 32) {
        float b[NV];
        load_slot(k, b);
        op.combine(a, b);
    }
}

// Reduction (Op) over every thread of the CTA and the cluster of each
// thread's a[0..NV); returns the same bits in every thread of the cluster.
template <bool CLUSTER, class Op, int NV>
__device__ __forceinline__ void exchange(float (&a)[NV], const Smem& sm,
                                         Exch& x, const Op& op) {
    warp_reduce<Op, NV>(a, op);
    push_fold<CLUSTER, Op, NV>(a, sm, x, op);
    warp_reduce<Op, NV>(a, op);
}

// The softmax statistics (OpSoftmaxT) reduced over the warp: the max first
// (a butterfly of one value), then every lane's partial moved to it once
// (rescale) and the sums added (the code by max).  The same bits in every
// lane, and one rescaling per partial where a combine tree rescales at
// every level.
template <int NF>
__device__ __forceinline__ void softmax_warp_reduce(float (&a)[OpSoftmaxT<NF>::kN],
                                                    const OpSoftmaxT<NF>& op) {
    using Op = OpSoftmaxT<NF>;
    float m = a[0];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    op.rescale(a, m);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        float b[Op::kN];
#pragma unroll
        for (int i = 1; i < Op::kN; ++i) b[i] = __shfl_xor_sync(0xffffffffu, a[i], o);
#pragma unroll
        for (int i = 1; i < Op::kN; ++i)
            a[i] = i == Op::kCode ? fmaxf(a[i], b[i]) : __fadd_rn(a[i], b[i]);
    }
}

// exchange() for the softmax statistics: the warp and the cluster stages
// each take the max first (softmax_warp_reduce); a lane folding more than
// one slot combines them with op.
template <bool CLUSTER, int NF>
__device__ __forceinline__ void softmax_exchange(float (&a)[OpSoftmaxT<NF>::kN],
                                                 const Smem& sm, Exch& x,
                                                 const OpSoftmaxT<NF>& op) {
    softmax_warp_reduce<NF>(a, op);
    push_fold<CLUSTER, OpSoftmaxT<NF>, OpSoftmaxT<NF>::kN>(a, sm, x, op);
    softmax_warp_reduce<NF>(a, op);
}

// Accumulators of S, V and (optionally) W at one inverse temperature: lanes
// (x, y) and (z, w) of each float4 go to the two halves of a packed pair.
// Each packed fp32x2 operation occupies both FMA sub-pipes, so the pass
// with W (10 packed operations per float4) is bound by the FMA pipes and
// the one without (6 per float4) by the ex2 unit: W is accumulated only
// where a Newton step will use it.
template <bool WITH_W>
struct Acc {
    float2 s, v, w;
    __device__ __forceinline__ void zero() {
        s = v = w = make_float2(0.f, 0.f);
    }
    // Adds the four classes of y at inverse temperature beta, b2 = {beta,
    // beta}, with x = beta (y + d) computed as fma(y, beta, bd2), bd2 =
    // {beta d, beta d}: y is stored relative to this thread's max, d is
    // that max's offset from the row's (V and W are kept relative to the
    // thread's max; thread_to_row() moves them).  UNIT: beta = 1 and
    // d = 0 (the T = 1 pass), where x = y exactly and the fma is skipped.
    template <bool UNIT = false>
    __device__ __forceinline__ void add(float4 y, float2 b2, float2 bd2) {
        const float2 y01 = make_float2(y.x, y.y);
        const float2 y23 = make_float2(y.z, y.w);
        const float2 x01 = UNIT ? y01 : fma2(y01, b2, bd2);
        const float2 x23 = UNIT ? y23 : fma2(y23, b2, bd2);
        const float2 e01 = make_float2(ex2(x01.x), ex2(x01.y));
        const float2 e23 = make_float2(ex2(x23.x), ex2(x23.y));
        s = add2(s, add2(e01, e23));
        if (WITH_W) {
            const float2 ey01 = mul2(e01, y01);
            const float2 ey23 = mul2(e23, y23);
            v = add2(v, add2(ey01, ey23));
            w = fma2(ey01, y01, w);
            w = fma2(ey23, y23, w);
        } else {
            v = fma2(e01, y01, v);
            v = fma2(e23, y23, v);
        }
    }
};

// V and W relative to this thread's max moved to the row's: y + d for y.
__device__ __forceinline__ void thread_to_row(float S, float& V, float* W,
                                              float d) {
    if (W) *W = fmaf(d, fmaf(d, S, 2.0f * V), *W);
    V = fmaf(d, S, V);
}

// T = 1 pass over this thread's float4s of the slice (q = t, t + nt, ...,
// the float4s it staged): rewrites them as y = max((l - m_t) log2 e, floor)
// with m_t this thread's max, and returns {m_t, S, V, W, code} relative to
// m_t for the softmax reduction (no W with a fan; the layout of
// OpSoftmaxT<NF>), followed by (S_k, V_k) at the NF fan
// points b_k = fb0 4^k, also relative to m_t: 2^(b_0 y) from the ex2 unit,
// each next power the previous squared twice.
template <int NF>
__device__ __forceinline__ void transform_pass(float4* row4, int q4, float m_t,
                                               float code, float fb0,
                                               float (&out)[OpSoftmaxT<NF>::kN]) {
    Acc<NF == 0> acc;  // W at T = 1 only without a fan (out[3] = 0 with one)
    acc.zero();
    float2 fs[NF > 0 ? NF : 1], fv[NF > 0 ? NF : 1];
#pragma unroll
    for (int k = 0; k < NF; ++k) fs[k] = fv[k] = make_float2(0.f, 0.f);
    const float2 one = make_float2(1.0f, 1.0f);
    const float2 zero = make_float2(0.0f, 0.0f);
    const float2 fb2 = make_float2(fb0, fb0);
    // (l - m_t) log2 e, floored, two lanes per packed operation (the same
    // roundings as the scalar subtract and multiply).
    const float2 neg_m = make_float2(-m_t, -m_t);
    const float2 l2e = make_float2(kLog2e, kLog2e);
    auto to_y = [neg_m, l2e](float4 l) {
        const float2 a = mul2(add2(make_float2(l.x, l.y), neg_m), l2e);
        const float2 b = mul2(add2(make_float2(l.z, l.w), neg_m), l2e);
        return make_float4(fmaxf(a.x, kYFloor), fmaxf(a.y, kYFloor),
                           fmaxf(b.x, kYFloor), fmaxf(b.y, kYFloor));
    };
    auto add_all = [&](float4 y) {
        acc.template add<true>(y, one, zero);
        if (NF > 0) {
            const float2 y01 = make_float2(y.x, y.y);
            const float2 y23 = make_float2(y.z, y.w);
            const float2 x01 = mul2(y01, fb2);
            const float2 x23 = mul2(y23, fb2);
            float2 e01 = make_float2(ex2(x01.x), ex2(x01.y));
            float2 e23 = make_float2(ex2(x23.x), ex2(x23.y));
#pragma unroll
            for (int k = 0; k < NF; ++k) {
                if (k > 0) {
                    e01 = mul2(e01, e01);
                    e01 = mul2(e01, e01);
                    e23 = mul2(e23, e23);
                    e23 = mul2(e23, e23);
                }
                fs[k] = add2(fs[k], add2(e01, e23));
                fv[k] = fma2(e01, y01, fv[k]);
                fv[k] = fma2(e23, y23, fv[k]);
            }
        }
    };
    // Four float4s per trip (independent chains), then the rest one by one.
    const int nt = blockDim.x;
    int q = threadIdx.x;
    for (; q + 3 * nt < q4; q += 4 * nt) {
        float4 y[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) y[i] = to_y(row4[q + i * nt]);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            row4[q + i * nt] = y[i];
            add_all(y[i]);
        }
    }
    // At most three left: a pair, then a single.
    if (q + nt < q4) {
        const float4 ya = to_y(row4[q]);
        const float4 yb = to_y(row4[q + nt]);
        row4[q] = ya;
        row4[q + nt] = yb;
        add_all(ya);
        add_all(yb);
        q += 2 * nt;
    }
    if (q < q4) {
        const float4 y = to_y(row4[q]);
        row4[q] = y;
        add_all(y);
    }
    constexpr int kCode = OpSoftmaxT<NF>::kCode, kFan = OpSoftmaxT<NF>::kFan;
    out[0] = m_t;
    out[1] = acc.s.x + acc.s.y;
    out[2] = acc.v.x + acc.v.y;
    if (NF == 0) out[3] = acc.w.x + acc.w.y;
    out[kCode] = code;
#pragma unroll
    for (int k = 0; k < NF; ++k) {
        out[kFan + 2 * k] = fs[k].x + fs[k].y;
        out[kFan + 1 + 2 * k] = fv[k].x + fv[k].y;
    }
}

// Number of partial sums a pass at P temperatures produces: S and V per
// point, plus W of point 0 when W0.
template <int P, bool W0>
struct PassOut {
    static constexpr int kN = 2 * P + (W0 ? 1 : 0);
    // Index of point p's S (its V follows).
    static __device__ __forceinline__ constexpr int s_idx(int p) {
        return p == 0 ? 0 : 2 * p + (W0 ? 1 : 0);
    }
};

// One pass over this thread's float4s of the slice at P inverse
// temperatures; out holds PassOut<P, W0>'s layout (W of point 0 at index 2).
// Thread t owns float4s t, t + nt, ... (four per trip, then one by one).
template <int P, bool W0>
__device__ __forceinline__ void eval_pass(const float4* row4, int q4,
                                          const float (&beta)[kMaxPoints],
                                          float d,
                                          float (&out)[PassOut<P, W0>::kN]) {
    Acc<W0> a0;
    Acc<false> ap[P > 1 ? P - 1 : 1];
    float2 b2[P], bd2[P];
    a0.zero();
#pragma unroll
    for (int p = 0; p < P; ++p) {
        if (p > 0) ap[p - 1].zero();
        b2[p] = make_float2(beta[p], beta[p]);
        bd2[p] = make_float2(beta[p] * d, beta[p] * d);
    }
    const int nt = blockDim.x;
    int q = threadIdx.x;
    for (; q + 3 * nt < q4; q += 4 * nt) {
        float4 y[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) y[i] = row4[q + i * nt];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            a0.add(y[i], b2[0], bd2[0]);
#pragma unroll
            for (int p = 1; p < P; ++p) ap[p - 1].add(y[i], b2[p], bd2[p]);
        }
    }
    // At most three left: a pair, then a single.
    if (q + nt < q4) {
        const float4 ya = row4[q];
        const float4 yb = row4[q + nt];
        a0.add(ya, b2[0], bd2[0]);
        a0.add(yb, b2[0], bd2[0]);
#pragma unroll
        for (int p = 1; p < P; ++p) {
            ap[p - 1].add(ya, b2[p], bd2[p]);
            ap[p - 1].add(yb, b2[p], bd2[p]);
        }
        q += 2 * nt;
    }
    if (q < q4) {
        const float4 ya = row4[q];
        a0.add(ya, b2[0], bd2[0]);
#pragma unroll
        for (int p = 1; p < P; ++p) ap[p - 1].add(ya, b2[p], bd2[p]);
    }
    {
        const float S0 = a0.s.x + a0.s.y;
        float V0 = a0.v.x + a0.v.y;
        float W0v = a0.w.x + a0.w.y;
        thread_to_row(S0, V0, W0 ? &W0v : nullptr, d);
        out[0] = S0;
        out[1] = V0;
        if (W0) out[2 % PassOut<P, W0>::kN] = W0v;
    }
#pragma unroll
    for (int p = 1; p < P; ++p) {
        const float Sp = ap[p - 1].s.x + ap[p - 1].s.y;
        float Vp = ap[p - 1].v.x + ap[p - 1].v.y;
        thread_to_row(Sp, Vp, nullptr, d);
        out[PassOut<P, W0>::s_idx(p)] = Sp;
        out[PassOut<P, W0>::s_idx(p) + 1] = Vp;
    }
}

// One search round with P grid points J: pass, exchange, update.  W0: the
// next round takes a Newton step from point 0, which needs its W.  d: this
// thread's offset (its max's y relative to the row's).
template <bool CLUSTER, int P, bool W0>
__device__ __forceinline__ void search_round(Search& st, const SearchCfg& cfg,
                                             const int (&J)[kMaxPoints],
                                             const float4* row4, int q4,
                                             float d, const Smem& sm, Exch& x) {
    float beta[kMaxPoints];
#pragma unroll
    for (int p = 0; p < kMaxPoints; ++p)
        beta[p] = p < P ? rcp_approx(cfg.g.at(J[p])) : 1.0f;
    constexpr int NV = PassOut<P, W0>::kN;
    float a[NV];
    eval_pass<P, W0>(row4, q4, beta, d, a);
    exchange<CLUSTER, OpSum, NV>(a, sm, x, OpSum{});
    float S[kMaxPoints], V[kMaxPoints], W[kMaxPoints];
#pragma unroll
    for (int p = 0; p < kMaxPoints; ++p) {
        const int i = PassOut<P, W0>::s_idx(p < P ? p : 0);
        S[p] = p < P ? a[i] : 1.0f;
        V[p] = p < P ? a[i + 1] : 0.0f;
        W[p] = 0.0f;
    }
    if (W0) W[0] = a[2 % NV];
    search_update(st, cfg, P, J, beta, S, V, W, W0);
}

__device__ __forceinline__ void store_scalar_lanes(float* dst, int q, int pad,
                                                   int len, float4 p) {
    const int j0 = 4 * q - pad;
    const float v[4] = {p.x, p.y, p.z, p.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int j = j0 + i;
        if (j >= 0 && j < len) dst[j] = v[i];
    }
}

// Output pass over this thread's float4s (q = t, t + nt, ...): p =
// 2^(beta (y + d)) * inv_s (or zeros) into dst[0, len).
__device__ __forceinline__ void write_out(const float4* row4, const Slice& s,
                                          float* dst, float beta, float d,
                                          float inv_s, bool zero) {
    const int pad_o = static_cast<int>((reinterpret_cast<uintptr_t>(dst) >> 2) & 3);
    const bool vec = pad_o == s.pad;
    const float2 b2 = make_float2(beta, beta);
    const float2 bd2 = make_float2(beta * d, beta * d);
    const float2 i2 = make_float2(inv_s, inv_s);
    auto prob = [&](int q) {
        if (zero) return make_float4(0.f, 0.f, 0.f, 0.f);
        const float4 y = row4[q];
        const float2 x01 = fma2(make_float2(y.x, y.y), b2, bd2);
        const float2 x23 = fma2(make_float2(y.z, y.w), b2, bd2);
        const float2 p01 = mul2(make_float2(ex2(x01.x), ex2(x01.y)), i2);
        const float2 p23 = mul2(make_float2(ex2(x23.x), ex2(x23.y)), i2);
        return make_float4(p01.x, p01.y, p23.x, p23.y);
    };
    const int nt = blockDim.x;
    int q = threadIdx.x;
    if (!vec) {
        // The output's alignment differs from the input's: element stores.
        for (; q < s.q4; q += nt)
            store_scalar_lanes(dst, q, s.pad, s.len, prob(q));
        return;
    }
    // Ragged head, aligned body four float4s per trip, ragged tail.
    float* const db = dst - s.pad;  // float4 q of the body is at db + 4q
    if (q < s.qb0) {
        store_scalar_lanes(dst, q, s.pad, s.len, prob(q));
        q += nt;
    }
    for (; q + 3 * nt < s.qb1; q += 4 * nt) {
        float4 p[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) p[i] = prob(q + i * nt);
#pragma unroll
        for (int i = 0; i < 4; ++i)
            __stcs(reinterpret_cast<float4*>(db + 4 * (q + i * nt)), p[i]);
    }
    // At most three left in the body: a pair, then a single.
    if (q + nt < s.qb1) {
        const float4 pa = prob(q), pb = prob(q + nt);
        __stcs(reinterpret_cast<float4*>(db + 4 * q), pa);
        __stcs(reinterpret_cast<float4*>(db + 4 * (q + nt)), pb);
        q += 2 * nt;
    }
    if (q < s.qb1) {
        __stcs(reinterpret_cast<float4*>(db + 4 * q), prob(q));
        q += nt;
    }
    if (q < s.q4) store_scalar_lanes(dst, q, s.pad, s.len, prob(q));
}

// MAXT: largest block the instantiation is launched with; MINB: blocks per
// SM the register allocation must allow (256 threads x 3 blocks for the
// throughput plans, 512 x 1 for the latency plans); ASYNC: stage with
// asynchronous copies (a compile-time choice: a run-time branch between
// the two staging loops cost the other path 1.4% at 32 x 50000).
template <bool CLUSTER, int MAXT, int MINB, bool ASYNC, class In, bool FAN>
__global__ void __launch_bounds__(MAXT, MINB)
cluster_kernel(RowTask t, int n, int slice_len) {
    extern __shared__ __align__(128) unsigned char smem[];
    const int nt = blockDim.x;
    const int warps = nt >> 5;
    const uint32_t rank = CLUSTER ? cluster_ctarank() : 0u;
    const int64_t cid = blockIdx.x / n;
    const int64_t ncl = gridDim.x / n;

    Smem sm;
    {
        const ClusterSmemLayout L = cluster_smem_layout(warps, n);
        sm.cslot = reinterpret_cast<float*>(smem + L.cslot);
        sm.cbar = reinterpret_cast<uint64_t*>(smem + L.cbar);
        sm.row4 = reinterpret_cast<float4*>(smem + L.row);
    }
    float4* row4 = sm.row4;

    if (threadIdx.x == 0) {
        // In a cluster each phase completes on one arrival (with the
        // expected bytes of the cluster's pushes); without one, on one
        // arrival per warp.
        const uint32_t count = CLUSTER ? 1u : static_cast<uint32_t>(warps);
        mbar_init(&sm.cbar[0], count);
        mbar_init(&sm.cbar[1], count);
        fence_mbar_init();
    }
    __syncthreads();
    // Peers push into this CTA's slots only after every CTA's mbarriers are
    // initialised: arrive now, wait just before the first exchange, so that
    // the cluster barrier's latency overlaps the first row's staging.
    if (CLUSTER) cluster_arrive();
    bool waited = false;

    const int64_t C = t.num_classes;
    const int64_t s0 = static_cast<int64_t>(rank) * slice_len;
    const int len = static_cast<int>(max(static_cast<int64_t>(0),
                                         min(static_cast<int64_t>(slice_len), C - s0)));
    const SearchCfg cfg{t.t_min, t.hi0, t.entropy_bound,
                        t.entropy_bound * kLog2e,
                        t.entropy_bound > 0.0f ? lg2_approx(t.entropy_bound) : 0.0f,
                        make_grid(t.t_min, fmaxf(t.hi0, t.t_min), t.max_iter)};
    Exch x{warps, n, rank, 0u, t.wait_limit_cycles, false};
    bool reported = false;
    // The fan (FAN instantiations, few-row launches): kFanPoints
    // temperatures evaluated with the T = 1 pass, which place the search's
    // first point.
    const int nfan = (FAN && t.fan_beta0 > 0.0f && !t.strict) ? kFanPoints : 0;

    for (int64_t r = cid; r < t.batch; r += ncl) {
        const typename In::T* src =
            static_cast<const typename In::T*>(t.logits) + r * C + s0;
        const Slice s = make_slice<In>(src, len);

        // Stage: thread t copies float4s q = t, t + nt, ... of the slice
        // (the float4s it owns in every later pass) into shared memory and
        // folds them into its own max and the finiteness check; the ragged
        // head and tail go element by element.  Launches with several CTAs
        // per SM (async_stage) copy the aligned body as 16-byte
        // asynchronous copies, all in flight at once, and fold after they
        // land (4096 x 32000: 4% faster, 256 x 131072: 8%); launches of
        // about one CTA per SM load it eight float4s at a time and fold
        // each trip as it arrives (32 x 50000: 0.5% faster than the copies,
        // the folding overlaps the next trip).  (Bulk copies were slower:
        // one SM's bulk-copy traffic arrived at about 16 bytes per clock,
        // against about 22 for per-thread loads with this many in flight.)
        float m_t = -INFINITY;  // this thread's max
        float bad = 0.0f;       // becomes NaN if any element is NaN or +-Inf
        bool nan_seen = false;
        auto load_ragged = [&](int q) {
            float e[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int j = 4 * q + i - s.pad;
                e[i] = -INFINITY;
                if (j >= 0 && j < s.len) {
                    e[i] = In::get(src + j);
                    m_t = fmaxf(m_t, e[i]);
                    bad = fmaf(e[i], 0.0f, bad);
                    nan_seen = nan_seen || isnan(e[i]);
                }
            }
            row4[q] = make_float4(e[0], e[1], e[2], e[3]);
        };
        auto fold = [&](float4 v) {
            m_t = fmaxf(m_t, fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w)));
            bad = fmaf(v.x, 0.0f, bad);
            bad = fmaf(v.y, 0.0f, bad);
            bad = fmaf(v.z, 0.0f, bad);
            bad = fmaf(v.w, 0.0f, bad);
        };
        {
            const typename In::T* gb = src - s.pad;  // float4 q of the body is at gb + 4q
            int q = threadIdx.x;
            if (q < s.qb0) {
                load_ragged(q);
                q += nt;
            }
            if (ASYNC) {
                // Each thread copies its own float4 slots, so after its own
                // wait it may widen (bf16) and fold them without a barrier.
                const int qb = q;
                for (; q < s.qb1; q += nt) In::copy4_async(&row4[q], gb + 4 * q);
                if (q < s.q4) load_ragged(q);
                cp_async_wait_all();
                for (q = qb; q + 3 * nt < s.qb1; q += 4 * nt) {
                    float4 v[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) v[i] = In::widen(row4[q + i * nt]);
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        if (In::kBytes != 4) row4[q + i * nt] = v[i];
                        fold(v[i]);
                    }
                }
                for (; q < s.qb1; q += nt) {
                    const float4 v = In::widen(row4[q]);
                    if (In::kBytes != 4) row4[q] = v;
                    fold(v);
                }
            } else {
                for (; q + 7 * nt < s.qb1; q += 8 * nt) {
                    float4 v[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) v[i] = In::get4(gb + 4 * (q + i * nt));
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        row4[q + i * nt] = v[i];
                        fold(v[i]);
                    }
                }
                for (; q < s.qb1; q += nt) {
                    const float4 v = In::get4(gb + 4 * q);
                    row4[q] = v;
                    fold(v);
                }
                if (q < s.q4) load_ragged(q);
            }
        }
        // Classify a non-finite slice (rare): 2 = NaN seen, 1 = only Inf.
        // Each thread rescans only the float4s it stored itself.
        float code = 0.0f;
        if (bad != bad) {
            for (int q = threadIdx.x < s.qb0 ? threadIdx.x + nt : threadIdx.x;
                 q < s.qb1; q += nt) {
                const float4 v = row4[q];
                if (isnan(v.x) || isnan(v.y) || isnan(v.z) || isnan(v.w))
                    nan_seen = true;
            }
            code = nan_seen ? 2.0f : 1.0f;
        }
        // T = 1 pass relative to this thread's max (with the fan's points
        // when there is one), then one reduction that forms the row's max,
        // its S, V, W at T = 1 and the fan's sums (rescaled to that max) and
        // its NaN/Inf code: no separate exchange of the max.
        // The reduced sums: {m, S, V, W, code} at T = 1 and (Sf, Vf) at the
        // fan's points.
        float s1[5];
        float Sf[kFanPoints] = {0.0f, 0.0f, 0.0f}, Vf[kFanPoints] = {0.0f, 0.0f, 0.0f};
        if (FAN && nfan > 0) {
            using OpF = OpSoftmaxT<kFanPoints>;
            float sf[OpF::kN];
            transform_pass<kFanPoints>(row4, s.q4, m_t, code, t.fan_beta0, sf);
            if (CLUSTER && !waited) {
                cluster_wait();
                waited = true;
            }
            softmax_exchange<CLUSTER, kFanPoints>(sf, sm, x, OpF{t.fan_beta0});
            s1[0] = sf[0];
            s1[1] = sf[1];
            s1[2] = sf[2];
            s1[3] = 0.0f;
            s1[4] = sf[OpF::kCode];
#pragma unroll
            for (int k = 0; k < kFanPoints; ++k) {
                Sf[k] = sf[OpF::kFan + 2 * k];
                Vf[k] = sf[OpF::kFan + 1 + 2 * k];
            }
        } else {
            transform_pass<0>(row4, s.q4, m_t, code, 0.0f, s1);
            if (CLUSTER && !waited) {
                cluster_wait();
                waited = true;
            }
            softmax_exchange<CLUSTER, 0>(s1, sm, x, OpSoftmax{0.0f});
        }
        const float m = s1[0];
        const int row_code = static_cast<int>(s1[4]);
        // This thread's y offset: y (row) = y (stored) + d.
        const float d = m_t > -INFINITY ? (m_t - m) * kLog2e : 0.0f;

        float* dst = t.out + r * C + s0;
        unsigned int bits = 0;
        int evals = 1 + (row_code == 0 ? nfan : 0);  // the T = 1 pass and the fan
        float T_row = NAN;
        float beta_out = 0.0f, inv_s = 0.0f;
        const bool searching =
            row_code == 0 && entropy_above(make_float2(s1[1], s1[2]), 1.0f, cfg.bound_bits);
        if (row_code != 0) {
            bits = row_code == 2 ? kBitNan : kBitInf;
        } else if (!searching) {
            T_row = 1.0f;
            beta_out = 1.0f;
            inv_s = 1.0f / s1[1];
        } else {
            Search st = search_begin(cfg, s1[1], s1[2], s1[3], t.strict != 0);
            if (!(cfg.t_min < cfg.hi0)) {
                // No interval to halve: T = t_min (section 5.4 check).
                st.f |= kFinal;
                const int J1[kMaxPoints] = {0, 0, 0};
                search_round<CLUSTER, 1, false>(st, cfg, J1, row4, s.q4, d, sm, x);
                ++evals;
            } else if (FAN && nfan > 0) {
                const float b0 = t.fan_beta0;
                const float fbeta[kFanPoints] = {b0, 4.0f * b0, 16.0f * b0};
                search_fan(st, cfg, fbeta, Sf, Vf, s1[1], s1[2]);
            }
            // One round per trip: plan (0 points: the search is over), then
            // the round's shape, one of five instantiations.
            while (true) {
                int J[kMaxPoints] = {0, 0, 0};
                const int np = (st.f & kDone) ? 0 : search_plan(st, cfg, J);
                const bool w0 = newton_next(st);
                if (np == 0) break;
                evals += np;
                if (np == 1 && w0)
                    search_round<CLUSTER, 1, true>(st, cfg, J, row4, s.q4, d, sm, x);
                else if (np == 1)
                    search_round<CLUSTER, 1, false>(st, cfg, J, row4, s.q4, d, sm, x);
                else if (np == 2 && w0)
                    search_round<CLUSTER, 2, true>(st, cfg, J, row4, s.q4, d, sm, x);
                else if (np == 2)
                    search_round<CLUSTER, 2, false>(st, cfg, J, row4, s.q4, d, sm, x);
                else
                    search_round<CLUSTER, 3, false>(st, cfg, J, row4, s.q4, d, sm, x);
            }
            if (st.f & kOverflow) bits |= kBitOverflow;
            T_row = search_result_T(st, cfg);
            beta_out = rcp_approx(T_row);
            inv_s = 1.0f / st.SA;
        }
        write_out(row4, s, dst, beta_out, d, inv_s, row_code != 0);
        if (rank == 0 && threadIdx.x == 0) {
            if (t.t_out) t.t_out[r] = T_row;
            if (t.evals_out) t.evals_out[r] = evals + (row_code != 0 ? 0 : 1);
            raise_error(t.err, bits);
        }
        if (x.dead && !reported) {
            raise_error(t.err, kBitTimeout);
            reported = true;
        }
        // The slice buffer is rewritten by the next row's loads.
        __syncthreads();
    }
    if (CLUSTER) {
        if (!waited) cluster_wait();
        // No cluster barrier at the end: every CTA of the cluster runs the
        // same exchanges, and once this CTA's last exchange has completed,
        // every push into its slots has landed and no peer will touch them
        // again.  After a timeout that no longer holds: give pushes that
        // peers had already issued time to land before the CTA exits (a
        // bounded sleep; st.async completes within microseconds).
        if (__syncthreads_or(x.dead)) {
            for (int i = 0; i < 1000; ++i) __nanosleep(1000);
        }
    }
}

template <bool CLUSTER, int MAXT, int MINB, bool ASYNC, class In, bool FAN = false>
cudaError_t launch_one(const RowTask& task, int cluster_size, int slice_len,
                       int threads, int smem_bytes, int64_t grid_ctas,
                       cudaStream_t stream, int attr_slot) {
    auto kern = cluster_kernel<CLUSTER, MAXT, MINB, ASYNC, In, FAN>;
    cudaError_t e = ensure_smem_attribute(reinterpret_cast<const void*>(kern),
                                          attr_slot, smem_bytes, CLUSTER);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid_ctas), 1, 1);
    cfg.blockDim = dim3(static_cast<unsigned>(threads), 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem_bytes);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    if (CLUSTER) {
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = static_cast<unsigned>(cluster_size);
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    } else {
        cfg.attrs = nullptr;
        cfg.numAttrs = 0;
    }
    return cudaLaunchKernelEx(&cfg, kern, task, cluster_size, slice_len);
}

template <bool ASYNC, class In>
cudaError_t launch_cluster_as(const RowTask& task, int cluster_size,
                              int slice_len, int threads, int smem_bytes,
                              int64_t grid_ctas, cudaStream_t stream) {
    const bool narrow = threads <= 256;
    // Attribute slots: fp32 0-7, bf16 19-26 (8-18 belong to the other
    // operations' kernels); the fan instantiations (clusters of CTAs of at
    // most 256 threads, registers for two such CTAs an SM: the fan's one-wave
    // launches need no more) 52-55.
    if (task.fan_beta0 > 0.0f && narrow && cluster_size > 1) {
        const int fslot = 52 + (In::kBytes == 2 ? 2 : 0) + (ASYNC ? 1 : 0);
        return launch_one<true, 256, 2, ASYNC, In, true>(task, cluster_size, slice_len,
                                                         threads, smem_bytes, grid_ctas,
                                                         stream, fslot);
    }
    const int slot = (In::kBytes == 2 ? 19 : 0) + (ASYNC ? 4 : 0) +
                     (cluster_size > 1 ? 1 : 0) + (narrow ? 0 : 2);
    if (cluster_size > 1)
        return narrow ? launch_one<true, 256, 3, ASYNC, In>(task, cluster_size, slice_len,
                                                            threads, smem_bytes, grid_ctas,
                                                            stream, slot)
                      : launch_one<true, 512, 1, ASYNC, In>(task, cluster_size, slice_len,
                                                            threads, smem_bytes, grid_ctas,
                                                            stream, slot);
    return narrow ? launch_one<false, 256, 3, ASYNC, In>(task, 1, slice_len, threads,
                                                         smem_bytes, grid_ctas, stream, slot)
                  : launch_one<false, 512, 1, ASYNC, In>(task, 1, slice_len, threads,
                                                         smem_bytes, grid_ctas, stream, slot);
}

}  // namespace

cudaError_t launch_cluster(const RowTask& task, int cluster_size,
                           int slice_len, int threads, int smem_bytes,
                           int64_t grid_ctas, cudaStream_t stream) {
    if (task.in_bf16)
        return task.async_stage
            ? launch_cluster_as<true, InBF16>(task, cluster_size, slice_len,
                                              threads, smem_bytes, grid_ctas,
                                              stream)
            : launch_cluster_as<false, InBF16>(task, cluster_size, slice_len,
                                               threads, smem_bytes, grid_ctas,
                                               stream);
    return task.async_stage
        ? launch_cluster_as<true, InF32>(task, cluster_size, slice_len, threads,
                                         smem_bytes, grid_ctas, stream)
        : launch_cluster_as<false, InF32>(task, cluster_size, slice_len, threads,
                                          smem_bytes, grid_ctas, stream);
}

}  // namespace cs
