// Cluster kernel: one thread-block cluster of n CTAs per row (n = 1: one CTA
// per row).  Each CTA holds its slice of the row in shared memory for the
// whole search, so the row is read from HBM once and written once.
//
// Method: "BURT-IMMA CUDA Kernel API Reference", section 2.1
// `constrained_softmax`, Description steps 1-4, with the error policy of
// sections 5.3 and 5.4.  Per row:
//   stage   every thread loads its part of the slice with 128-bit loads
//           (eight in flight per thread), stores it to shared memory and
//           folds it into m = max_i l_i (T-independent, computed once) and
//           a finiteness check, which are exchanged across the cluster;
//   T = 1   one pass turns the slice into y_i = (l_i - m) log2(e) in place
//           and sums S = sum 2^y_i, V = sum y_i 2^y_i, W = sum y_i^2 2^y_i;
//           H(1) = ln2 (log2 S - V/S) decides whether a search is needed;
//   search  rounds of the temperature search of cs_search.cuh: each round
//           evaluates (S, V) at 1-3 temperatures in one pass over the slice
//           (plus W at the first one when a Newton step follows) and
//           reduces them; the search returns the bisection's final lo and
//           S(lo);
//   output  p_i = 2^(beta_lo y_i) / S(lo), written with 128-bit streaming
//           stores.
//
// Reduction.  Every warp reduces its partial sums with a shuffle tree and
// writes them to a slot; after a __syncthreads warp 0 reduces the per-warp
// slots with a second shuffle tree.  In a cluster, warp 0 then pushes the
// CTA's sums into every CTA (st.async, counted on an mbarrier), waits for
// the cluster's pushes and adds them in rank order.  Warp 0 broadcasts the
// result through shared memory after a second __syncthreads.  All threads of
// the cluster thus see bit-identical sums and take the same decisions.
// Slots are double-buffered, which is safe because no thread can reach
// exchange k+2 before every thread has left exchange k.
//
// Every wait is bounded (cs::kWaitLimitCycles by default).  A thread whose
// wait times out records CS_ERR_TIMEOUT and from then on neither waits,
// pushes nor issues copies, but keeps the kernel's control flow so that all
// threads still meet at every __syncthreads and cluster barrier.
#include <math.h>

#include "cs_search.cuh"

namespace cs {
namespace {

using namespace csd;

// Geometry of one CTA's slice in shared memory.  Element j of the slice
// lives at row[pad + j], so 16-byte aligned global addresses land on
// 16-byte aligned shared addresses.  Float4 q in [qb0, qb1) comes in by
// 128-bit loads; the head (q = 0 when pad > 0) and tail float4s element by
// element.
struct Slice {
    int pad;
    int len;
    int q4;       // float4s of the slice in shared memory
    int qb0, qb1; // 16-byte aligned body
    int head_q;   // -1 if none
    int tail_q;   // -1 if none
};

__device__ __forceinline__ Slice make_slice(const float* src, int len) {
    Slice s;
    s.pad = static_cast<int>((reinterpret_cast<uintptr_t>(src) >> 2) & 3);
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
    float* cslot;     // [2][n][kSlotVals] cluster slots (double-buffered)
    float* wslot;     // [2][warps][kSlotVals] per-warp slots (double-buffered)
    float* bcast;     // [kSlotVals] broadcast of reduced sums
    uint64_t* cbar;   // [2] cluster-exchange mbarriers
    float4* row4;     // the slice
};

// Exchange state of one thread (every thread runs every exchange).
struct Exch {
    int warps;
    int n;
    uint32_t rank;
    uint32_t lk;      // exchanges so far (per-warp slot buffer)
    uint32_t xk;      // cluster exchanges so far (cluster slot buffer, phase)
    uint64_t limit;
    bool dead;
};

// Shuffle-tree all-reduce over the warp; every lane ends with the same
// (bit-identical) values.
template <int NV, bool IS_MAX>
__device__ __forceinline__ void warp_reduce(float (&a)[NV]) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            const float b = __shfl_xor_sync(0xffffffffu, a[i], o);
            a[i] = IS_MAX ? fmaxf(a[i], b) : a[i] + b;
        }
    }
}

// Cluster leg: warp 0 pushes the CTA's sums a[0..NV) into slot `rank` of
// every CTA; the waiting threads wait for the cluster's pushes and replace
// a with the combination over ranks, in rank order.  Every thread of the
// CTA calls it (keeping the exchange count); only waiters wait and combine.
template <int NV, bool IS_MAX>
__device__ __forceinline__ void cluster_leg(float (&a)[NV], const Smem& sm,
                                            Exch& x, bool waiter) {
    constexpr int NE = NV + (NV & 1);   // pushed as pairs
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t buf = x.xk & 1u;
    const uint32_t parity = (x.xk >> 1) & 1u;
    ++x.xk;
    float* cs = sm.cslot + buf * x.n * kSlotVals;
    if (!x.dead) {
        if (threadIdx.x == 0) mbar_arrive_expect_tx(&sm.cbar[buf], x.n * NE * 4);
        if (warp == 0 && lane < x.n) {
            const uint32_t bar = map_to_rank(smem_addr(&sm.cbar[buf]), lane);
#pragma unroll
            for (int i = 0; i < NE; i += 2) {
                const uint32_t dst = map_to_rank(
                    smem_addr(&cs[x.rank * kSlotVals + i]), lane);
                const float hi_half = (i + 1 < NV) ? a[(i + 1 < NV) ? i + 1 : 0] : 0.0f;
                push_pair(dst, a[i], hi_half, bar);
            }
        }
        if (waiter && !mbar_wait<true>(&sm.cbar[buf], parity, x.limit))
            x.dead = true;
    }
    if (waiter) {
#pragma unroll
        for (int i = 0; i < NV; ++i) a[i] = cs[i];
        for (int r = 1; r < x.n; ++r) {
#pragma unroll
            for (int i = 0; i < NV; ++i) {
                const float b = cs[r * kSlotVals + i];
                a[i] = IS_MAX ? fmaxf(a[i], b) : a[i] + b;
            }
        }
    }
}

// Sum (or max) over every thread of the CTA and the cluster of each thread's
// a[0..NV); returns the same bits in every thread of the cluster.
template <bool CLUSTER, int NV, bool IS_MAX>
__device__ __forceinline__ void exchange(float (&a)[NV], const Smem& sm,
                                         Exch& x) {
    static_assert(NV <= kSlotVals, "payload");
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    warp_reduce<NV, IS_MAX>(a);
    float* ws = sm.wslot + (x.lk & 1u) * x.warps * kSlotVals;
    ++x.lk;
    if (lane == 0) {
#pragma unroll
        for (int i = 0; i < NV; ++i) ws[warp * kSlotVals + i] = a[i];
    }
    __syncthreads();
    // Warp 0 reduces the per-warp slots (and exchanges across the cluster),
    // then broadcasts.  (Letting every warp reduce the slots and wait on the
    // cluster barrier saves one CTA barrier but measured slower: the extra
    // reductions and waiters cost more than the barrier.)
    if (warp == 0) {
        // Lane groups of w2 >= warps lanes (a power of two) each hold every
        // warp's slot and reduce it with a log2(w2)-level shuffle tree.
        const float idn = IS_MAX ? -INFINITY : 0.0f;
        const int w2 = x.warps <= 4 ? 4 : (x.warps <= 8 ? 8 : 16);
        const int sl = lane & (w2 - 1);
#pragma unroll
        for (int i = 0; i < NV; ++i)
            a[i] = sl < x.warps ? ws[sl * kSlotVals + i] : idn;
        for (int o = w2 >> 1; o > 0; o >>= 1) {
#pragma unroll
            for (int i = 0; i < NV; ++i) {
                const float b = __shfl_xor_sync(0xffffffffu, a[i], o);
                a[i] = IS_MAX ? fmaxf(a[i], b) : a[i] + b;
            }
        }
    }
    if (CLUSTER) cluster_leg<NV, IS_MAX>(a, sm, x, warp == 0);
    if (warp == 0 && lane == 0) {
#pragma unroll
        for (int i = 0; i < NV; ++i) sm.bcast[i] = a[i];
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < NV; ++i) a[i] = sm.bcast[i];
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
    __device__ __forceinline__ void add(float4 y, float2 b2) {
        const float2 y01 = make_float2(y.x, y.y);
        const float2 y23 = make_float2(y.z, y.w);
        const float2 x01 = mul2(y01, b2);
        const float2 x23 = mul2(y23, b2);
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

// T = 1 pass: rewrites this thread's float4s of the slice as
// y = max((l - m) log2 e, floor) and returns the partial S, V, W at beta = 1.
__device__ __forceinline__ void transform_pass(float4* row4, int q4, float m,
                                               float (&out)[3]) {
    Acc<true> acc;
    acc.zero();
    const float2 one = make_float2(1.0f, 1.0f);
    auto to_y = [m](float4 l) {
        return make_float4(fmaxf((l.x - m) * kLog2e, kYFloor),
                           fmaxf((l.y - m) * kLog2e, kYFloor),
                           fmaxf((l.z - m) * kLog2e, kYFloor),
                           fmaxf((l.w - m) * kLog2e, kYFloor));
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
            acc.add(y[i], one);
        }
    }
    for (; q < q4; q += nt) {
        const float4 y = to_y(row4[q]);
        row4[q] = y;
        acc.add(y, one);
    }
    out[0] = acc.s.x + acc.s.y;
    out[1] = acc.v.x + acc.v.y;
    out[2] = acc.w.x + acc.w.y;
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
                                          float (&out)[PassOut<P, W0>::kN]) {
    Acc<W0> a0;
    Acc<false> ap[P > 1 ? P - 1 : 1];
    float2 b2[P];
    a0.zero();
#pragma unroll
    for (int p = 0; p < P; ++p) {
        if (p > 0) ap[p - 1].zero();
        b2[p] = make_float2(beta[p], beta[p]);
    }
    const int nt = blockDim.x;
    int q = threadIdx.x;
    for (; q + 3 * nt < q4; q += 4 * nt) {
        float4 y[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) y[i] = row4[q + i * nt];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            a0.add(y[i], b2[0]);
#pragma unroll
            for (int p = 1; p < P; ++p) ap[p - 1].add(y[i], b2[p]);
        }
    }
    for (; q < q4; q += nt) {
        const float4 ya = row4[q];
        a0.add(ya, b2[0]);
#pragma unroll
        for (int p = 1; p < P; ++p) ap[p - 1].add(ya, b2[p]);
    }
    out[0] = a0.s.x + a0.s.y;
    out[1] = a0.v.x + a0.v.y;
    if (W0) out[2 % PassOut<P, W0>::kN] = a0.w.x + a0.w.y;
#pragma unroll
    for (int p = 1; p < P; ++p) {
        out[PassOut<P, W0>::s_idx(p)] = ap[p - 1].s.x + ap[p - 1].s.y;
        out[PassOut<P, W0>::s_idx(p) + 1] = ap[p - 1].v.x + ap[p - 1].v.y;
    }
}

// One search round with P temperatures: pass, exchange, update.  W0: the
// next round takes a Newton step from point 0, which needs its W.
template <bool CLUSTER, int P, bool W0>
__device__ __forceinline__ void search_round(Search& st, const SearchCfg& cfg,
                                             const float (&T)[kMaxPoints],
                                             const int (&J)[kMaxPoints],
                                             const float4* row4, int q4,
                                             const Smem& sm, Exch& x) {
    float beta[kMaxPoints];
#pragma unroll
    for (int p = 0; p < kMaxPoints; ++p) beta[p] = p < P ? rcp_approx(T[p]) : 1.0f;
    constexpr int NV = PassOut<P, W0>::kN;
    float a[NV];
    eval_pass<P, W0>(row4, q4, beta, a);
    exchange<CLUSTER, NV, false>(a, sm, x);
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

// Output pass: p = 2^(beta y) * inv_s (or zeros) into dst[0, len).
__device__ __forceinline__ void write_out(const float4* row4, const Slice& s,
                                          float* dst, float beta, float inv_s,
                                          bool zero) {
    const int pad_o = static_cast<int>((reinterpret_cast<uintptr_t>(dst) >> 2) & 3);
    const bool vec = pad_o == s.pad;
    const float2 b2 = make_float2(beta, beta);
    const float2 i2 = make_float2(inv_s, inv_s);
    auto prob = [&](int q) {
        if (zero) return make_float4(0.f, 0.f, 0.f, 0.f);
        const float4 y = row4[q];
        const float2 x01 = mul2(make_float2(y.x, y.y), b2);
        const float2 x23 = mul2(make_float2(y.z, y.w), b2);
        const float2 p01 = mul2(make_float2(ex2(x01.x), ex2(x01.y)), i2);
        const float2 p23 = mul2(make_float2(ex2(x23.x), ex2(x23.y)), i2);
        return make_float4(p01.x, p01.y, p23.x, p23.y);
    };
    const int nt = blockDim.x;
    if (!vec) {
        // The output's alignment differs from the input's: element stores.
        for (int q = threadIdx.x; q < s.q4; q += nt)
            store_scalar_lanes(dst, q, s.pad, s.len, prob(q));
        return;
    }
    // Aligned body, four float4s per trip; then the ragged head and tail.
    float* const db = dst - s.pad;  // float4 q of the body is at db + 4q
    int q = s.qb0 + threadIdx.x;
    for (; q + 3 * nt < s.qb1; q += 4 * nt) {
        float4 p[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) p[i] = prob(q + i * nt);
#pragma unroll
        for (int i = 0; i < 4; ++i)
            __stcs(reinterpret_cast<float4*>(db + 4 * (q + i * nt)), p[i]);
    }
    for (; q < s.qb1; q += nt)
        __stcs(reinterpret_cast<float4*>(db + 4 * q), prob(q));
    if (threadIdx.x == 0 && s.head_q >= 0)
        store_scalar_lanes(dst, s.head_q, s.pad, s.len, prob(s.head_q));
    if (threadIdx.x == nt - 1 && s.tail_q >= 0)
        store_scalar_lanes(dst, s.tail_q, s.pad, s.len, prob(s.tail_q));
}

// MAXT: largest block the instantiation is launched with; MINB: blocks per
// SM the register allocation must allow (256 threads x 3 blocks for the
// throughput plans, 512 x 1 for the latency plans).
template <bool CLUSTER, int MAXT, int MINB>
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
        sm.wslot = reinterpret_cast<float*>(smem + L.wslot);
        sm.bcast = reinterpret_cast<float*>(smem + L.bcast);
        sm.cbar = reinterpret_cast<uint64_t*>(smem + L.cbar);
        sm.row4 = reinterpret_cast<float4*>(smem + L.row);
    }
    float* row = reinterpret_cast<float*>(sm.row4);
    float4* row4 = sm.row4;

    if (threadIdx.x == 0) {
        mbar_init(&sm.cbar[0], 1u);
        mbar_init(&sm.cbar[1], 1u);
        fence_mbar_init();
    }
    __syncthreads();
    if (CLUSTER) cluster_sync();

    const int64_t C = t.num_classes;
    const int64_t s0 = static_cast<int64_t>(rank) * slice_len;
    const int len = static_cast<int>(max(static_cast<int64_t>(0),
                                         min(static_cast<int64_t>(slice_len), C - s0)));
    const SearchCfg cfg{t.t_min, t.hi0, t.entropy_bound,
                        t.entropy_bound * kLog2e,
                        make_grid(t.t_min, fmaxf(t.hi0, t.t_min), t.max_iter)};
    Exch x{warps, n, rank, 0u, 0u, t.wait_limit_cycles, false};
    bool reported = false;

    for (int64_t r = cid; r < t.batch; r += ncl) {
        const float* src = t.logits + r * C + s0;
        const Slice s = make_slice(src, len);

        // Stage: every thread loads its float4s of the slice's aligned body
        // with 128-bit streaming loads, eight in flight at a time, stores
        // them to shared memory and folds them into the row max and the
        // finiteness check; threads 0-7 fetch the ragged head/tail float4s
        // element by element.  (Bulk copies into shared memory were slower:
        // one SM's bulk-copy traffic arrived at about 16 bytes per clock,
        // against about 22 for plain loads with this many in flight.)
        float mc[2] = {-INFINITY, 0.0f};  // local max; NaN/Inf code
        float bad = 0.0f;  // becomes NaN if any element is NaN or +-Inf
        bool nan_seen = false;
        if (threadIdx.x < 8) {
            const int q = threadIdx.x < 4 ? s.head_q : s.tail_q;
            if (q >= 0) {
                const int idx = 4 * q + (threadIdx.x & 3);
                const int j = idx - s.pad;
                float v = -INFINITY;
                if (j >= 0 && j < s.len) {
                    v = src[j];
                    mc[0] = v;
                    bad = v * 0.0f;
                    nan_seen = isnan(v);
                }
                row[idx] = v;
            }
        }
        {
            const float* gb = src - s.pad;  // float4 q of the body is at gb + 4q
            int q = s.qb0 + threadIdx.x;
            for (; q + 7 * nt < s.qb1; q += 8 * nt) {
                float4 v[8];
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    v[i] = __ldcs(reinterpret_cast<const float4*>(gb + 4 * (q + i * nt)));
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    row4[q + i * nt] = v[i];
                    mc[0] = fmaxf(mc[0], fmaxf(fmaxf(v[i].x, v[i].y), fmaxf(v[i].z, v[i].w)));
                    bad = fmaf(v[i].x, 0.0f, bad);
                    bad = fmaf(v[i].y, 0.0f, bad);
                    bad = fmaf(v[i].z, 0.0f, bad);
                    bad = fmaf(v[i].w, 0.0f, bad);
                }
            }
            for (; q < s.qb1; q += nt) {
                const float4 v = __ldcs(reinterpret_cast<const float4*>(gb + 4 * q));
                row4[q] = v;
                mc[0] = fmaxf(mc[0], fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w)));
                bad = fmaf(v.x, 0.0f, bad);
                bad = fmaf(v.y, 0.0f, bad);
                bad = fmaf(v.z, 0.0f, bad);
                bad = fmaf(v.w, 0.0f, bad);
            }
        }
        // Classify a non-finite row (rare): 2 = NaN seen, 1 = only Inf.
        // Each thread rescans only the float4s it stored itself.
        if (bad != bad) {
            mc[1] = 1.0f;
            for (int q = s.qb0 + threadIdx.x; q < s.qb1; q += nt) {
                const float4 v = row4[q];
                if (isnan(v.x) || isnan(v.y) || isnan(v.z) || isnan(v.w))
                    nan_seen = true;
            }
            if (nan_seen) mc[1] = 2.0f;
        }
        exchange<CLUSTER, 2, true>(mc, sm, x);
        const float m = mc[0];
        const int row_code = static_cast<int>(mc[1]);

        float* dst = t.out + r * C + s0;
        unsigned int bits = 0;
        float T_row = NAN;
        float beta_out = 0.0f, inv_s = 0.0f;
        if (row_code == 0) {
            float s1[3];
            transform_pass(row4, s.q4, m, s1);
            exchange<CLUSTER, 3, false>(s1, sm, x);
            if (!entropy_above(make_float2(s1[0], s1[1]), 1.0f, cfg.bound_bits)) {
                T_row = 1.0f;
                beta_out = 1.0f;
                inv_s = 1.0f / s1[0];
            } else {
                Search st = search_begin(cfg, s1[0], s1[1], s1[2], t.strict != 0, false);
                if (!(cfg.t_min < cfg.hi0)) {
                    // No interval to halve: T = t_min (section 5.4 check).
                    st.final_round = true;
                    st.T_out = cfg.t_min;
                    const float T1[kMaxPoints] = {cfg.t_min, 0.f, 0.f};
                    const int J1[kMaxPoints] = {0, 0, 0};
                    search_round<CLUSTER, 1, false>(st, cfg, T1, J1, row4, s.q4, sm, x);
                }
                while (!st.done) {
                    float T[kMaxPoints];
                    int J[kMaxPoints];
                    const int np = search_plan(st, cfg, T, J);
                    const bool w0 = newton_next(st);
                    if (np == 1 && w0)
                        search_round<CLUSTER, 1, true>(st, cfg, T, J, row4, s.q4, sm, x);
                    else if (np == 1)
                        search_round<CLUSTER, 1, false>(st, cfg, T, J, row4, s.q4, sm, x);
                    else if (np == 2 && w0)
                        search_round<CLUSTER, 2, true>(st, cfg, T, J, row4, s.q4, sm, x);
                    else if (np == 2)
                        search_round<CLUSTER, 2, false>(st, cfg, T, J, row4, s.q4, sm, x);
                    else if (np == 3)
                        search_round<CLUSTER, 3, false>(st, cfg, T, J, row4, s.q4, sm, x);
                }
                if (st.overflow) bits |= kBitOverflow;
                T_row = st.T_out;
                beta_out = rcp_approx(st.T_out);
                inv_s = 1.0f / st.S_out;
            }
        } else {
            bits = row_code == 2 ? kBitNan : kBitInf;
        }
        write_out(row4, s, dst, beta_out, inv_s, row_code != 0);
        if (rank == 0 && threadIdx.x == 0) {
            if (t.t_out) t.t_out[r] = T_row;
            raise_error(t.err, bits);
        }
        if (x.dead && !reported) {
            raise_error(t.err, kBitTimeout);
            reported = true;
        }
        // The slice buffer is rewritten by the next row's loads.
        __syncthreads();
    }
    if (CLUSTER) cluster_sync();
}

template <bool CLUSTER, int MAXT, int MINB>
cudaError_t launch_one(const RowTask& task, int cluster_size, int slice_len,
                       int threads, int smem_bytes, int64_t grid_ctas,
                       cudaStream_t stream, int attr_slot) {
    auto kern = cluster_kernel<CLUSTER, MAXT, MINB>;
    cudaError_t e = ensure_smem_attribute(reinterpret_cast<const void*>(kern),
                                          attr_slot, smem_bytes);
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

}  // namespace

cudaError_t launch_cluster(const RowTask& task, int cluster_size,
                           int slice_len, int threads, int smem_bytes,
                           int64_t grid_ctas, cudaStream_t stream) {
    const bool narrow = threads <= 256;
    if (cluster_size > 1)
        return narrow ? launch_one<true, 256, 3>(task, cluster_size, slice_len,
                                                 threads, smem_bytes, grid_ctas,
                                                 stream, 1)
                      : launch_one<true, 512, 1>(task, cluster_size, slice_len,
                                                 threads, smem_bytes, grid_ctas,
                                                 stream, 3);
    return narrow ? launch_one<false, 256, 3>(task, 1, slice_len, threads,
                                              smem_bytes, grid_ctas, stream, 0)
                  : launch_one<false, 512, 1>(task, 1, slice_len, threads,
                                              smem_bytes, grid_ctas, stream, 2);
}

}  // namespace cs
