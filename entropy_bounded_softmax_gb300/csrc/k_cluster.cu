// Cluster kernel: one thread-block cluster of n CTAs per row (n = 1: one CTA
// per row).  Each CTA holds its slice of the row in shared memory for the
// whole search, so the row is read from HBM once and written once.
//
// Method: "BURT-IMMA CUDA Kernel API Reference", section 2.1
// `constrained_softmax`, Description steps 1-4, with the error policy of
// sections 5.3 and 5.4.  Per row:
//   stage   bulk copies (cp.async.bulk) of the slice into shared memory, in
//           chunks, each on its own mbarrier, so the max pass starts on the
//           first chunk while the rest are in flight;
//   max     m = max_i l_i (T-independent, computed once) and a finiteness
//           check, exchanged across the cluster;
//   T = 1   one pass turns the slice into y_i = (l_i - m) log2(e) in place
//           and sums S = sum 2^y_i and V = sum y_i 2^y_i;
//   search  each bisection step evaluates, at beta = 1/mid,
//           S(beta) = sum 2^(beta y_i) and V(beta) = sum y_i 2^(beta y_i);
//           with p_i = 2^(beta y_i) / S the entropy in nats is
//           H = ln 2 (log2 S - beta V / S), and H > bound is decided as
//           S (log2 S - bound log2 e) - beta V > 0;
//   output  p_i = 2^(beta_lo y_i) / S(lo), reusing S(lo) from the step that
//           set lo, written with 128-bit streaming stores.
//
// Slice mode.  Every warp scans its float4s of the slice.  The CTA reduces
// with one shuffle tree per warp, a __syncthreads, warp 0 summing the
// per-warp partials (and, in a cluster, pushing the CTA's sum to every CTA
// with st.async and waiting on an mbarrier for the others) and a second
// __syncthreads that broadcasts the result.  Every CTA sums in rank order,
// so all threads of the cluster see bit-identical sums and take the same
// decision.
//
// Active set.  Every later step evaluates at beta = 1/mid >= 1/hi, so a class
// with y_i < -K hi contributes less than 2^-K to S (which is >= 1: the
// maximum contributes 1) at every remaining step.  With K = 36 + log2(C)
// all such classes together change S and beta V by less than 2^-30 of
// their values, far below fp32 resolution.  After hi drops, a slice pass
// also compacts each warp's still-active classes (ballot + popc) into its
// own shared-memory segment.  If no warp anywhere in the cluster overflows
// its segment (and the active classes are few enough for one warp per
// CTA), the whole cluster switches in that same step to active-set mode:
// warp 0 of each CTA runs the rest of the search alone over the segments
// while the other warps wait for the output pass.  In that mode one
// exchange decides up to three bisection steps: the warp evaluates the 7
// midpoints of the next three levels (each computed exactly as the
// one-step-at-a-time search computes it) and walks them with the same
// decisions, so the result is that of the sequential search.  The full
// slice stays in place for the output pass, so every p_i is still computed.
//
// Every wait is bounded (cs::kWaitLimitCycles by default).  A thread whose
// wait times out records CS_ERR_TIMEOUT and from then on neither waits,
// pushes nor issues copies, but keeps the kernel's control flow so that all
// threads still meet at every __syncthreads and cluster barrier.
#include <math.h>

#include "cs_device.cuh"

namespace cs {
namespace {

using namespace csd;

constexpr int kSpecLevels = 3;   // bisection levels per active-set exchange
constexpr int kSlotFloats = 16;  // cluster slot payload (>= 2 * 7)
constexpr int kSearchWarpMax = 1024;  // active classes per CTA for one warp

__device__ __forceinline__ float4 floor4() {
    return make_float4(kYFloor, kYFloor, kYFloor, kYFloor);
}

// Geometry of one CTA's slice in shared memory.  Element j of the slice
// lives at row[pad + j], so 16-byte aligned global addresses land on
// 16-byte aligned shared addresses.  Float4 q in [qb0, qb1) comes in by
// bulk copy; the head (q = 0 when pad > 0) and tail float4s by plain loads.
struct Slice {
    int pad;
    int len;
    int q4;       // float4s of the slice in shared memory
    int qb0, qb1; // bulk-copied body
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

__device__ __forceinline__ int chunk_begin(const Slice& s, int nch, int c) {
    const int body = s.qb1 - s.qb0;
    return s.qb0 + static_cast<int>((static_cast<int64_t>(body) * c) / nch);
}

// Shared-memory objects of one CTA (cs::cluster_smem_bytes sizes them).
struct Smem {
    float* cslot;     // [2][n][kSlotFloats] cluster slots (double-buffered)
    float4* wslot;    // [warps] per-warp partials of slice-mode exchanges
    float4* bcast;    // [2] slice-mode result; active-set result
    int* segcnt;      // [warps] classes in each warp's active segment
    uint64_t* cbar;   // [2] cluster-exchange mbarriers
    uint64_t* lbar;   // [kLoadChunks] bulk-copy mbarriers
    float* wbuf;      // [warps][cap_w] active segments
    float4* row4;     // the slice
};

// Cluster-exchange state of one thread (only warp 0 exchanges).
struct Clu {
    int n;
    uint32_t rank;
    uint32_t xk;      // cluster exchanges so far (slot buffer and phase)
    uint64_t limit;
    bool dead;
};

// Shuffle-tree all-reduce of the first NV entries of a over the warp; every
// lane ends with the same (bit-identical) values.
template <int NV, bool IS_MAX, int N>
__device__ __forceinline__ void warp_reduce(float (&a)[N]) {
    static_assert(NV <= N, "size");
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            const float b = __shfl_xor_sync(0xffffffffu, a[i], o);
            a[i] = IS_MAX ? fmaxf(a[i], b) : a[i] + b;
        }
    }
}

// Called by warp 0 of every CTA of the cluster with the CTA's value of
// a[0..NV) (identical in all lanes); replaces it with the cluster-wide
// combination, formed in rank order and identical in every CTA.
template <int NV, bool IS_MAX, int N>
__device__ __forceinline__ void cluster_combine(float (&a)[N], const Smem& sm,
                                                Clu& c) {
    static_assert(NV % 2 == 0 && NV <= kSlotFloats && NV <= N, "payload");
    const int lane = threadIdx.x & 31;
    const uint32_t buf = c.xk & 1u;
    const uint32_t parity = (c.xk >> 1) & 1u;
    ++c.xk;
    float* cs = sm.cslot + buf * c.n * kSlotFloats;
    if (!c.dead) {
        if (lane == 0) mbar_arrive_expect_tx(&sm.cbar[buf], c.n * NV * 4);
        if (lane < c.n) {
            const uint32_t bar = map_to_rank(smem_addr(&sm.cbar[buf]), lane);
#pragma unroll
            for (int i = 0; i < NV; i += 2) {
                const uint32_t dst = map_to_rank(
                    smem_addr(&cs[c.rank * kSlotFloats + i]), lane);
                push_pair(dst, a[i], a[i + 1], bar);
            }
        }
        if (!mbar_wait<true>(&sm.cbar[buf], parity, c.limit)) c.dead = true;
    }
#pragma unroll
    for (int i = 0; i < NV; ++i)
        a[i] = lane < c.n ? cs[lane * kSlotFloats + i]
                          : (IS_MAX ? -INFINITY : 0.0f);
    warp_reduce<NV, IS_MAX>(a);
}

// Slice-mode exchange across all warps of the CTA (and the cluster): the
// first NV components of v are summed (or maxed) over every thread.
template <bool CLUSTER, int NV, bool IS_MAX>
__device__ __forceinline__ float4 slice_exchange(float4 v, const Smem& sm,
                                                 Clu& c) {
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int warps = blockDim.x >> 5;
    float a[4] = {v.x, v.y, v.z, v.w};
    warp_reduce<NV, IS_MAX>(a);
    if (lane == 0) sm.wslot[warp] = make_float4(a[0], a[1], a[2], a[3]);
    __syncthreads();
    if (warp == 0) {
        const float idn = IS_MAX ? -INFINITY : 0.0f;
        const float4 w = lane < warps ? sm.wslot[lane]
                                      : make_float4(idn, idn, idn, idn);
        a[0] = w.x;
        a[1] = w.y;
        a[2] = w.z;
        a[3] = w.w;
        warp_reduce<NV, IS_MAX>(a);
        if (CLUSTER) cluster_combine<NV, IS_MAX>(a, sm, c);
        if (lane == 0) sm.bcast[0] = make_float4(a[0], a[1], a[2], a[3]);
    }
    __syncthreads();
    return sm.bcast[0];
}

// T = 1 pass: rewrites this thread's float4s of the slice as
// y = max((l - m) log2 e, floor) and returns the partial (S, V) at beta = 1.
__device__ __forceinline__ float2 transform_pass(float4* row4, int q4,
                                                 float m) {
    SV4 acc;
    acc.zero();
    const float2 one = make_float2(1.0f, 1.0f);
    for (int q = threadIdx.x; q < q4; q += blockDim.x) {
        float4 y = row4[q];
        y.x = fmaxf((y.x - m) * kLog2e, kYFloor);
        y.y = fmaxf((y.y - m) * kLog2e, kYFloor);
        y.z = fmaxf((y.z - m) * kLog2e, kYFloor);
        y.w = fmaxf((y.w - m) * kLog2e, kYFloor);
        row4[q] = y;
        acc.add(y, one);
    }
    return acc.total();
}

// Full pass over this thread's float4s of the slice at inverse temperature
// beta.  Thread t owns float4s t, t + nt, ...; the loop runs a warp-uniform
// number of times (two float4s per trip) so that GATHER can use warp votes.
// GATHER: also appends every class with y >= thr to the warp's segment wb
// (capacity cap); *cnt returns the warp's count, > cap on overflow.
template <bool GATHER>
__device__ __forceinline__ float2 slice_pass(const float4* row4, int q4,
                                             float beta, float thr, float* wb,
                                             int cap, int* cnt) {
    SV4 acc;
    acc.zero();
    const float2 b2 = make_float2(beta, beta);
    const int nt = blockDim.x;
    const int lane = threadIdx.x & 31;
    const int warp_base = threadIdx.x & ~31;
    const unsigned lt = (1u << lane) - 1u;
    int cw = 0;
    for (int qb = warp_base; qb < q4; qb += 2 * nt) {
        const int qa = qb + lane;
        const int qc = qa + nt;
        const float4 ya = qa < q4 ? row4[qa] : floor4();
        const float4 yc = qc < q4 ? row4[qc] : floor4();
        acc.add(ya, b2);
        acc.add(yc, b2);
        if (GATHER && cw <= cap) {
            const float v[8] = {ya.x, ya.y, ya.z, ya.w, yc.x, yc.y, yc.z, yc.w};
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const bool a = v[k] >= thr;
                const unsigned msk = __ballot_sync(0xffffffffu, a);
                const int pos = cw + __popc(msk & lt);
                if (a && pos < cap) wb[pos] = v[k];
                cw += __popc(msk);
            }
        }
    }
    if (GATHER) *cnt = cw;
    return acc.total();
}

// Midpoint of the search, in the fp32 arithmetic every variant uses.
__device__ __forceinline__ float midpoint(float lo, float hi) {
    return 0.5f * (lo + hi);
}

// Search state (identical in every thread that runs the search).
struct Search {
    float lo, hi, s_lo;
    bool lo_eval, hi_eval;
    int k;            // bisection steps taken
};

// Applies one evaluated step at `mid` with the cluster sums (S, V) at beta;
// returns true if mid was infeasible (hi moved).
__device__ __forceinline__ bool apply_step(Search& st, float mid, float beta,
                                           float S, float V,
                                           float bound_bits) {
    ++st.k;
    if (entropy_above(make_float2(S, V), beta, bound_bits)) {
        st.hi = mid;
        st.hi_eval = true;
        return true;
    }
    st.lo = mid;
    st.lo_eval = true;
    st.s_lo = S;
    return false;
}

// True when no step remains: max_iter steps taken, or the next fp32
// midpoint equals an end already evaluated (every further step would
// repeat that evaluation and change nothing).
__device__ __forceinline__ bool search_finished(const Search& st,
                                                int max_iter) {
    if (st.k >= max_iter) return true;
    const float mid = midpoint(st.lo, st.hi);
    return (mid == st.lo && st.lo_eval) || (mid == st.hi && st.hi_eval);
}

// Active-set mode, run by warp 0 alone: evaluates the P = 2^D - 1
// midpoints of the next D levels in one pass over the CTA's segments,
// combines them across the cluster, then walks them with the sequential
// search's decisions.
template <bool CLUSTER, int D>
__device__ __forceinline__ void active_step(Search& st, const Smem& sm,
                                            int warps, int cap_w,
                                            float bound_bits, int max_iter,
                                            Clu& c) {
    constexpr int P = (1 << D) - 1;
    const int lane = threadIdx.x & 31;
    // Heap of midpoints: node i (0-based) has children 2i+1 (the lower half,
    // taken when mid_i is infeasible) and 2i+2 (the upper half).
    float mids[P], los[P], his[P], beta[P];
    los[0] = st.lo;
    his[0] = st.hi;
#pragma unroll
    for (int i = 0; i < P; ++i) {
        mids[i] = midpoint(los[i], his[i]);
        beta[i] = __frcp_rn(mids[i]);
        if (2 * i + 2 < P) {
            los[2 * i + 1] = los[i];
            his[2 * i + 1] = mids[i];
            los[2 * i + 2] = mids[i];
            his[2 * i + 2] = his[i];
        }
    }
    float a[2 * P];
#pragma unroll
    for (int i = 0; i < 2 * P; ++i) a[i] = 0.0f;
    for (int w = 0; w < warps; ++w) {
        const float* seg = sm.wbuf + w * cap_w;
        const int cnt = sm.segcnt[w];
        for (int j = lane; j < cnt; j += 32) {
            const float y = seg[j];
#pragma unroll
            for (int i = 0; i < P; ++i) {
                const float e = ex2(y * beta[i]);
                a[2 * i] += e;
                a[2 * i + 1] = fmaf(e, y, a[2 * i + 1]);
            }
        }
    }
    warp_reduce<2 * P, false>(a);
    if (CLUSTER) cluster_combine<2 * P, false>(a, sm, c);
    int node = 0;
#pragma unroll
    for (int d = 0; d < D; ++d) {
        if (search_finished(st, max_iter)) break;
        // Select node's values with compares (no dynamic register indexing).
        float m = mids[0], b = beta[0], S = a[0], V = a[1];
#pragma unroll
        for (int i = 1; i < P; ++i) {
            if (i == node) {
                m = mids[i];
                b = beta[i];
                S = a[2 * i];
                V = a[2 * i + 1];
            }
        }
        const bool infeasible = apply_step(st, m, b, S, V, bound_bits);
        node = infeasible ? 2 * node + 1 : 2 * node + 2;
    }
}

// Drops the classes below thr from every segment, in place (warp 0).
__device__ __forceinline__ void refilter_segments(const Smem& sm, int warps,
                                                  int cap_w, float thr) {
    const int lane = threadIdx.x & 31;
    const unsigned lt = (1u << lane) - 1u;
    for (int w = 0; w < warps; ++w) {
        float* seg = sm.wbuf + w * cap_w;
        const int cnt = sm.segcnt[w];
        int nc = 0;
        for (int j0 = 0; j0 < cnt; j0 += 32) {
            const int j = j0 + lane;
            const float y = j < cnt ? seg[j] : kYFloor;
            const bool keep = j < cnt && y >= thr;
            const unsigned msk = __ballot_sync(0xffffffffu, keep);
            __syncwarp();  // every lane has read its entry of this round
            if (keep) seg[nc + __popc(msk & lt)] = y;
            nc += __popc(msk);
        }
        __syncwarp();
        if (lane == 0) sm.segcnt[w] = nc;
        __syncwarp();
    }
}

// S and V at beta over the active segments (warp 0), cluster-wide.
template <bool CLUSTER>
__device__ __forceinline__ float2 active_eval(const Smem& sm, int warps,
                                              int cap_w, float beta, Clu& c) {
    const int lane = threadIdx.x & 31;
    float a[2] = {0.0f, 0.0f};
    for (int w = 0; w < warps; ++w) {
        const float* seg = sm.wbuf + w * cap_w;
        const int cnt = sm.segcnt[w];
        for (int j = lane; j < cnt; j += 32) {
            const float e = ex2(seg[j] * beta);
            a[0] += e;
            a[1] = fmaf(e, seg[j], a[1]);
        }
    }
    warp_reduce<2, false>(a);
    if (CLUSTER) cluster_combine<2, false>(a, sm, c);
    return make_float2(a[0], a[1]);
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
    for (int q = threadIdx.x; q < s.q4; q += blockDim.x) {
        float4 p = make_float4(0.f, 0.f, 0.f, 0.f);
        if (!zero) {
            const float4 y = row4[q];
            const float2 x01 = mul2(make_float2(y.x, y.y), b2);
            const float2 x23 = mul2(make_float2(y.z, y.w), b2);
            const float2 p01 = mul2(make_float2(ex2(x01.x), ex2(x01.y)), i2);
            const float2 p23 = mul2(make_float2(ex2(x23.x), ex2(x23.y)), i2);
            p = make_float4(p01.x, p01.y, p23.x, p23.y);
        }
        if (vec && q >= s.qb0 && q < s.qb1) {
            __stcs(reinterpret_cast<float4*>(dst + (4 * q - s.pad)), p);
        } else {
            store_scalar_lanes(dst, q, s.pad, s.len, p);
        }
    }
}

template <bool CLUSTER>
__global__ void __launch_bounds__(kClusterMaxThreads, 1)
cluster_kernel(RowTask t, int n, int slice_len, int cap_w) {
    extern __shared__ __align__(128) unsigned char smem[];
    const int nt = blockDim.x;
    const int warps = nt >> 5;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = CLUSTER ? cluster_ctarank() : 0u;
    const int64_t cid = blockIdx.x / n;
    const int64_t ncl = gridDim.x / n;

    Smem sm;
    {
        const ClusterSmemLayout L = cluster_smem_layout(warps, n, cap_w);
        sm.cslot = reinterpret_cast<float*>(smem + L.cslot);
        sm.wslot = reinterpret_cast<float4*>(smem + L.wslot);
        sm.bcast = reinterpret_cast<float4*>(smem + L.bcast);
        sm.segcnt = reinterpret_cast<int*>(smem + L.segcnt);
        sm.cbar = reinterpret_cast<uint64_t*>(smem + L.cbar);
        sm.lbar = reinterpret_cast<uint64_t*>(smem + L.lbar);
        sm.wbuf = reinterpret_cast<float*>(smem + L.wbuf);
        sm.row4 = reinterpret_cast<float4*>(smem + L.row);
    }
    float* row = reinterpret_cast<float*>(sm.row4);
    float4* row4 = sm.row4;

    if (threadIdx.x == 0) {
        mbar_init(&sm.cbar[0], 1u);
        mbar_init(&sm.cbar[1], 1u);
        for (int c = 0; c < kLoadChunks; ++c) mbar_init(&sm.lbar[c], 1u);
        fence_mbar_init();
    }
    __syncthreads();
    if (CLUSTER) cluster_sync();

    const int64_t C = t.num_classes;
    const int64_t s0 = static_cast<int64_t>(rank) * slice_len;
    const int len = static_cast<int>(max(static_cast<int64_t>(0),
                                         min(static_cast<int64_t>(slice_len), C - s0)));
    const float bound_bits = t.entropy_bound * kLog2e;
    const bool prune = cap_w > 0 && t.prune_k > 0.0f;
    Clu clu{n, rank, 0u, t.wait_limit_cycles, false};
    uint32_t lphase = 0;       // parity bit per load chunk
    bool reported = false;

    for (int64_t r = cid; r < t.batch; r += ncl) {
        const float* src = t.logits + r * C + s0;
        const Slice s = make_slice(src, len);
        const int body = s.qb1 - s.qb0;
        const int nch = body > 0 ? min(kLoadChunks, body) : 0;

        // Stage: thread 0 issues the bulk copies; threads 0-7 fetch the
        // ragged head/tail float4s with plain loads.
        if (threadIdx.x == 0 && !clu.dead) {
            fence_proxy_async_smem();
            for (int c = 0; c < nch; ++c) {
                const int qa = chunk_begin(s, nch, c);
                const int qz = chunk_begin(s, nch, c + 1);
                const uint32_t bytes = static_cast<uint32_t>(qz - qa) * 16u;
                mbar_arrive_expect_tx(&sm.lbar[c], bytes);
                bulk_load(row4 + qa, src + (4 * qa - s.pad), bytes, &sm.lbar[c]);
            }
        }
        float m_loc = -INFINITY;
        float bad = 0.0f;  // becomes NaN if any element is NaN or +-Inf
        if (threadIdx.x < 8) {
            const int q = threadIdx.x < 4 ? s.head_q : s.tail_q;
            if (q >= 0) {
                const int idx = 4 * q + (threadIdx.x & 3);
                const int j = idx - s.pad;
                float v = -INFINITY;
                if (j >= 0 && j < s.len) {
                    v = src[j];
                    m_loc = v;
                    bad = v * 0.0f;
                }
                row[idx] = v;
            }
        }
        __syncthreads();

        // Max pass, chunk by chunk as the copies land.
        for (int c = 0; c < nch; ++c) {
            if (!clu.dead &&
                !mbar_wait<false>(&sm.lbar[c], (lphase >> c) & 1u, clu.limit))
                clu.dead = true;
            lphase ^= 1u << c;
            const int qa = chunk_begin(s, nch, c);
            const int qz = chunk_begin(s, nch, c + 1);
            for (int q = qa + threadIdx.x; q < qz; q += nt) {
                const float4 v = row4[q];
                m_loc = fmaxf(m_loc, fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w)));
                bad = fmaf(v.x, 0.0f, bad);
                bad = fmaf(v.y, 0.0f, bad);
                bad = fmaf(v.z, 0.0f, bad);
                bad = fmaf(v.w, 0.0f, bad);
            }
        }
        // Classify a non-finite row (rare): 2 = NaN seen, 1 = only Inf.
        float code = 0.0f;
        if (bad != bad) {
            code = 1.0f;
            for (int q = threadIdx.x; q < s.q4; q += nt) {
                const float4 v = row4[q];
                const int j0 = 4 * q - s.pad;
                const float e[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int j = j0 + i;
                    if (j >= 0 && j < s.len && isnan(e[i])) code = 2.0f;
                }
            }
        }
        const float4 mc = slice_exchange<CLUSTER, 2, true>(
            make_float4(m_loc, code, 0.f, 0.f), sm, clu);
        const float m = mc.x;
        const int row_code = static_cast<int>(mc.y);

        float* dst = t.out + r * C + s0;
        unsigned int bits = 0;
        float T_row = NAN;
        float beta_out = 0.0f, inv_s = 0.0f;
        if (row_code == 0) {
            const float2 p1 = transform_pass(row4, s.q4, m);
            const float4 sv = slice_exchange<CLUSTER, 2, false>(
                make_float4(p1.x, p1.y, 0.f, 0.f), sm, clu);
            if (!entropy_above(make_float2(sv.x, sv.y), 1.0f, bound_bits)) {
                T_row = 1.0f;
                beta_out = 1.0f;
                inv_s = 1.0f / sv.x;
            } else {
                Search st{t.t_min, t.hi0, 0.0f, false, t.hi0 == 1.0f, 0};
                bool gather = false;   // gather active classes in this step
                bool active = false;   // switched to active-set mode
                if (st.lo < st.hi) {
                    // Slice mode: every warp, one step per exchange.
                    while (!search_finished(st, t.max_iter)) {
                        const float mid = midpoint(st.lo, st.hi);
                        const float b = __frcp_rn(mid);
                        float4 sv4;
                        if (gather) {
                            int cw = 0;
                            const float2 pp = slice_pass<true>(
                                row4, s.q4, b, -t.prune_k * st.hi,
                                sm.wbuf + warp * cap_w, cap_w, &cw);
                            if (lane == 0) sm.segcnt[warp] = cw;
                            // z: warps that overflowed; w: classes gathered.
                            sv4 = slice_exchange<CLUSTER, 4, false>(
                                make_float4(pp.x, pp.y,
                                            lane == 0 && cw > cap_w ? 1.f : 0.f,
                                            lane == 0 ? static_cast<float>(cw) : 0.f),
                                sm, clu);
                        } else {
                            const float2 pp = slice_pass<false>(
                                row4, s.q4, b, 0.0f, nullptr, 0, nullptr);
                            sv4 = slice_exchange<CLUSTER, 2, false>(
                                make_float4(pp.x, pp.y, 0.f, 0.f), sm, clu);
                        }
                        const bool hi_moved =
                            apply_step(st, mid, b, sv4.x, sv4.y, bound_bits);
                        if (gather) {
                            gather = false;
                            if (sv4.z == 0.0f &&
                                sv4.w <= static_cast<float>(kSearchWarpMax * n)) {
                                active = true;
                                break;
                            }
                        }
                        if (prune && hi_moved) gather = true;
                    }
                }
                if (active) {
                    // Active-set mode: warp 0 of each CTA finishes alone.
                    if (warp == 0) {
                        float filtered_hi = st.hi;
                        refilter_segments(sm, warps, cap_w, -t.prune_k * st.hi);
                        while (!search_finished(st, t.max_iter)) {
                            if (st.hi < filtered_hi) {
                                refilter_segments(sm, warps, cap_w,
                                                  -t.prune_k * st.hi);
                                filtered_hi = st.hi;
                            }
                            const int left = t.max_iter - st.k;
                            if (left >= kSpecLevels)
                                active_step<CLUSTER, kSpecLevels>(
                                    st, sm, warps, cap_w, bound_bits,
                                    t.max_iter, clu);
                            else if (left == 2)
                                active_step<CLUSTER, 2>(st, sm, warps, cap_w,
                                                        bound_bits, t.max_iter,
                                                        clu);
                            else
                                active_step<CLUSTER, 1>(st, sm, warps, cap_w,
                                                        bound_bits, t.max_iter,
                                                        clu);
                        }
                        if (!st.lo_eval) {
                            // lo is still t_min: evaluate it (section 5.4).
                            const float b_lo = __frcp_rn(st.lo);
                            const float2 e = active_eval<CLUSTER>(
                                sm, warps, cap_w, b_lo, clu);
                            st.s_lo = e.x;
                            if (entropy_above(e, b_lo, bound_bits))
                                bits |= kBitOverflow;
                        }
                        if (lane == 0)
                            sm.bcast[1] = make_float4(st.lo, st.s_lo,
                                                      __uint_as_float(bits), 0.f);
                    }
                    __syncthreads();
                    const float4 res = sm.bcast[1];
                    st.lo = res.x;
                    st.s_lo = res.y;
                    bits = __float_as_uint(res.z);
                } else if (!st.lo_eval) {
                    // lo is still t_min: evaluate it (section 5.4).
                    const float b_lo = __frcp_rn(st.lo);
                    const float2 pp = slice_pass<false>(row4, s.q4, b_lo, 0.0f,
                                                        nullptr, 0, nullptr);
                    const float4 sv4 = slice_exchange<CLUSTER, 2, false>(
                        make_float4(pp.x, pp.y, 0.f, 0.f), sm, clu);
                    st.s_lo = sv4.x;
                    if (entropy_above(make_float2(sv4.x, sv4.y), b_lo,
                                      bound_bits))
                        bits |= kBitOverflow;
                }
                T_row = st.lo;
                beta_out = __frcp_rn(st.lo);
                inv_s = 1.0f / st.s_lo;
            }
        } else {
            bits = row_code == 2 ? kBitNan : kBitInf;
        }
        write_out(row4, s, dst, beta_out, inv_s, row_code != 0);
        if (rank == 0 && threadIdx.x == 0) {
            if (t.t_out) t.t_out[r] = T_row;
            raise_error(t.err, bits);
        }
        if (clu.dead && !reported) {
            raise_error(t.err, kBitTimeout);
            reported = true;
        }
        // The slice buffer is rewritten by the next row's copies.
        __syncthreads();
    }
    if (clu.dead && threadIdx.x == 0) {
        // Give copies still in flight a bounded chance to land before exit.
        for (int c = 0; c < kLoadChunks; ++c)
            mbar_wait<false>(&sm.lbar[c], ((lphase >> c) & 1u) ^ 1u,
                             t.wait_limit_cycles);
    }
    if (CLUSTER) cluster_sync();
}

}  // namespace

cudaError_t launch_cluster(const RowTask& task, int cluster_size,
                           int slice_len, int threads, int cap_w,
                           int smem_bytes, int64_t grid_ctas,
                           cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid_ctas), 1, 1);
    cfg.blockDim = dim3(static_cast<unsigned>(threads), 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem_bytes);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    if (cluster_size > 1) {
        auto kern = cluster_kernel<true>;
        cudaError_t e = ensure_smem_attribute(
            reinterpret_cast<const void*>(kern), 1, smem_bytes);
        if (e != cudaSuccess) return e;
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = static_cast<unsigned>(cluster_size);
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        return cudaLaunchKernelEx(&cfg, kern, task, cluster_size, slice_len,
                                  cap_w);
    }
    auto kern = cluster_kernel<false>;
    cudaError_t e = ensure_smem_attribute(reinterpret_cast<const void*>(kern),
                                          0, smem_bytes);
    if (e != cudaSuccess) return e;
    cfg.attrs = nullptr;
    cfg.numAttrs = 0;
    return cudaLaunchKernelEx(&cfg, kern, task, 1, slice_len, cap_w);
}

}  // namespace cs
