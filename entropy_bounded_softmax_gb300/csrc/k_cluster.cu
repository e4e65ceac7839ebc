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
// Reduction.  Every warp reduces its (S, V) with a shuffle tree and writes
// the pair to a slot; after one __syncthreads every warp reduces the slots
// with a second shuffle tree.  In a cluster, warp 0 then pushes the CTA's
// pair into every CTA (st.async, counted on an mbarrier) and every thread
// sums the cluster's pairs in rank order once the mbarrier completes.  All
// threads of the cluster thus see bit-identical sums and take the same
// decision.  Slots are double-buffered, which is safe because no thread can
// reach exchange k+2 before every thread has left exchange k.
//
// Active set.  Every later step evaluates at beta = 1/mid >= 1/hi, so a class
// with y_i < -K hi contributes less than 2^-K to S (which is >= 1: the
// maximum contributes 1) at every remaining step.  With K = 36 + log2(C)
// all such classes together change S and beta V by less than 2^-30 of
// their values, far below fp32 resolution.  After hi drops, a warp still
// scanning the slice compacts its active classes (ballot + popc) into its
// own shared-memory segment during the next pass; if they fit, later steps
// read only the segment (and drop classes again whenever hi drops).  The
// full slice stays in place for the output pass, so every p_i is still
// computed.

// Every wait is bounded (cs::kWaitLimitCycles by default).  A thread whose
// wait times out records CS_ERR_TIMEOUT and from then on neither waits,
// pushes nor issues copies, but keeps the kernel's control flow so that all
// threads still meet at every __syncthreads and cluster barrier.
#include <math.h>

#include "cs_device.cuh"

namespace cs {
namespace {

using namespace csd;

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

// Shared-memory objects of one CTA (cs::cluster_smem_layout places them).
struct Smem {
    float2* cslot;    // [2][n] cluster slots (double-buffered)
    float2* wslot;    // [2][warps] per-warp slots (double-buffered)
    uint64_t* cbar;   // [2] cluster-exchange mbarriers
    uint64_t* lbar;   // [kLoadChunks] bulk-copy mbarriers
    float* wbuf;      // [warps][cap_w] active segments
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

__device__ __forceinline__ float2 combine2(float2 a, float2 b, bool is_max) {
    return is_max ? make_float2(fmaxf(a.x, b.x), fmaxf(a.y, b.y))
                  : make_float2(a.x + b.x, a.y + b.y);
}

// Sum (or max) of every thread's v over the CTA and the cluster; returns
// the same bits in every thread of the cluster.
template <bool CLUSTER, bool IS_MAX>
__device__ __forceinline__ float2 exchange(float2 v, const Smem& sm,
                                           Exch& x) {
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    v = IS_MAX ? warp_max2(v) : warp_sum2(v);
    float2* ws = sm.wslot + (x.lk & 1u) * x.warps;
    ++x.lk;
    if (lane == 0) ws[warp] = v;
    __syncthreads();
    const float idn = IS_MAX ? -INFINITY : 0.0f;
    v = lane < x.warps ? ws[lane] : make_float2(idn, idn);
    v = IS_MAX ? warp_max2(v) : warp_sum2(v);
    if (CLUSTER) {
        const uint32_t buf = x.xk & 1u;
        const uint32_t parity = (x.xk >> 1) & 1u;
        ++x.xk;
        float2* cs = sm.cslot + buf * x.n;
        if (!x.dead) {
            if (threadIdx.x == 0) mbar_arrive_expect_tx(&sm.cbar[buf], x.n * 8);
            if (warp == 0 && lane < x.n) {
                const uint32_t dst = map_to_rank(smem_addr(&cs[x.rank]), lane);
                const uint32_t bar = map_to_rank(smem_addr(&sm.cbar[buf]), lane);
                push_pair(dst, v.x, v.y, bar);
            }
            if (!mbar_wait<true>(&sm.cbar[buf], parity, x.limit)) x.dead = true;
        }
        v = cs[0];
        for (int r = 1; r < x.n; ++r) v = combine2(v, cs[r], IS_MAX);
    }
    return v;
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
    if (GATHER) {
        *cnt = cw;
        __syncwarp();
    }
    return acc.total();
}

// Pass over the warp's active segment.  RECOMPACT: also drops the classes
// below thr, compacting the segment in place (entries only move to lower
// positions, and every lane reads its entry of a round before any lane
// writes).
template <bool RECOMPACT>
__device__ __forceinline__ float2 segment_pass(float* wb, int* cnt, float beta,
                                               float thr) {
    const int lane = threadIdx.x & 31;
    const unsigned lt = (1u << lane) - 1u;
    const int c = *cnt;
    float s = 0.0f, v = 0.0f;
    int nc = 0;
    for (int j0 = 0; j0 < c; j0 += 32) {
        const int j = j0 + lane;
        const float y = j < c ? wb[j] : kYFloor;
        const float e = ex2(y * beta);
        s += e;
        v = fmaf(e, y, v);
        if (RECOMPACT) {
            const bool a = j < c && y >= thr;
            const unsigned msk = __ballot_sync(0xffffffffu, a);
            __syncwarp();
            if (a) wb[nc + __popc(msk & lt)] = y;
            nc += __popc(msk);
        }
    }
    if (RECOMPACT) {
        *cnt = nc;
        __syncwarp();
    }
    return make_float2(s, v);
}

// What the next pass of this warp reads (uniform within the warp).
struct ActiveSet {
    float* wb;          // this warp's segment
    int cap;            // its capacity (0: active set off)
    int cnt;            // classes in the segment
    bool in_segment;    // the warp reads its segment instead of the slice
    bool refilter;      // hi dropped: gather (slice) or recompact (segment)
    float thr;          // y >= thr is active (thr = -K hi)
};

__device__ __forceinline__ float2 search_partial(const float4* row4, int q4,
                                                 float beta, ActiveSet& a) {
    if (a.in_segment) {
        if (a.refilter) {
            a.refilter = false;
            return segment_pass<true>(a.wb, &a.cnt, beta, a.thr);
        }
        return segment_pass<false>(a.wb, &a.cnt, beta, a.thr);
    }
    if (a.refilter) {
        a.refilter = false;
        int c = 0;
        const float2 part = slice_pass<true>(row4, q4, beta, a.thr, a.wb,
                                             a.cap, &c);
        if (c <= a.cap) {
            a.in_segment = true;
            a.cnt = c;
        }
        return part;
    }
    return slice_pass<false>(row4, q4, beta, 0.0f, nullptr, 0, nullptr);
}

// Midpoint of the search, in the fp32 arithmetic every variant uses.
__device__ __forceinline__ float midpoint(float lo, float hi) {
    return 0.5f * (lo + hi);
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
    const uint32_t rank = CLUSTER ? cluster_ctarank() : 0u;
    const int64_t cid = blockIdx.x / n;
    const int64_t ncl = gridDim.x / n;

    Smem sm;
    {
        const ClusterSmemLayout L = cluster_smem_layout(warps, n, cap_w);
        sm.cslot = reinterpret_cast<float2*>(smem + L.cslot);
        sm.wslot = reinterpret_cast<float2*>(smem + L.wslot);
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
    Exch x{warps, n, rank, 0u, 0u, t.wait_limit_cycles, false};
    uint32_t lphase = 0;       // parity bit per load chunk
    bool reported = false;

    for (int64_t r = cid; r < t.batch; r += ncl) {
        const float* src = t.logits + r * C + s0;
        const Slice s = make_slice(src, len);
        const int body = s.qb1 - s.qb0;
        const int nch = body > 0 ? min(kLoadChunks, body) : 0;

        // Stage: thread 0 issues the bulk copies; threads 0-7 fetch the
        // ragged head/tail float4s with plain loads.
        if (threadIdx.x == 0 && !x.dead) {
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
            if (!x.dead &&
                !mbar_wait<false>(&sm.lbar[c], (lphase >> c) & 1u, x.limit))
                x.dead = true;
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
        const float2 mc = exchange<CLUSTER, true>(make_float2(m_loc, code), sm, x);
        const float m = mc.x;
        const int row_code = static_cast<int>(mc.y);

        float* dst = t.out + r * C + s0;
        unsigned int bits = 0;
        float T_row = NAN;
        float beta_out = 0.0f, inv_s = 0.0f;
        if (row_code == 0) {
            float2 sv = exchange<CLUSTER, false>(transform_pass(row4, s.q4, m),
                                                 sm, x);
            if (!entropy_above(sv, 1.0f, bound_bits)) {
                T_row = 1.0f;
                beta_out = 1.0f;
                inv_s = 1.0f / sv.x;
            } else {
                ActiveSet a{sm.wbuf + warp * cap_w, prune ? cap_w : 0, 0,
                            false, false, 0.0f};
                float lo = t.t_min, hi = t.hi0;
                bool lo_eval = false;
                bool hi_eval = hi == 1.0f;   // H(1) > bound is known
                float s_lo = 0.0f;
                if (lo < hi) {
                    for (int k = 0; k < t.max_iter; ++k) {
                        const float mid = midpoint(lo, hi);
                        // Exact early exit: the fp32 midpoint has reached an
                        // end whose side is already known, so every further
                        // step repeats the same evaluation.
                        if ((mid == lo && lo_eval) || (mid == hi && hi_eval)) break;
                        const float b = rcp_approx(mid);
                        sv = exchange<CLUSTER, false>(
                            search_partial(row4, s.q4, b, a), sm, x);
                        if (entropy_above(sv, b, bound_bits)) {
                            hi = mid;
                            hi_eval = true;
                            if (a.cap > 0) {
                                a.thr = -t.prune_k * hi;
                                a.refilter = true;
                            }
                        } else {
                            lo = mid;
                            lo_eval = true;
                            s_lo = sv.x;
                        }
                    }
                }
                const float b_lo = rcp_approx(lo);
                if (!lo_eval) {
                    // lo is still t_min: evaluate it (section 5.4 check).
                    sv = exchange<CLUSTER, false>(
                        search_partial(row4, s.q4, b_lo, a), sm, x);
                    s_lo = sv.x;
                    if (entropy_above(sv, b_lo, bound_bits)) bits |= kBitOverflow;
                }
                T_row = lo;
                beta_out = b_lo;
                inv_s = 1.0f / s_lo;
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
        // The slice buffer is rewritten by the next row's copies.
        __syncthreads();
    }
    if (x.dead && threadIdx.x == 0) {
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
