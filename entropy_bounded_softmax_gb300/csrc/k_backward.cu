// Backward kernels of the constrained softmax.  For every row,
//
//     grad_l = (1/T) p (g - <g, p>),
//
// with p the forward's output, g the upstream gradient and T the row's
// temperature ("BURT-IMMA CUDA Kernel API Reference", section 6.3,
// ConstrainedSoftmaxFunction.backward: the softmax Jacobian-vector product,
// to which the 1/T of softmax(l / T) is restored; T is a grid point chosen
// by comparisons, piecewise constant in l, so it adds no term of its own).
// A row whose T is not a positive finite number (NaN marks a row the
// forward zeroed) gets zeros.
//
// Each class is read twice (p, g) and written once: 12 bytes, one pass over
// HBM, no tensor-core work.  The only cross-thread step is the row's dot
// product <g, p>, so both kernels load the row, reduce, and then write it
// from where they staged it:
//   row-group  G lanes of a warp share a short row and keep it in
//              registers; the dot product is a G-lane shuffle sum;
//   cluster    n CTAs share a long row (n = 1: one CTA); each stages its
//              slice of p (and of g when both fit) in shared memory,
//              reduces its partial dot product over warps, and the CTAs
//              exchange them over distributed shared memory.
//
// Element j of a row segment sits at lane (j + pad) % 4 of float4
// (j + pad) / 4, pad being p's alignment (in floats) at the segment start.
// A float4 that is whole and whose tensor shares that alignment moves with
// one 128-bit access; the rest (ragged ends, a tensor with another
// alignment) element by element.
#include <math.h>

#include "cs_device.cuh"

namespace cs {
namespace {

using namespace csd;

__device__ __forceinline__ int pad_of(const void* a) {
    return static_cast<int>((reinterpret_cast<uintptr_t>(a) >> 2) & 3);
}

// Float4 q of the segment a[0, len) (a's own pad pa) in the layout of pad
// `pad`; elements outside [0, len) read as 0.  STREAM: evict-first loads
// (data read once); otherwise default caching (g read again later).
template <bool STREAM>
__device__ __forceinline__ float4 load4(const float* a, int pa, int pad,
                                        int len, int q) {
    const int j0 = 4 * q - pad;
    if (pa == pad && j0 >= 0 && j0 + 4 <= len) {
        const float4* v = reinterpret_cast<const float4*>(a + j0);
        return STREAM ? __ldcs(v) : *v;
    }
    float e[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int j = j0 + i;
        e[i] = 0.0f;
        if (j >= 0 && j < len) e[i] = a[j];
    }
    return make_float4(e[0], e[1], e[2], e[3]);
}

// Stores float4 q of the layout into a[0, len) (a's own pad pa).
__device__ __forceinline__ void store4(float* a, int pa, int pad, int len,
                                       int q, float4 v) {
    const int j0 = 4 * q - pad;
    if (pa == pad && j0 >= 0 && j0 + 4 <= len) {
        __stcs(reinterpret_cast<float4*>(a + j0), v);
        return;
    }
    const float e[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int j = j0 + i;
        if (j >= 0 && j < len) a[j] = e[i];
    }
}

// Stages float4 q of the layout (pad) of segment a (own pad pa) into
// shared memory at dst: one asynchronous 16-byte copy when whole and
// aligned, else element by element (zeros outside [0, len)).
__device__ __forceinline__ void stage4(float4* dst, const float* a, int pa,
                                       int pad, int len, int q) {
    const int j0 = 4 * q - pad;
    if (pa == pad && j0 >= 0 && j0 + 4 <= len) {
        cp_async16(dst, a + j0);
        return;
    }
    *dst = load4<true>(a, pa, pad, len, q);
}

// acc += p * g, lanes (x, y) and (z, w) in two packed pairs.
__device__ __forceinline__ void dot_add(float2& a, float2& b, float4 p,
                                        float4 g) {
    a = fma2(make_float2(p.x, p.y), make_float2(g.x, g.y), a);
    b = fma2(make_float2(p.z, p.w), make_float2(g.z, g.w), b);
}

// (p / T) (g - dot), or zeros for a row without a valid temperature.
__device__ __forceinline__ float4 grad4(float4 p, float4 g, float dot,
                                        float inv_t, bool ok) {
    if (!ok) return make_float4(0.f, 0.f, 0.f, 0.f);
    const float2 it = make_float2(inv_t, inv_t);
    const float2 nd = make_float2(-dot, -dot);
    const float2 a = mul2(mul2(make_float2(p.x, p.y), it),
                          add2(make_float2(g.x, g.y), nd));
    const float2 b = mul2(mul2(make_float2(p.z, p.w), it),
                          add2(make_float2(g.z, g.w), nd));
    return make_float4(a.x, a.y, b.x, b.y);
}

// The row's temperature as a multiplier: ok is false unless 0 < T < inf.
__device__ __forceinline__ float inv_temperature(float T, bool& ok) {
    ok = T > 0.0f && T < INFINITY;
    return ok ? __frcp_rn(T) : 0.0f;
}

// ------------------------------------------------------------------ row-group
// G lanes per row (a power of two dividing 32), E float4s of p and of g per
// lane in registers: lane i holds float4s i, i + G, ..., i + (E - 1) G.
template <int G, int E>
__global__ void __launch_bounds__(kBwdGroupThreads)
bwd_rowgroup_kernel(BwdTask t) {
    const int64_t gtid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const int64_t r = gtid / G;
    const int lane = static_cast<int>(gtid & (G - 1));
    const bool live = r < t.batch;
    const int C = t.num_classes;
    const int64_t off = live ? r * C : 0;
    const float* p = t.probs + off;
    const float* g = t.grad_out + off;
    float* o = t.grad_in + off;
    const int pad = pad_of(p);
    const int pg = pad_of(g);
    const int q4 = (pad + C + 3) >> 2;

    float4 pv[E], gv[E];
#pragma unroll
    for (int k = 0; k < E; ++k) {
        const int q = lane + k * G;
        pv[k] = gv[k] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (live && q < q4) {
            pv[k] = load4<true>(p, pad, pad, C, q);
            gv[k] = load4<true>(g, pg, pad, C, q);
        }
    }
    float2 a = make_float2(0.f, 0.f), b = make_float2(0.f, 0.f);
#pragma unroll
    for (int k = 0; k < E; ++k) dot_add(a, b, pv[k], gv[k]);
    float dot = (a.x + a.y) + (b.x + b.y);
    // Every lane of the group ends with the same bits (a + b = b + a).
#pragma unroll
    for (int m = G >> 1; m > 0; m >>= 1)
        dot += __shfl_xor_sync(0xffffffffu, dot, m);

    if (!live) return;
    bool ok;
    const float inv_t = inv_temperature(t.t[r], ok);
    const int po = pad_of(o);
#pragma unroll
    for (int k = 0; k < E; ++k) {
        const int q = lane + k * G;
        if (q < q4) store4(o, po, pad, C, q, grad4(pv[k], gv[k], dot, inv_t, ok));
    }
}

template <int G, int E>
cudaError_t launch_rg(const BwdTask& t, cudaStream_t stream) {
    const int64_t threads = t.batch * G;
    const int64_t blocks = (threads + kBwdGroupThreads - 1) / kBwdGroupThreads;
    bwd_rowgroup_kernel<G, E><<<static_cast<unsigned>(blocks), kBwdGroupThreads,
                                0, stream>>>(t);
    return cudaGetLastError();
}

template <int G>
cudaError_t launch_rg_e(const BwdTask& t, int e4, cudaStream_t stream) {
    switch (e4) {
        case 1: return launch_rg<G, 1>(t, stream);
        case 2: return launch_rg<G, 2>(t, stream);
        case 4: return launch_rg<G, 4>(t, stream);
        case 8: return launch_rg<G, 8>(t, stream);
        default: return cudaErrorInvalidValue;
    }
}

// -------------------------------------------------------------------- cluster
__device__ __forceinline__ void cluster_arrive_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_wait() {
    asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_wait_acquire() {
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ void fence_acq_rel_cluster() {
    asm volatile("fence.acq_rel.cluster;" ::: "memory");
}

// Plain store into (possibly remote) shared memory of the cluster.
__device__ __forceinline__ void st_cluster(uint32_t addr, float v) {
    asm volatile("st.shared::cluster.f32 [%0], %1;" :: "r"(addr), "f"(v)
                 : "memory");
}

// One cluster of n CTAs per row (rows cid, cid + clusters, ...).  CTA
// `rank` owns classes [rank L, rank L + L) of the row, L = slice_len (a
// multiple of 4), and thread i of it float4s i, i + nt, ... of that slice in
// every phase:
//   load     every float4 of p (and of g if STAGE_G) the thread owns as
//            one 16-byte asynchronous copy into shared memory, all in
//            flight at once; after they land, the thread's sum of p * g;
//   reduce   warp shuffle sum, per-warp slots and one __syncthreads, after
//            which every thread adds the slots in warp order; in a cluster,
//            thread i < n stores the CTA's sum into slot `rank` of CTA i
//            and fences, one cluster barrier, and every thread adds the n
//            slots in rank order.  All threads of the cluster hold the
//            same bits;
//   output   grad from the staged p (and g, or g read again: it was read
//            moments before, so it normally comes from L2).
// Slots are double-buffered by row parity: a CTA can store into a slot
// buffer again only after the next row's barrier, which its readers reach
// after reading it.
template <bool CLUSTER, bool STAGE_G>
__global__ void __launch_bounds__(kBwdMaxThreads, 2)
bwd_cluster_kernel(BwdTask t, int n, int slice_len) {
    extern __shared__ __align__(128) unsigned char smem[];
    float* cslot = reinterpret_cast<float*>(smem);   // [2][kMaxCluster]
    float* wslot = cslot + 2 * kMaxCluster;           // [2][32]
    float4* sp = reinterpret_cast<float4*>(smem + kBwdSmemHeader);
    float4* sg = sp + (slice_len / 4 + 1);
    const int nt = blockDim.x;
    const int warps = nt >> 5;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = CLUSTER ? cluster_ctarank() : 0u;
    const int64_t cid = blockIdx.x / n;
    const int64_t ncl = gridDim.x / n;
    const int64_t C = t.num_classes;
    const int64_t s0 = static_cast<int64_t>(rank) * slice_len;
    const int len = static_cast<int>(max(static_cast<int64_t>(0),
                                         min(static_cast<int64_t>(slice_len), C - s0)));
    // Remote stores need every CTA of the cluster running: this arrive is
    // matched by the wait before the first one.
    if (CLUSTER) cluster_arrive_relaxed();
    bool waited = false;

    uint32_t k = 0;
    for (int64_t r = cid; r < t.batch; r += ncl, ++k) {
        const int64_t off = r * C + s0;
        const float* p = t.probs + off;
        const float* g = t.grad_out + off;
        float* o = t.grad_in + off;
        const int pad = pad_of(p);
        const int pg = pad_of(g);
        const int q4 = len > 0 ? (pad + len + 3) >> 2 : 0;

        // Every float4 of the thread's share in flight at once.
        for (int q = threadIdx.x; q < q4; q += nt) {
            stage4(sp + q, p, pad, pad, len, q);
            if (STAGE_G) stage4(sg + q, g, pg, pad, len, q);
        }
        cp_async_wait_all();
        float2 a = make_float2(0.f, 0.f), b = make_float2(0.f, 0.f);
        int q = threadIdx.x;
        for (; q + 3 * nt < q4; q += 4 * nt) {
            float4 gv[4];
#pragma unroll
            for (int i = 0; i < 4; ++i)
                gv[i] = STAGE_G ? sg[q + i * nt] : load4<false>(g, pg, pad, len, q + i * nt);
#pragma unroll
            for (int i = 0; i < 4; ++i) dot_add(a, b, sp[q + i * nt], gv[i]);
        }
        for (; q < q4; q += nt)
            dot_add(a, b, sp[q], STAGE_G ? sg[q] : load4<false>(g, pg, pad, len, q));

        float dot = (a.x + a.y) + (b.x + b.y);
#pragma unroll
        for (int m = 16; m > 0; m >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, m);
        float* ws = wslot + (k & 1u) * 32;
        if (lane == 0) ws[warp] = dot;
        __syncthreads();
        dot = 0.0f;
        for (int w = 0; w < warps; ++w) dot += ws[w];
        if (CLUSTER) {
            float* cs = cslot + (k & 1u) * kMaxCluster;
            if (!waited) {
                cluster_wait();
                waited = true;
            }
            // Only the storing threads fence; the barrier itself is relaxed
            // on arrival and acquires on the wait (a release on every
            // thread's arrival cost 2% at 256 x 131072).
            if (threadIdx.x < static_cast<unsigned>(n)) {
                st_cluster(map_to_rank(smem_addr(&cs[rank]), threadIdx.x), dot);
                fence_acq_rel_cluster();
            }
            cluster_arrive_relaxed();
            cluster_wait_acquire();
            dot = 0.0f;
            for (int i = 0; i < n; ++i) dot += cs[i];
        }

        bool ok;
        const float inv_t = inv_temperature(t.t[r], ok);
        const int po = pad_of(o);
        q = threadIdx.x;
        for (; q + 3 * nt < q4; q += 4 * nt) {
            float4 gv[4];
#pragma unroll
            for (int i = 0; i < 4; ++i)
                gv[i] = STAGE_G ? sg[q + i * nt] : load4<true>(g, pg, pad, len, q + i * nt);
#pragma unroll
            for (int i = 0; i < 4; ++i)
                store4(o, po, pad, len, q + i * nt,
                       grad4(sp[q + i * nt], gv[i], dot, inv_t, ok));
        }
        for (; q < q4; q += nt) {
            const float4 gv = STAGE_G ? sg[q] : load4<true>(g, pg, pad, len, q);
            store4(o, po, pad, len, q, grad4(sp[q], gv, dot, inv_t, ok));
        }
    }
    if (CLUSTER && !waited) cluster_wait();
}

template <bool CLUSTER, bool STAGE_G>
cudaError_t launch_cl(const BwdTask& t, int n, int slice_len, int threads,
                      int smem_bytes, int64_t grid_ctas, cudaStream_t stream,
                      int slot) {
    auto kern = bwd_cluster_kernel<CLUSTER, STAGE_G>;
    cudaError_t e = ensure_smem_attribute(reinterpret_cast<const void*>(kern),
                                          slot, smem_bytes, CLUSTER);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid_ctas), 1, 1);
    cfg.blockDim = dim3(static_cast<unsigned>(threads), 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem_bytes);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    if (CLUSTER) {
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = static_cast<unsigned>(n);
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    return cudaLaunchKernelEx(&cfg, kern, t, n, slice_len);
}

}  // namespace

cudaError_t launch_backward_rowgroup(const BwdTask& task, int lanes_per_row,
                                     int elems_per_lane, cudaStream_t stream) {
    const int e4 = elems_per_lane / 4;
    switch (lanes_per_row) {
        case 1: return launch_rg_e<1>(task, e4, stream);
        case 2: return launch_rg_e<2>(task, e4, stream);
        case 4: return launch_rg_e<4>(task, e4, stream);
        case 8: return launch_rg_e<8>(task, e4, stream);
        case 16: return launch_rg_e<16>(task, e4, stream);
        case 32: return launch_rg_e<32>(task, e4, stream);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_backward_cluster(const BwdTask& task, int cluster_size,
                                    int slice_len, int threads, int smem_bytes,
                                    bool stage_g, int64_t grid_ctas,
                                    cudaStream_t stream) {
    if (cluster_size > 1)
        return stage_g ? launch_cl<true, true>(task, cluster_size, slice_len,
                                               threads, smem_bytes, grid_ctas,
                                               stream, 8)
                       : launch_cl<true, false>(task, cluster_size, slice_len,
                                                threads, smem_bytes, grid_ctas,
                                                stream, 9);
    return stage_g ? launch_cl<false, true>(task, 1, slice_len, threads,
                                            smem_bytes, grid_ctas, stream, 10)
                   : launch_cl<false, false>(task, 1, slice_len, threads,
                                             smem_bytes, grid_ctas, stream, 11);
}

}  // namespace cs
