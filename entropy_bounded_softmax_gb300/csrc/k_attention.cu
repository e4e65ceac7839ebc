// attention_softmax kernels ("BURT-IMMA CUDA Kernel API Reference",
// section 2.6).  scores is [B, H, S, S]; row r = (b H + h) S + i holds query
// i's scores against keys j = 0..S-1.  Per row:
//   1. v_j = scores_j + mask[b, j] (fp32 addition; mask NULL = 0; a mask of
//      -inf removes key j);
//   2. causal: keys j > i are removed and never read;
//   3. p = softmax over the kept keys with the max subtracted, 0 on removed
//      keys: p_j = 2^((v_j - m) log2 e) / sum.
// Section 5.3: a NaN or an infinity among the scores and mask values the
// row uses (a mask of -inf excepted) zeroes the row and sets NAN_INPUT (NaN
// seen) or INF_INPUT in the error word.  A row whose keys are all removed
// is written as zeros without a flag.
//
// Each kept score is read once and every output written once: 8 bytes per
// element without causal, (4 (i + 1) + 4 S) bytes for causal row i; the
// mask row is shared by the H S rows of its batch and stays in cache.
//   row-group  G lanes of a warp share a row (S up to 1024) and keep it in
//              registers; max and sum are G-lane butterflies;
//   row-CTA    one CTA per row (longer rows): the kept scores are copied
//              into shared memory with 16-byte cp.async, then three passes
//              there (v and the thread max; 2^y and the thread sum; the
//              output), each followed by a CTA reduction for the first two.
#include <math.h>

#include "cs_device.cuh"

namespace cs {
namespace {

using namespace csd;

__device__ __forceinline__ int pad_of(const void* a) {
    return static_cast<int>((reinterpret_cast<uintptr_t>(a) >> 2) & 3);
}

// Element j of a row sits at lane (j + pad) % 4 of float4 (j + pad) / 4,
// pad being the scores row's alignment in floats.  Loads float4 q of row
// a (own pad pa) for j < end; other lanes get `fill`.
template <bool STREAM>
__device__ __forceinline__ float4 load4f(const float* a, int pa, int pad,
                                         int end, int q, float fill) {
    const int j0 = 4 * q - pad;
    if (pa == pad && j0 >= 0 && j0 + 4 <= end) {
        const float4* v = reinterpret_cast<const float4*>(a + j0);
        return STREAM ? __ldcs(v) : __ldg(v);
    }
    float e[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int j = j0 + i;
        e[i] = fill;
        if (j >= 0 && j < end) e[i] = STREAM ? __ldcs(a + j) : __ldg(a + j);
    }
    return make_float4(e[0], e[1], e[2], e[3]);
}

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

// Step 1 on four lanes: v = s + m (m = 0 without a mask).  bad becomes NaN
// when a score is NaN or infinite or a mask value is NaN or +inf; lanes
// past the kept keys hold s = -inf, m = 0 and are not checked.  Whether a
// NaN was among them (the error code) is settled on the rare path by
// rescan_nan().
struct Step1 {
    float bad = 0.0f;
    __device__ __forceinline__ float one(float s, float m, bool kept,
                                         bool masked) {
        if (kept) {
            bad = fmaf(s, 0.0f, bad);
            if (masked) bad = fmaf(m == -INFINITY ? 0.0f : m, 0.0f, bad);
        }
        return __fadd_rn(s, m);
    }
    template <bool MASKED>
    __device__ __forceinline__ float4 apply(float4 s, float4 m, int q,
                                            int pad, int end) {
        const int j0 = 4 * q - pad;
        if (j0 >= 0 && j0 + 4 <= end)     // whole float4 kept
            return make_float4(one(s.x, m.x, true, MASKED),
                               one(s.y, m.y, true, MASKED),
                               one(s.z, m.z, true, MASKED),
                               one(s.w, m.w, true, MASKED));
        return make_float4(one(s.x, m.x, j0 >= 0 && j0 < end, MASKED),
                           one(s.y, m.y, j0 + 1 >= 0 && j0 + 1 < end, MASKED),
                           one(s.z, m.z, j0 + 2 >= 0 && j0 + 2 < end, MASKED),
                           one(s.w, m.w, j0 + 3 >= 0 && j0 + 3 < end, MASKED));
    }
};

// Rare path of a row with a non-finite input: whether a NaN is among its
// kept scores and mask values (read again from global memory, before any
// of the row is written).
__device__ bool rescan_nan(const float* s, const float* m, int end) {
    bool nan = false;
    for (int j = 0; j < end; ++j) nan = nan || isnan(s[j]) || (m && isnan(m[j]));
    return nan;
}

__device__ __forceinline__ float max4(float4 v) {
    return fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w));
}

// 2^((v - m) log2 e) on four lanes (-inf gives 0).
__device__ __forceinline__ float4 exp4(float4 v, float m) {
    return make_float4(ex2((v.x - m) * kLog2e), ex2((v.y - m) * kLog2e),
                       ex2((v.z - m) * kLog2e), ex2((v.w - m) * kLog2e));
}

__device__ __forceinline__ float4 scale4(float4 v, float f) {
    const float2 a = mul2(make_float2(v.x, v.y), make_float2(f, f));
    const float2 b = mul2(make_float2(v.z, v.w), make_float2(f, f));
    return make_float4(a.x, a.y, b.x, b.y);
}

struct RowRef {
    const float* s;    // scores row
    const float* m;    // mask row or null
    float* o;          // output row
    int end;           // kept keys: [0, end)
};

__device__ __forceinline__ RowRef row_ref(const AttnTask& t, int64_t r) {
    const int64_t S = t.seq_len;
    const int64_t b = r / (static_cast<int64_t>(t.heads) * S);
    const int i = static_cast<int>(r % S);
    RowRef x;
    x.s = t.scores + r * S;
    x.m = t.mask ? t.mask + b * S : nullptr;
    x.o = t.out + r * S;
    x.end = t.causal ? i + 1 : static_cast<int>(S);
    return x;
}

// ------------------------------------------------------------------ row-group
template <int G, int E>
__global__ void __launch_bounds__(kAttnGroupThreads)
attn_rowgroup_kernel(AttnTask t) {
    const int64_t gtid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const int64_t r = gtid / G;
    const int lane = static_cast<int>(gtid & (G - 1));
    const bool live = r < t.rows;
    const int S = t.seq_len;
    const RowRef x = row_ref(t, live ? r : 0);
    const int pad = pad_of(x.s);
    const int pm = x.m ? pad_of(x.m) : 0;
    const int q4 = (pad + S + 3) >> 2;
    const int qk = live ? (pad + x.end + 3) >> 2 : 0;   // float4s with kept keys

    float4 v[E];
#pragma unroll
    for (int k = 0; k < E; ++k) {
        const int q = lane + k * G;
        v[k] = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
        if (q < qk) v[k] = load4f<true>(x.s, pad, pad, x.end, q, -INFINITY);
    }
    Step1 st;
    float mx = -INFINITY;
#pragma unroll
    for (int k = 0; k < E; ++k) {
        const int q = lane + k * G;
        if (q < qk) {
            if (x.m)
                v[k] = st.apply<true>(v[k], load4f<false>(x.m, pm, pad, x.end, q, 0.0f),
                                      q, pad, x.end);
            else
                v[k] = st.apply<false>(v[k], make_float4(0.f, 0.f, 0.f, 0.f), q,
                                       pad, x.end);
        }
        mx = fmaxf(mx, max4(v[k]));
    }
    float bad = st.bad;
#pragma unroll
    for (int o = G >> 1; o > 0; o >>= 1) {
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        bad += __shfl_xor_sync(0xffffffffu, bad, o);
    }
    const bool zero = bad != bad || mx == -INFINITY;
    float2 sum = make_float2(0.f, 0.f);
#pragma unroll
    for (int k = 0; k < E; ++k) {
        const int q = lane + k * G;
        if (q < qk && !zero) {
            v[k] = exp4(v[k], mx);
            sum = add2(sum, add2(make_float2(v[k].x, v[k].y), make_float2(v[k].z, v[k].w)));
        }
    }
    float tot = sum.x + sum.y;
#pragma unroll
    for (int o = G >> 1; o > 0; o >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, o);
    // The row's error code, read before any of it is written (in place).
    unsigned int code = 0;
    if (bad != bad) {
        const unsigned int gmask = (G == 32 ? 0xffffffffu : ((1u << G) - 1u))
                                   << ((threadIdx.x & 31) & ~(G - 1));
        if (lane == 0 && live) code = rescan_nan(x.s, x.m, x.end) ? kBitNan : kBitInf;
        __syncwarp(gmask);
    }
    if (!live) return;
    const float inv = zero ? 0.0f : __frcp_rn(tot);
    const int po = pad_of(x.o);
#pragma unroll
    for (int k = 0; k < E; ++k) {
        const int q = lane + k * G;
        if (q < q4) store4(x.o, po, pad, S, q, (q < qk && !zero) ? scale4(v[k], inv)
                                                                 : make_float4(0.f, 0.f, 0.f, 0.f));
    }
    if (lane == 0) raise_error(t.err, code);
}

template <int G, int E>
cudaError_t launch_rg(const AttnTask& t, cudaStream_t stream) {
    const int64_t threads = t.rows * G;
    const int64_t blocks = (threads + kAttnGroupThreads - 1) / kAttnGroupThreads;
    attn_rowgroup_kernel<G, E><<<static_cast<unsigned>(blocks), kAttnGroupThreads,
                                 0, stream>>>(t);
    return cudaGetLastError();
}

template <int G>
cudaError_t launch_rg_e(const AttnTask& t, int e4, cudaStream_t stream) {
    switch (e4) {
        case 1: return launch_rg<G, 1>(t, stream);
        case 2: return launch_rg<G, 2>(t, stream);
        case 4: return launch_rg<G, 4>(t, stream);
        case 8: return launch_rg<G, 8>(t, stream);
        default: return cudaErrorInvalidValue;
    }
}

// -------------------------------------------------------------------- row-CTA
// CTA-wide reduction of (max of a, sum of c, max of d) through per-warp
// slots; every thread gets the same bits.  slot: 48 floats of shared
// memory; a slot is written again only after the caller's next
// __syncthreads.
__device__ __forceinline__ void cta_reduce(float& a, float& c, float& d,
                                           float* slot) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
        c += __shfl_xor_sync(0xffffffffu, c, o);
        d = fmaxf(d, __shfl_xor_sync(0xffffffffu, d, o));
    }
    const int warps = static_cast<int>(blockDim.x >> 5);
    const int w0 = threadIdx.x >> 5;
    if ((threadIdx.x & 31) == 0) {
        slot[w0] = a;
        slot[16 + w0] = c;
        slot[32 + w0] = d;
    }
    __syncthreads();
    a = slot[0];
    c = slot[16];
    d = slot[32];
    for (int w = 1; w < warps; ++w) {
        a = fmaxf(a, slot[w]);
        c += slot[16 + w];
        d = fmaxf(d, slot[32 + w]);
    }
}

// One CTA per row (rows blockIdx.x, + gridDim.x, ...).  Thread t owns
// float4s t, t + nt, ... of the row in every pass.
__global__ void __launch_bounds__(kAttnMaxThreads)
attn_cta_kernel(AttnTask t) {
    extern __shared__ __align__(128) unsigned char smem[];
    float* slot_a = reinterpret_cast<float*>(smem);          // [48]
    float* slot_b = slot_a + 48;                              // [48]
    float4* row4 = reinterpret_cast<float4*>(smem + kAttnSmemHeader);
    const int nt = blockDim.x;
    const int S = t.seq_len;
    for (int64_t r = blockIdx.x; r < t.rows; r += gridDim.x) {
        const RowRef x = row_ref(t, r);
        const int pad = pad_of(x.s);
        const int pm = x.m ? pad_of(x.m) : 0;
        const int q4 = (pad + S + 3) >> 2;
        const int qk = (pad + x.end + 3) >> 2;
        // Copy the kept scores in (whole aligned float4s asynchronously).
        for (int q = threadIdx.x; q < qk; q += nt) {
            const int j0 = 4 * q - pad;
            if (j0 >= 0 && j0 + 4 <= x.end) cp_async16(&row4[q], x.s + j0);
            else row4[q] = load4f<true>(x.s, pad, pad, x.end, q, -INFINITY);
        }
        cp_async_wait_all();
        // Pass 1: v = s + m in place, the thread's max and check.
        Step1 st;
        float mx = -INFINITY;
        for (int q = threadIdx.x; q < qk; q += nt) {
            const float4 v = x.m
                ? st.apply<true>(row4[q], load4f<false>(x.m, pm, pad, x.end, q, 0.0f),
                                 q, pad, x.end)
                : st.apply<false>(row4[q], make_float4(0.f, 0.f, 0.f, 0.f), q,
                                  pad, x.end);
            row4[q] = v;
            mx = fmaxf(mx, max4(v));
        }
        float bad = st.bad, unused_d = 0.0f;
        cta_reduce(mx, bad, unused_d, slot_a);
        const bool zero = bad != bad || mx == -INFINITY;
        // Pass 2: 2^y in place and the thread's sum.
        float2 sum = make_float2(0.f, 0.f);
        for (int q = threadIdx.x; q < (zero ? 0 : qk); q += nt) {
            const float4 e = exp4(row4[q], mx);
            row4[q] = e;
            sum = add2(sum, add2(make_float2(e.x, e.y), make_float2(e.z, e.w)));
        }
        float unused_a = -INFINITY, tot = sum.x + sum.y, unused_b = 0.0f;
        cta_reduce(unused_a, tot, unused_b, slot_b);
        const float inv = zero ? 0.0f : __frcp_rn(tot);
        // The row's error code, read before any of it is written (in place).
        unsigned int code = 0;
        if (bad != bad) {
            if (threadIdx.x == 0) code = rescan_nan(x.s, x.m, x.end) ? kBitNan : kBitInf;
            __syncthreads();
        }
        // Pass 3: the output, zeros past the kept keys and on zeroed rows.
        const int po = pad_of(x.o);
        const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int q = threadIdx.x; q < q4; q += nt)
            store4(x.o, po, pad, S, q, (q < qk && !zero) ? scale4(row4[q], inv) : z);
        if (threadIdx.x == 0) raise_error(t.err, code);
        // The row buffer and slots are rewritten by the next row.
        __syncthreads();
    }
}

}  // namespace

cudaError_t launch_attention_rowgroup(const AttnTask& task, int lanes_per_row,
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

cudaError_t launch_attention_cta(const AttnTask& task, int threads,
                                 int smem_bytes, int64_t grid_ctas,
                                 cudaStream_t stream) {
    const void* kern = reinterpret_cast<const void*>(attn_cta_kernel);
    cudaError_t e = ensure_smem_attribute(kern, 12, smem_bytes, false);
    if (e != cudaSuccess) return e;
    attn_cta_kernel<<<static_cast<unsigned>(grid_ctas), threads,
                      static_cast<size_t>(smem_bytes), stream>>>(task);
    return cudaGetLastError();
}

}  // namespace cs
