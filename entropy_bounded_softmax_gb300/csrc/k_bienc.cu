// biencoder_attention ("BURT-IMMA CUDA Kernel API Reference", section 2.5),
// fused: for every (batch, head) pair bh and query i,
//   1. s_j = fl(dot(q_i, k_j) * scale), the dot product accumulated in fp32
//      with one fused multiply-add per d in order d = 0..D-1 (the fp32
//      evaluation the oracle fixes, so both sides search the same logits);
//   2. attn = constrained_softmax(s) over the K context items (section 2.1,
//      with sections 5.3 and 5.4): the row-group search of cs_rowgroup.cuh;
//   3. out_i = sum_j attn_j v_j.
// Nothing between the steps goes to global memory (the scores and weights
// live in registers and shared memory); optionally the weights and the
// temperatures are written out too.
//
// One CTA per bh and run of query tiles (R = threads / G rows a tile,
// about 128 rows a CTA): the keys (transposed, d-major) and values of bh are
// staged in shared memory once, then each tile's queries in turn.  G lanes share a query row: lane `sub` owns keys
// j = 4 (i G + sub) + c (i < 2, c < 4), eight per lane, read as float4s of
// the transposed keys, and output columns 4 (sub + k G) .. + 3.
#include <math.h>

#include "cs_rowgroup.cuh"

namespace cs {
namespace {

using namespace csd;

constexpr int kBiencE4 = 2;   // float4s of keys per lane: 8 keys

struct BiencSmem {
    float* kt;   // [D][kp] keys, transposed
    float* vs;   // [K][D] values (STEP3)
    float* qs;   // [R][D + 4] query rows
    float* ps;   // [R][kp + 4] attention weights (STEP3)
};

// STEP3: all three steps (the fp32 FMA contraction of step 3 included);
// otherwise steps 1 and 2 only, the weights written to t.p_out (row
// stride t.p_stride) for the tensor-core step 3 of k_bienc_pv.cu, and
// neither the values nor the weights staged in shared memory.
template <int G, bool STEP3>
__global__ void __launch_bounds__(bienc_threads(G))
bienc_kernel(BiencTask t, int tiles, int tiles_per_cta) {
    constexpr int R = bienc_threads(G) / G;
    extern __shared__ __align__(16) float smem_f[];
    const int K = t.K, D = t.D;
    const int kp = bienc_kp(K);
    BiencSmem sm;
    sm.kt = smem_f;
    sm.vs = sm.kt + D * kp;
    sm.qs = sm.vs + (STEP3 ? K * D : 0);
    sm.ps = sm.qs + R * (D + 4);

    const int ctas_per_bh = (tiles + tiles_per_cta - 1) / tiles_per_cta;
    const int64_t bh = blockIdx.x / ctas_per_bh;
    const int tile0 = (blockIdx.x % ctas_per_bh) * tiles_per_cta;
    const int tile1 = min(tiles, tile0 + tiles_per_cta);
    const float* kg = t.k + bh * K * D;
    const float* vg = t.v + bh * K * D;

    // A tile's queries go into qs by 16-byte asynchronous copies (D is a
    // multiple of 4 and the bases are 16-byte aligned), issued as soon as
    // the previous tile's queries have been read, so that they land while
    // that tile searches and accumulates its outputs.
    const int D4 = D >> 2;
    auto stage_queries = [&](int tile) {
        const int i0 = tile * R;
        const int nrows = min(R, t.Q - i0);
        const float* qg = t.q + (bh * t.Q + i0) * D;
        for (int e = threadIdx.x; e < nrows * D4; e += blockDim.x) {
            const int r = e / D4, c4 = e - r * D4;
            cp_async16(sm.qs + r * (D + 4) + 4 * c4, qg + r * D + 4 * c4);
        }
    };
    if (tile0 < tile1) stage_queries(tile0);

    // Stage the keys (transposed, zero past K) and values of bh once.  A
    // thread reads four consecutive d of one key (16 bytes) and writes them
    // to four rows of the transposed buffer; consecutive threads take
    // consecutive keys, so each of those shared stores hits 32 different
    // banks.  The values are copied as they are, 16 bytes at a time.
    for (int e = threadIdx.x; e < K * D4; e += blockDim.x) {
        const int j = e % K, c4 = e / K;
        const float4 kv = __ldg(reinterpret_cast<const float4*>(kg + j * D) + c4);
        sm.kt[(4 * c4 + 0) * kp + j] = kv.x;
        sm.kt[(4 * c4 + 1) * kp + j] = kv.y;
        sm.kt[(4 * c4 + 2) * kp + j] = kv.z;
        sm.kt[(4 * c4 + 3) * kp + j] = kv.w;
    }
    for (int e = threadIdx.x; e < D * (kp - K); e += blockDim.x)
        sm.kt[(e / (kp - K)) * kp + K + e % (kp - K)] = 0.0f;
    if (STEP3)
        for (int e = threadIdx.x; e < K * D4; e += blockDim.x)
            cp_async16(sm.vs + 4 * e, vg + 4 * e);

    for (int tile = tile0; tile < tile1; ++tile) {
        const int i0 = tile * R;
        const int nrows = min(R, t.Q - i0);
        // This thread's copies of the tile's queries have landed; after the
        // barrier every thread's have (and the keys and values are staged).
        cp_async_wait_all();
        __syncthreads();

        const int lane = threadIdx.x & 31;
        const int sub = lane & (G - 1);
        const int rr = threadIdx.x / G;
        const unsigned gmask =
            G == 32 ? 0xffffffffu : (((1u << G) - 1u) << (lane & ~(G - 1)));
        const bool live = rr < nrows;
        const float* qr = sm.qs + (live ? rr : 0) * (D + 4);

        // Step 1: eight scores per lane, each an in-order fma chain over d.
        float4 acc[kBiencE4];
#pragma unroll
        for (int i = 0; i < kBiencE4; ++i) acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int d4 = 0; d4 < D; d4 += 4) {
            const float4 qv = *reinterpret_cast<const float4*>(qr + d4);
            const float qd[4] = {qv.x, qv.y, qv.z, qv.w};
#pragma unroll
            for (int dd = 0; dd < 4; ++dd) {
                const float* krow = sm.kt + (d4 + dd) * kp;
#pragma unroll
                for (int i = 0; i < kBiencE4; ++i) {
                    const int j0 = 4 * (i * G + sub);
                    if (j0 < kp) {
                        const float4 kv = *reinterpret_cast<const float4*>(krow + j0);
                        acc[i].x = fmaf(qd[dd], kv.x, acc[i].x);
                        acc[i].y = fmaf(qd[dd], kv.y, acc[i].y);
                        acc[i].z = fmaf(qd[dd], kv.z, acc[i].z);
                        acc[i].w = fmaf(qd[dd], kv.w, acc[i].w);
                    }
                }
            }
        }
        float4 y[kBiencE4];
        float m = -INFINITY, bad = 0.0f;
#pragma unroll
        for (int i = 0; i < kBiencE4; ++i) {
            const float a[4] = {acc[i].x, acc[i].y, acc[i].z, acc[i].w};
            float s[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int j = 4 * (i * G + sub) + c;
                s[c] = -INFINITY;
                if (live && j < K) {
                    s[c] = __fmul_rn(a[c], t.scale);
                    m = fmaxf(m, s[c]);
                    bad = fmaf(s[c], 0.0f, bad);
                }
            }
            y[i] = make_float4(s[0], s[1], s[2], s[3]);
        }
        // Every thread has read its query row: the next tile's queries may
        // overwrite qs while this tile goes on.
        __syncthreads();
        if (tile + 1 < tile1) stage_queries(tile + 1);

        // Step 2: the row's constrained softmax.
        const SearchCfg cfg{t.t_min, t.hi0, t.entropy_bound,
                            t.entropy_bound * kLog2e,
                            t.entropy_bound > 0.0f ? lg2_approx(t.entropy_bound) : 0.0f,
                            make_grid(t.t_min, fmaxf(t.hi0, t.t_min), t.max_iter)};
        RowSolution sol{NAN, 0.0f, 0.0f, 0u, 0, true};
        if (live)   // uniform over the lane group
            sol = solve_row<G, kBiencE4>(y, m, bad, cfg, t.entropy_bound * kLog2e,
                                         false, gmask);
        float* pr = sm.ps + (live ? rr : 0) * (kp + 4);
        const int64_t row = bh * t.Q + i0 + rr;
#pragma unroll
        for (int i = 0; i < kBiencE4; ++i) {
            const float yy[4] = {y[i].x, y[i].y, y[i].z, y[i].w};
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int j = 4 * (i * G + sub) + c;
                if (live && j < K) {
                    const float p = sol.zero ? 0.0f : ex2(yy[c] * sol.beta_out) * sol.inv_s;
                    if (STEP3) {
                        pr[j] = p;
                        if (t.attn_out) __stcs(t.attn_out + row * K + j, p);
                    } else {
                        // Read back by the step-3 kernel moments later (L2).
                        t.p_out[row * t.p_stride + j] = p;
                    }
                }
            }
        }
        if (!STEP3) {
            if (live && sub == 0) {
                if (t.t_out) t.t_out[row] = sol.T_row;
                raise_error(t.err, sol.bits);
            }
            continue;
        }
        __syncwarp(gmask);

        // Step 3: four output columns at a time, keys in order.
        if (live) {
            float* og = t.out + row * D;
            for (int c0 = 4 * sub; c0 < D; c0 += 4 * G) {
                float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
                for (int j = 0; j < K; ++j) {
                    const float p = pr[j];
                    const float4 v = *reinterpret_cast<const float4*>(sm.vs + j * D + c0);
                    o.x = fmaf(p, v.x, o.x);
                    o.y = fmaf(p, v.y, o.y);
                    o.z = fmaf(p, v.z, o.z);
                    o.w = fmaf(p, v.w, o.w);
                }
                __stcs(reinterpret_cast<float4*>(og + c0), o);
            }
            if (sub == 0) {
                if (t.t_out) t.t_out[row] = sol.T_row;
                raise_error(t.err, sol.bits);
            }
        }
        // The weights row (ps) is read only by its own lane group (after its
        // __syncwarp), and the next tile's qs is guarded by the barrier at
        // the top of the loop: no barrier here.
    }
}

template <bool STEP3>
cudaError_t launch_bienc_as(const BiencTask& task, int lanes_per_row,
                            int smem_bytes, cudaStream_t stream) {
    const int rows_per_tile = bienc_threads(lanes_per_row) / lanes_per_row;
    const int tiles = (task.Q + rows_per_tile - 1) / rows_per_tile;
    const int tiles_per_cta = bienc_tiles_per_cta(task.Q, lanes_per_row);
    const int64_t grid = static_cast<int64_t>(task.BH) *
                         ((tiles + tiles_per_cta - 1) / tiles_per_cta);
    const void* kern = nullptr;
    switch (lanes_per_row) {
        case 1: kern = reinterpret_cast<const void*>(bienc_kernel<1, STEP3>); break;
        case 2: kern = reinterpret_cast<const void*>(bienc_kernel<2, STEP3>); break;
        case 4: kern = reinterpret_cast<const void*>(bienc_kernel<4, STEP3>); break;
        case 8: kern = reinterpret_cast<const void*>(bienc_kernel<8, STEP3>); break;
        case 16: kern = reinterpret_cast<const void*>(bienc_kernel<16, STEP3>); break;
        case 32: kern = reinterpret_cast<const void*>(bienc_kernel<32, STEP3>); break;
        default: return cudaErrorInvalidValue;
    }
    // One attribute slot per lane count: 13..18 (all three steps), 28..33
    // (steps 1 and 2).
    int slot = STEP3 ? 13 : 28;
    for (int g = lanes_per_row; g > 1; g >>= 1) ++slot;
    cudaError_t e = ensure_smem_attribute(kern, slot, smem_bytes, false);
    if (e != cudaSuccess) return e;
    const dim3 gd(static_cast<unsigned>(grid)), bd(bienc_threads(lanes_per_row));
    switch (lanes_per_row) {
        case 1: bienc_kernel<1, STEP3><<<gd, bd, smem_bytes, stream>>>(task, tiles, tiles_per_cta); break;
        case 2: bienc_kernel<2, STEP3><<<gd, bd, smem_bytes, stream>>>(task, tiles, tiles_per_cta); break;
        case 4: bienc_kernel<4, STEP3><<<gd, bd, smem_bytes, stream>>>(task, tiles, tiles_per_cta); break;
        case 8: bienc_kernel<8, STEP3><<<gd, bd, smem_bytes, stream>>>(task, tiles, tiles_per_cta); break;
        case 16: bienc_kernel<16, STEP3><<<gd, bd, smem_bytes, stream>>>(task, tiles, tiles_per_cta); break;
        default: bienc_kernel<32, STEP3><<<gd, bd, smem_bytes, stream>>>(task, tiles, tiles_per_cta); break;
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bienc(const BiencTask& task, int lanes_per_row,
                         int smem_bytes, cudaStream_t stream) {
    return task.p_out
        ? launch_bienc_as<false>(task, lanes_per_row, smem_bytes, stream)
        : launch_bienc_as<true>(task, lanes_per_row, smem_bytes, stream);
}

}  // namespace cs
