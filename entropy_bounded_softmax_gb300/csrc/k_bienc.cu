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
// staged in shared memory once, then each tile's queries in turn.
//
// Step 1 is register-blocked: a thread computes a 4-row x 4-item block of
// the tile's scores, so every query and key value read from shared memory
// serves four products (the reads of a row-per-lane layout, a float4 of keys
// per four products plus the query, made shared memory the bound).  Each
// score is still one fma chain over d in order.  The blocks go to a scores
// tile in shared memory, from which the search takes its own layout: G
// lanes share a query row, lane `sub` owning items j = 4 (i G + sub) + c
// (i < E4, c < 4), 4 E4 per lane, and output columns 4 (sub + k G) .. + 3.
#include <math.h>

#include "cs_rowgroup.cuh"

namespace cs {
namespace {

using namespace csd;

struct BiencSmem {
    float* kt;   // [D][kp] keys, transposed
    float* vs;   // [K][D] values (STEP3)
    float* qs;   // [R][D + 4] query rows
    float* ss;   // [R][ss_stride] scores, then (STEP3) attention weights
};

// STEP3: all three steps (the fp32 FMA contraction of step 3 included);
// otherwise steps 1 and 2 only, the weights written to t.p_out (row
// stride t.p_stride) for the tensor-core step 3 of k_bienc_pv.cu, and
// neither the values nor the weights staged in shared memory.
template <int G, int E4, bool STEP3>
__global__ void __launch_bounds__(bienc_threads(G), 2048 / bienc_threads(G) / 2)
bienc_kernel(BiencTask t, int tiles, int tiles_per_cta) {
    constexpr int R = bienc_threads(G) / G;
    extern __shared__ __align__(16) float smem_f[];
    const int K = t.K, D = t.D;
    const int kp = bienc_kp(K);
    const int ssw = bienc_ss_stride(K, G);
    BiencSmem sm;
    sm.kt = smem_f;
    sm.vs = sm.kt + D * kp;
    sm.qs = sm.vs + (STEP3 ? K * D : 0);
    sm.ss = sm.qs + R * (D + 4);
    // This thread's step-1 block: rows 4 br .. + 3, items 4 bj .. + 3
    // (consecutive threads take consecutive item blocks); at most R kp / 16
    // <= threads blocks.
    const int nbj = kp >> 2;
    const int br = threadIdx.x / nbj;
    const int bj = threadIdx.x - br * nbj;
    const bool blk = br < (R >> 2);

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

        // Step 1: the thread's 4 x 4 block of scores, each an in-order fma
        // chain over d; two chains per packed fma (each half rounded as its
        // own fmaf).
        if (blk) {
            float2 acc[4][2];
#pragma unroll
            for (int r = 0; r < 4; ++r) acc[r][0] = acc[r][1] = make_float2(0.f, 0.f);
            const float* q0 = sm.qs + 4 * br * (D + 4);
            const float* k0 = sm.kt + 4 * bj;
            for (int d4 = 0; d4 < D; d4 += 4) {
                float4 qv[4];
#pragma unroll
                for (int r = 0; r < 4; ++r)
                    qv[r] = *reinterpret_cast<const float4*>(q0 + r * (D + 4) + d4);
#pragma unroll
                for (int dd = 0; dd < 4; ++dd) {
                    const float4 kv = *reinterpret_cast<const float4*>(k0 + (d4 + dd) * kp);
                    const float2 k01 = make_float2(kv.x, kv.y);
                    const float2 k23 = make_float2(kv.z, kv.w);
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        const float qd = dd == 0 ? qv[r].x : dd == 1 ? qv[r].y
                                       : dd == 2 ? qv[r].z : qv[r].w;
                        const float2 q2 = make_float2(qd, qd);
                        acc[r][0] = fma2(q2, k01, acc[r][0]);
                        acc[r][1] = fma2(q2, k23, acc[r][1]);
                    }
                }
            }
            const float2 sc = make_float2(t.scale, t.scale);
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const float2 s01 = mul2(acc[r][0], sc);
                const float2 s23 = mul2(acc[r][1], sc);
                *reinterpret_cast<float4*>(sm.ss + (4 * br + r) * ssw + 4 * bj) =
                    make_float4(s01.x, s01.y, s23.x, s23.y);
            }
        }
        // Every thread has read the tile's queries and the scores are in
        // place: the next tile's queries may overwrite qs while this tile
        // goes on.
        __syncthreads();
        if (tile + 1 < tile1) stage_queries(tile + 1);

        const int lane = threadIdx.x & 31;
        const int sub = lane & (G - 1);
        const int rr = threadIdx.x / G;
        const unsigned gmask =
            G == 32 ? 0xffffffffu : (((1u << G) - 1u) << (lane & ~(G - 1)));
        const bool live = rr < nrows;
        float* pr = sm.ss + (live ? rr : 0) * ssw;
        float4 y[E4];
        float m = -INFINITY, bad = 0.0f;
#pragma unroll
        for (int i = 0; i < E4; ++i) {
            const int j0 = 4 * (i * G + sub);
            float s[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
            if (live && j0 < kp) {
                const float4 v4 = *reinterpret_cast<const float4*>(pr + j0);
                s[0] = v4.x;
                s[1] = v4.y;
                s[2] = v4.z;
                s[3] = v4.w;
            }
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                if (live && j0 + c < K) {
                    m = fmaxf(m, s[c]);
                    bad = fmaf(s[c], 0.0f, bad);
                } else {
                    s[c] = -INFINITY;
                }
            }
            y[i] = make_float4(s[0], s[1], s[2], s[3]);
        }

        // Step 2: the row's constrained softmax.
        const SearchCfg cfg{t.t_min, t.hi0, t.entropy_bound,
                            t.entropy_bound * kLog2e,
                            t.entropy_bound > 0.0f ? lg2_approx(t.entropy_bound) : 0.0f,
                            make_grid(t.t_min, fmaxf(t.hi0, t.t_min), t.max_iter)};
        RowSolution sol{NAN, 0.0f, 0.0f, 0u, 0, true};
        if (live)   // uniform over the lane group
            sol = solve_row<G, E4, true>(y, m, bad, cfg, t.entropy_bound * kLog2e,
                                   false, gmask);
        const int64_t row = bh * t.Q + i0 + rr;
#pragma unroll
        for (int i = 0; i < E4; ++i) {
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
        // The weights row (in ss) is read only by its own lane group (after
        // its __syncwarp), and the next tile's qs is guarded by the barrier at
        // the top of the loop: no barrier here.
    }
}

template <int E4, bool STEP3>
cudaError_t launch_bienc_as(const BiencTask& task, int lanes_per_row,
                            int smem_bytes, cudaStream_t stream) {
    const int rows_per_tile = bienc_threads(lanes_per_row) / lanes_per_row;
    const int tiles = (task.Q + rows_per_tile - 1) / rows_per_tile;
    const int tiles_per_cta = bienc_tiles_per_cta(task.Q, lanes_per_row);
    const int64_t grid = static_cast<int64_t>(task.BH) *
                         ((tiles + tiles_per_cta - 1) / tiles_per_cta);
    const void* kern = nullptr;
    switch (lanes_per_row) {
        case 1: kern = reinterpret_cast<const void*>(bienc_kernel<1, E4, STEP3>); break;
        case 2: kern = reinterpret_cast<const void*>(bienc_kernel<2, E4, STEP3>); break;
        case 4: kern = reinterpret_cast<const void*>(bienc_kernel<4, E4, STEP3>); break;
        case 8: kern = reinterpret_cast<const void*>(bienc_kernel<8, E4, STEP3>); break;
        case 16: kern = reinterpret_cast<const void*>(bienc_kernel<16, E4, STEP3>); break;
        case 32: kern = reinterpret_cast<const void*>(bienc_kernel<32, E4, STEP3>); break;
        default: return cudaErrorInvalidValue;
    }
    // One attribute slot per lane count: 13..18 (all three steps) and
    // 28..33 (steps 1 and 2) with eight keys a lane, 40..45 and 46..51 with
    // sixteen.
    int slot = E4 == 2 ? (STEP3 ? 13 : 28) : (STEP3 ? 40 : 46);
    for (int g = lanes_per_row; g > 1; g >>= 1) ++slot;
    cudaError_t e = ensure_smem_attribute(kern, slot, smem_bytes, false);
    if (e != cudaSuccess) return e;
    const dim3 gd(static_cast<unsigned>(grid)), bd(bienc_threads(lanes_per_row));
    switch (lanes_per_row) {
        case 1: bienc_kernel<1, E4, STEP3><<<gd, bd, smem_bytes, stream>>>(task, tiles, tiles_per_cta); break;
        case 2: bienc_kernel<2, E4, STEP3><<<gd, bd, smem_bytes, stream>>>(task, tiles, tiles_per_cta); break;
        case 4: bienc_kernel<4, E4, STEP3><<<gd, bd, smem_bytes, stream>>>(task, tiles, tiles_per_cta); break;
        case 8: bienc_kernel<8, E4, STEP3><<<gd, bd, smem_bytes, stream>>>(task, tiles, tiles_per_cta); break;
        case 16: bienc_kernel<16, E4, STEP3><<<gd, bd, smem_bytes, stream>>>(task, tiles, tiles_per_cta); break;
        default: bienc_kernel<32, E4, STEP3><<<gd, bd, smem_bytes, stream>>>(task, tiles, tiles_per_cta); break;
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bienc(const BiencTask& task, int lanes_per_row,
                         int keys_per_lane, int smem_bytes,
                         cudaStream_t stream) {
    if (keys_per_lane == 16)
        return task.p_out
            ? launch_bienc_as<4, false>(task, lanes_per_row, smem_bytes, stream)
            : launch_bienc_as<4, true>(task, lanes_per_row, smem_bytes, stream);
    if (keys_per_lane != 8) return cudaErrorInvalidValue;
    return task.p_out
        ? launch_bienc_as<2, false>(task, lanes_per_row, smem_bytes, stream)
        : launch_bienc_as<2, true>(task, lanes_per_row, smem_bytes, stream);
}

}  // namespace cs
