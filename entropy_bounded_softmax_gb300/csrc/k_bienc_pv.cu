// Step 3 of biencoder_attention ("BURT-IMMA CUDA Kernel API Reference",
// section 2.5 Description step 3, out = attn @ context_values) on the
// 5th-generation tensor cores, as a second kernel after the fused scores
// and search kernel (k_bienc.cu) has written the weights P [bh, Q, K].
//
// One CTA per (bh, 128 query rows): out[128 x D] = P[128 x K] . V[K x D],
// a tcgen05.mma of kind::tf32 with M = 128, N = D rounded up to 16, K in
// steps of 8, the fp32 accumulator in tensor memory.  fp32 accuracy comes
// from three TF32 products per fp32 product: with x_hi the TF32 nearest x
// and x_lo the TF32 nearest x - x_hi,
//   P V ~ P_hi V_hi + P_hi V_lo + P_lo V_hi,
// which leaves out only P_lo V_lo and the two lo roundings (about 2^-21 of
// |P||V| each), next to the fp32 accumulation's own rounding.
//
// Operands go to shared memory as TF32 values in the MMA's canonical
// K-major layout without swizzle: 8-row x 16-byte core matrices (8 rows x
// 4 context items), core (row group m, item group g) at
// (g * rows / 8 + m) * 128 bytes, so the descriptor's leading (K-direction)
// byte offset is rows / 8 * 128 and its stride (row-direction) offset 128.
// The context is staged kPvKc items at a time, the tensor memory
// accumulating across chunks.  Warp w then reads rows 32 w .. 32 w + 31 of the
// accumulator (its quarter of the tensor-memory lanes) and stores them.
#include "cs_tcgen05.cuh"

namespace cs {
namespace {

using namespace csd;

constexpr int kPvThreads = 128;   // one warpgroup

__global__ void __launch_bounds__(kPvThreads, 1)
bienc_pv_kernel(PvTask t) {
    extern __shared__ __align__(1024) unsigned char smem[];
    const int Np = pv_np(t.D);
    const PvSmemLayout L = pv_smem_layout(Np);
    float* a_hi = reinterpret_cast<float*>(smem + L.a_hi);
    float* a_lo = reinterpret_cast<float*>(smem + L.a_lo);
    float* b_hi = reinterpret_cast<float*>(smem + L.b_hi);
    float* b_lo = reinterpret_cast<float*>(smem + L.b_lo);
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + L.bar);
    uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + L.tslot);

    const int tiles = (t.Q + kPvM - 1) / kPvM;
    const int64_t bh = blockIdx.x / tiles;
    const int i0 = (blockIdx.x % tiles) * kPvM;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (warp == 0) tmem_alloc(tslot, kPvTmemCols);
    if (threadIdx.x == 0) {
        mbar_init(bar, 1u);
        fence_mbar_init();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tslot;

    const uint32_t idesc = idesc_tf32(kPvM, Np);
    const uint32_t lbo_a = (kPvM / 8) * 128;
    const uint32_t lbo_b = static_cast<uint32_t>(Np / 8) * 128;
    const uint32_t sbo = 128;
    const bool p_vec = (t.p_stride % 4 == 0) &&
                       (reinterpret_cast<uintptr_t>(t.p) % 16 == 0);
    const float* vg = t.v + bh * static_cast<int64_t>(t.K) * t.D;
    const int nchunk = (t.K + kPvKc - 1) / kPvKc;
    bool ok = true;
    for (int kc = 0; kc < nchunk; ++kc) {
        const int k0 = kc * kPvKc;
        // A = P[i0 .. i0 + 127][k0 .. k0 + kPvKc - 1].  Warp w stages rows
        // 32 w .. 32 w + 31: in each of its steps, lane l takes row
        // 8 rb + l % 8 of the warp's rows and item group 4 gb + l / 8 (16
        // bytes), so a warp's load covers 8 rows x 64 bytes and its store
        // four whole core matrices.  All of a thread's loads are issued
        // before any is used.
        constexpr int kSteps = 4 * (kPvKc / 16);
        constexpr int kGb = kPvKc / 16;
        {
            float4 v[kSteps];
#pragma unroll
            for (int st = 0; st < kSteps; ++st) {
                const int rb = st / kGb, gb = st % kGb;
                const int r = warp * 32 + rb * 8 + (lane & 7);
                const int g = gb * 4 + (lane >> 3);
                const int row = i0 + r, j = k0 + 4 * g;
                v[st] = make_float4(0.f, 0.f, 0.f, 0.f);
                if (row < t.Q) {
                    const float* src = t.p + (bh * t.Q + row) * t.p_stride + j;
                    if (p_vec && j + 3 < t.K) {
                        v[st] = __ldcs(reinterpret_cast<const float4*>(src));
                    } else {
                        if (j + 0 < t.K) v[st].x = src[0];
                        if (j + 1 < t.K) v[st].y = src[1];
                        if (j + 2 < t.K) v[st].z = src[2];
                        if (j + 3 < t.K) v[st].w = src[3];
                    }
                }
            }
#pragma unroll
            for (int st = 0; st < kSteps; ++st) {
                const int rb = st / kGb, gb = st % kGb;
                const int r = warp * 32 + rb * 8 + (lane & 7);
                const int g = gb * 4 + (lane >> 3);
                const float4 hi = make_float4(to_tf32(v[st].x), to_tf32(v[st].y),
                                              to_tf32(v[st].z), to_tf32(v[st].w));
                const float4 lo = make_float4(
                    to_tf32(v[st].x - hi.x), to_tf32(v[st].y - hi.y),
                    to_tf32(v[st].z - hi.z), to_tf32(v[st].w - hi.w));
                const int off = (g * (kPvM / 8) + (r >> 3)) * 32 + (r & 7) * 4;
                *reinterpret_cast<float4*>(a_hi + off) = hi;
                *reinterpret_cast<float4*>(a_lo + off) = lo;
            }
        }
        // B: row n of the N x K operand is column n of V.  A thread takes
        // four consecutive columns 4 n4 .. 4 n4 + 3 and an item group g:
        // four 16-byte loads of V rows k0 + 4 g .. + 3 (consecutive threads,
        // consecutive columns), transposed in registers into the four
        // columns' 16-byte core-matrix rows.
        for (int e = threadIdx.x; e < (Np / 4) * (kPvKc / 4); e += kPvThreads) {
            const int n4 = e % (Np / 4), g = e / (Np / 4);
            float w[4][4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int k = k0 + 4 * g + i;
                float4 row = make_float4(0.f, 0.f, 0.f, 0.f);
                if (k < t.K && 4 * n4 < t.D)
                    row = __ldg(reinterpret_cast<const float4*>(
                        vg + static_cast<int64_t>(k) * t.D + 4 * n4));
                w[i][0] = row.x;
                w[i][1] = row.y;
                w[i][2] = row.z;
                w[i][3] = row.w;
            }
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int n = 4 * n4 + c;
                const float4 hi = make_float4(to_tf32(w[0][c]), to_tf32(w[1][c]),
                                              to_tf32(w[2][c]), to_tf32(w[3][c]));
                const float4 lo = make_float4(
                    to_tf32(w[0][c] - hi.x), to_tf32(w[1][c] - hi.y),
                    to_tf32(w[2][c] - hi.z), to_tf32(w[3][c] - hi.w));
                const int off = (g * (Np / 8) + (n >> 3)) * 32 + (n & 7) * 4;
                *reinterpret_cast<float4*>(b_hi + off) = hi;
                *reinterpret_cast<float4*>(b_lo + off) = lo;
            }
        }
        fence_proxy_async_smem();
        __syncthreads();
        if (threadIdx.x == 0) {
            tc_fence_after_sync();
            const uint32_t ah0 = smem_addr(a_hi), al0 = smem_addr(a_lo);
            const uint32_t bh0 = smem_addr(b_hi), bl0 = smem_addr(b_lo);
            for (int ks = 0; ks < kPvKc / 8; ++ks) {
                const uint32_t ao = 2u * ks * lbo_a, bo = 2u * ks * lbo_b;
                const uint64_t da_hi = smem_desc(ah0 + ao, lbo_a, sbo);
                const uint64_t da_lo = smem_desc(al0 + ao, lbo_a, sbo);
                const uint64_t db_hi = smem_desc(bh0 + bo, lbo_b, sbo);
                const uint64_t db_lo = smem_desc(bl0 + bo, lbo_b, sbo);
                mma_tf32(tmem, da_hi, db_hi, idesc, kc > 0 || ks > 0);
                mma_tf32(tmem, da_hi, db_lo, idesc, true);
                mma_tf32(tmem, da_lo, db_hi, idesc, true);
            }
            mma_commit(bar);
        }
        // The MMAs have read this chunk (and written the accumulator) once
        // the mbarrier's phase completes; only then may the next chunk
        // overwrite the operands.
        bool landed = mbar_wait<false>(bar, static_cast<uint32_t>(kc & 1),
                                       t.wait_limit_cycles);
        if (!landed) {
            // Give the MMAs in flight a second bounded wait before the
            // tensor memory is freed below.
            mbar_wait<false>(bar, static_cast<uint32_t>(kc & 1), t.wait_limit_cycles);
        }
        ok = __syncthreads_and(landed);   // the same decision in every thread
        if (!ok) break;
    }
    tc_fence_after_sync();
    if (ok) {
        const int r = warp * 32 + lane;
        const int row = i0 + r;
        float* og = t.out + (bh * t.Q + row) * static_cast<int64_t>(t.D);
        for (int c0 = 0; c0 < Np; c0 += 16) {
            float v[16];
            tmem_ld16(tmem + (static_cast<uint32_t>(warp * 32) << 16) +
                          static_cast<uint32_t>(c0), v);
            if (row < t.Q) {
#pragma unroll
                for (int i = 0; i < 16; i += 4) {
                    if (c0 + i < t.D)
                        __stcs(reinterpret_cast<float4*>(og + c0 + i),
                               make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]));
                }
            }
        }
    }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, kPvTmemCols);
    if (!ok && threadIdx.x == 0) raise_error(t.err, kBitTimeout);
}

}  // namespace

cudaError_t launch_bienc_pv(const PvTask& task, cudaStream_t stream) {
    const int Np = pv_np(task.D);
    const int smem = static_cast<int>(pv_smem_bytes(Np));
    cudaError_t e = ensure_smem_attribute(reinterpret_cast<const void*>(bienc_pv_kernel),
                                          27, smem, false);
    if (e != cudaSuccess) return e;
    const int64_t tiles = (task.Q + kPvM - 1) / kPvM;
    const int64_t grid = static_cast<int64_t>(task.BH) * tiles;
    bienc_pv_kernel<<<static_cast<unsigned>(grid), kPvThreads, smem, stream>>>(task);
    return cudaGetLastError();
}

}  // namespace cs
