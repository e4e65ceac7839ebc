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
// The context (at most d_head <= 64 items) is staged whole:
//   - P by 16-byte asynchronous copies straight into that layout (a
//     16-byte unit of the layout is four consecutive items of one row, as
//     in memory; items past K and rows past Q are zero-filled), then split
//     in place into the hi half and, beside it, the lo half;
//   - V by 16-byte loads along d, transposed 4 x 4 in registers and split.
// After the MMAs, warps w and w + 4 read rows 32 (w % 4) .. + 31 of the
// accumulator (their quarter of the tensor-memory lanes) into a shared
// output tile over the spent operands, from which the CTA writes the
// tile's rows (contiguous in the output) with coalesced 16-byte stores.
#include "cs_tcgen05.cuh"

namespace cs {
namespace {

using namespace csd;

constexpr int kPvThreads = 256;   // two warpgroups

__global__ void __launch_bounds__(kPvThreads, 1)
bienc_pv_kernel(PvTask t) {
    extern __shared__ __align__(1024) unsigned char smem[];
    const int Kp = pv_kp(t.K);
    const int Np = pv_np(t.D);
    const PvSmemLayout L = pv_smem_layout(Kp, Np, t.D);
    float* a_hi = reinterpret_cast<float*>(smem + L.a_hi);
    float* a_lo = reinterpret_cast<float*>(smem + L.a_lo);
    float* b_hi = reinterpret_cast<float*>(smem + L.b_hi);
    float* b_lo = reinterpret_cast<float*>(smem + L.b_lo);
    float* stage = reinterpret_cast<float*>(smem + L.stage);
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + L.bar);
    uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + L.tslot);

    const int tiles = (t.Q + kPvM - 1) / kPvM;
    const int64_t bh = blockIdx.x / tiles;
    const int i0 = (blockIdx.x % tiles) * kPvM;
    const int nrows = min(kPvM, t.Q - i0);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int G4 = Kp >> 2;   // item groups of four

    // A = P[i0 .. i0 + 127][0 .. Kp - 1], raw fp32 into a_hi.  Thread t
    // copies item group g = t / 8 % 16 of rows 8 rb + t % 8, rb = t / 128,
    // t / 128 + 2, ..., so that a warp's copies read 8 rows x 64 contiguous
    // bytes and each quarter-warp fills one whole core matrix.
    const float* prow0 = t.p + (bh * t.Q + i0) * t.p_stride;
    const bool p_vec = (t.p_stride % 4 == 0) &&
                       (reinterpret_cast<uintptr_t>(t.p) % 16 == 0);
    if (p_vec) {
        const int r8 = threadIdx.x & 7, g = (threadIdx.x >> 3) & 15;
        if (g < G4) {
            const int kv = min(max(t.K - 4 * g, 0), 4);   // items present
#pragma unroll 4
            for (int rb = threadIdx.x >> 7; rb < kPvM / 8; rb += kPvThreads / kPvM) {
                const int r = rb * 8 + r8;
                const int valid = r < nrows ? kv : 0;
                const float* src = valid ? prow0 + r * t.p_stride + 4 * g : t.p;
                cp_async16_zfill(a_hi + (g * (kPvM / 8) + rb) * 32 + r8 * 4, src,
                                 static_cast<uint32_t>(valid * 4));
            }
        }
    } else {
        for (int e = threadIdx.x; e < kPvM * Kp; e += kPvThreads) {
            const int r = e / Kp, k = e - r * Kp;
            const float x = (r < nrows && k < t.K) ? prow0[r * t.p_stride + k] : 0.0f;
            a_hi[((k >> 2) * (kPvM / 8) + (r >> 3)) * 32 + (r & 7) * 4 + (k & 3)] = x;
        }
    }

    if (warp == 0) tmem_alloc(tslot, kPvTmemCols);
    if (threadIdx.x == 0) {
        mbar_init(bar, 1u);
        fence_mbar_init();
    }

    // B: row n of the N x K operand is column n of V.  A thread takes four
    // consecutive columns 4 n4 .. 4 n4 + 3 and an item group g: four 16-byte
    // loads of V rows 4 g .. + 3 (consecutive threads, consecutive columns),
    // transposed in registers into the four columns' 16-byte core-matrix
    // rows, hi and lo.
    const float* vg = t.v + bh * static_cast<int64_t>(t.K) * t.D;
    for (int e = threadIdx.x; e < (Np / 4) * G4; e += kPvThreads) {
        const int n4 = e % (Np / 4), g = e / (Np / 4);
        float w[4][4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int k = 4 * g + i;
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

    // P has landed (this thread's copies; after the barrier everyone's):
    // split it in place, 16-byte unit by unit.
    cp_async_wait_all();
    __syncthreads();
#pragma unroll 4
    for (int e = threadIdx.x; e < kPvM * G4; e += kPvThreads) {
        const float4 x = reinterpret_cast<const float4*>(a_hi)[e];
        const float4 hi = make_float4(to_tf32(x.x), to_tf32(x.y), to_tf32(x.z),
                                      to_tf32(x.w));
        const float4 lo = make_float4(to_tf32(x.x - hi.x), to_tf32(x.y - hi.y),
                                      to_tf32(x.z - hi.z), to_tf32(x.w - hi.w));
        reinterpret_cast<float4*>(a_hi)[e] = hi;
        reinterpret_cast<float4*>(a_lo)[e] = lo;
    }
    fence_proxy_async_smem();
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tslot;

    if (threadIdx.x == 0) {
        const uint32_t idesc = idesc_tf32(kPvM, Np);
        const uint32_t lbo_a = (kPvM / 8) * 128;
        const uint32_t lbo_b = static_cast<uint32_t>(Np / 8) * 128;
        const uint32_t sbo = 128;
        const uint32_t ah0 = smem_addr(a_hi), al0 = smem_addr(a_lo);
        const uint32_t bh0 = smem_addr(b_hi), bl0 = smem_addr(b_lo);
        for (int ks = 0; ks < Kp / 8; ++ks) {
            const uint32_t ao = 2u * ks * lbo_a, bo = 2u * ks * lbo_b;
            const uint64_t da_hi = smem_desc(ah0 + ao, lbo_a, sbo);
            const uint64_t da_lo = smem_desc(al0 + ao, lbo_a, sbo);
            const uint64_t db_hi = smem_desc(bh0 + bo, lbo_b, sbo);
            const uint64_t db_lo = smem_desc(bl0 + bo, lbo_b, sbo);
            mma_tf32(tmem, da_hi, db_hi, idesc, ks > 0);
            mma_tf32(tmem, da_hi, db_lo, idesc, true);
            mma_tf32(tmem, da_lo, db_hi, idesc, true);
        }
        mma_commit(bar);
    }
    // The MMAs have read the operands and written the accumulator once the
    // mbarrier's phase completes.
    bool landed = mbar_wait<false>(bar, 0u, t.wait_limit_cycles);
    if (!landed) {
        // Give the MMAs in flight a second bounded wait before the shared
        // memory is overwritten and the tensor memory freed below.
        mbar_wait<false>(bar, 0u, t.wait_limit_cycles);
    }
    const bool ok = __syncthreads_and(landed);   // the same in every thread
    tc_fence_after_sync();
    const int SD = t.D + 4;   // output tile row stride (floats)
    if (ok) {
        // Row r of the accumulator into row r of the output tile, 16
        // columns at a time, warps w and w + 4 taking alternate column
        // chunks of their quarter of the lanes (rows SD apart: the eight rows
        // of a quarter-warp's 16-byte stores fall in different banks).
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;
        for (int c0 = 16 * (warp >> 2); c0 < Np; c0 += 32) {
            float part[16];
            tmem_ld16(tmem + (static_cast<uint32_t>(quarter * 32) << 16) +
                          static_cast<uint32_t>(c0), part);
#pragma unroll
            for (int i = 0; i < 16; i += 4)
                if (c0 + i < t.D)
                    *reinterpret_cast<float4*>(stage + r * SD + c0 + i) =
                        make_float4(part[i], part[i + 1], part[i + 2], part[i + 3]);
        }
    }
    tc_fence_before_sync();
    __syncthreads();
    if (ok) {
        // The tile's rows are contiguous in the output: thread t stores
        // 16-byte unit t % 16 of rows t / 16, t / 16 + 16, ... (a warp two
        // whole rows at D = 64).
        const int u = threadIdx.x & 15;
        if (u < (t.D >> 2)) {
            float* og = t.out + (bh * t.Q + i0) * static_cast<int64_t>(t.D) + 4 * u;
#pragma unroll 4
            for (int r = threadIdx.x >> 4; r < nrows; r += kPvThreads / 16)
                __stcs(reinterpret_cast<float4*>(og + r * t.D),
                       *reinterpret_cast<const float4*>(stage + r * SD + 4 * u));
        }
    }
    if (warp == 0) tmem_dealloc(tmem, kPvTmemCols);
    if (!ok && threadIdx.x == 0) raise_error(t.err, kBitTimeout);
}

}  // namespace

cudaError_t launch_bienc_pv(const PvTask& task, cudaStream_t stream) {
    const int smem = static_cast<int>(pv_smem_bytes(task.K, task.D));
    cudaError_t e = ensure_smem_attribute(reinterpret_cast<const void*>(bienc_pv_kernel),
                                          27, smem, false);
    if (e != cudaSuccess) return e;
    const int64_t tiles = (task.Q + kPvM - 1) / kPvM;
    const int64_t grid = static_cast<int64_t>(task.BH) * tiles;
    bienc_pv_kernel<<<static_cast<unsigned>(grid), kPvThreads, smem, stream>>>(task);
    return cudaGetLastError();
}

}  // namespace cs
