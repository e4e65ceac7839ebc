// Step 3 of biencoder_attention ("BURT-IMMA CUDA Kernel API Reference",
// section 2.5 Description step 3, out = attn @ context_values) on the
// 5th-generation tensor cores, as a second kernel after the fused scores
// and search kernel (k_bienc.cu) has written the weights P [bh, Q, K].
//
// A tile is (bh, 128 query rows): out[128 x D] = P[128 x K] . V[K x D], a
// tcgen05.mma of kind::tf32 with M = 128, N = D rounded up to 16, K in
// steps of 8, the fp32 accumulator in tensor memory.  fp32 accuracy comes
// from three TF32 products per fp32 product: with x_hi the TF32 nearest x
// and x_lo the TF32 nearest x - x_hi,
//   P V ~ P_hi V_hi + P_hi V_lo + P_lo V_hi,
// which leaves out only P_lo V_lo and the two lo roundings (about 2^-21 of
// |P||V| each), next to the fp32 accumulation's own rounding.
//
// Operands: P's halves in the MMA's 128-byte swizzled K-major layout
// (chunks of 32 items: 128 rows of 128 bytes, each 8-row atom's 16-byte
// units permuted by the row index mod 8, as the tensor-memory-access unit
// writes a box of 32 x 128 fp32 with 128-byte swizzling); V^T's in the
// canonical layout without swizzle (8-row x 16-byte core matrices, core
// (row group m, item group g) at (g * rows / 8 + m) * 128 bytes).  The
// context (at most d_head <= 64 items) is staged whole.
//
// Persistent CTAs (one per SM at most) take contiguous runs of tiles, so V
// changes rarely, and split the work between warp roles that hand tiles on
// through mbarriers:
//   loader (warp 13)        once the MMAs that read a stage last have
//                           completed, copies the next tile's P into its hi
//                           half: one 2-D tensor copy per 32-item chunk
//                           (items past K and rows past the tensor come in
//                           as zeros);
//   producers (warps 0-7)   split the landed tile in place into its hi half
//                           and, at the same offsets, its lo half; stage
//                           V^T (hi, lo) when bh changes; mark the stage
//                           full.  (Rows that are not 16-byte aligned are
//                           loaded by the producers element by element.)
//   MMA issuer (warp 12)    waits for a full stage and a free accumulator
//                           (two in tensor memory), issues the 3 x Kp / 8
//                           MMAs from one thread and commits them to the
//                           stage's empty barrier and the accumulator's
//                           full barrier;
//   epilogue (warps 8-11)   reads rows 32 (w % 4) .. + 31 of the
//                           accumulator (warp w's quarter of the
//                           tensor-memory lanes) into a shared output tile,
//                           frees the accumulator, and writes the tile's
//                           rows (contiguous in the output) with coalesced
//                           16-byte stores.
// So a tile's copies, split, MMAs and stores overlap those of its
// neighbours.  Every wait is bounded; after a timeout the CTA records it,
// raises a shared abort flag, and every role skips its remaining waits and
// work.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <string.h>

#include "cs_tcgen05.cuh"

namespace cs {
namespace {

using namespace csd;

constexpr int kPvProducers = 256;                  // warps 0-7
constexpr int kPvEpilogue = 128;                   // warps 8-11
constexpr int kPvMmaWarp = 12;
constexpr int kPvLoadWarp = 13;
constexpr int kPvThreads = kPvProducers + kPvEpilogue + 64;
constexpr uint32_t kBarProducers = 1;              // named barrier ids
constexpr uint32_t kBarEpilogue = 2;
constexpr int kChunkBytes = kPvM * 128;            // one 32-item chunk

__global__ void __launch_bounds__(kPvThreads, 1)
bienc_pv_kernel(PvTask t, const __grid_constant__ CUtensorMap tmap, int use_tma) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    // The swizzled operands need 1024-byte aligned atoms: the layout starts
    // at the first such boundary (the allocation has that much slack).
    unsigned char* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    const int Kp = pv_kp(t.K);
    const int Np = pv_np(t.D);
    const int nchunk = pv_chunks(t.K);
    const PvSmemLayout L = pv_smem_layout(t.K, Np, t.D);
    float* b_hi = reinterpret_cast<float*>(smem + L.b_hi);
    float* b_lo = reinterpret_cast<float*>(smem + L.b_lo);
    float* stage = reinterpret_cast<float*>(smem + L.stage);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L.bar);
    uint64_t* full = bars;          // [2] stage s holds a tile's split P (and V^T)
    uint64_t* empty = bars + 2;     // [2] the MMAs that read stage s completed
    uint64_t* acc_full = bars + 4;  // [2] accumulator a holds a tile's result
    uint64_t* acc_empty = bars + 6; // [2] the epilogue has read accumulator a
    uint64_t* landed = bars + 8;    // [2] stage s's hi half holds the raw P
    volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + L.flag);
    uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + L.tslot);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int tiles_per_bh = (t.Q + kPvM - 1) / kPvM;
    const int64_t tiles = static_cast<int64_t>(t.BH) * tiles_per_bh;
    const int64_t j0 = tiles * blockIdx.x / gridDim.x;
    const int nt = static_cast<int>(tiles * (blockIdx.x + 1) / gridDim.x - j0);
    const int G4 = Kp >> 2;   // item groups of four (V^T)

    if (threadIdx.x == 0) {
        for (int s = 0; s < 2; ++s) {
            mbar_init(&full[s], kPvProducers);
            mbar_init(&empty[s], 1u);
            mbar_init(&acc_full[s], 1u);
            mbar_init(&acc_empty[s], kPvEpilogue);
            mbar_init(&landed[s], 1u);
        }
        *abort_flag = 0u;
        fence_mbar_init();
    }
    if (warp == kPvMmaWarp) tmem_alloc(tslot, kPvTmemCols);
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tslot;

    // A bounded wait taken by every thread of a role, with one outcome for
    // all of them (a named-barrier AND among the role's `count` threads, or
    // the warp's vote), so that the role's control flow stays uniform and
    // its barriers stay matched; it gives up at once after an abort, and
    // raises the abort when it times out.
    auto wait = [&](uint64_t* b, int phase, uint32_t bar_id, uint32_t count) -> bool {
        bool ok = *abort_flag == 0u &&
                  mbar_wait<false>(b, static_cast<uint32_t>(phase & 1), t.wait_limit_cycles);
        ok = bar_id ? named_barrier_and(bar_id, count, ok)
                    : __all_sync(0xffffffffu, ok);
        if (!ok) *abort_flag = 1u;
        return ok;
    };
    auto tile_rows = [&](int64_t j, int64_t& bh, int& i0) {
        bh = j / tiles_per_bh;
        i0 = static_cast<int>(j - bh * tiles_per_bh) * kPvM;
        return min(kPvM, t.Q - i0);
    };
    auto a_hi_of = [&](int st) { return smem + 2 * st * L.a_half; };
    auto a_lo_of = [&](int st) { return smem + (2 * st + 1) * L.a_half; };

    if (warp < kPvProducers / 32) {
        // ------------------------------------------------------ producers
        const int pt = threadIdx.x;   // 0 .. 255
        int64_t bh_staged = -1;
        for (int i = 0; i < nt; ++i) {
            const int st = i & 1;
            int64_t bh;
            int i0;
            const int nrows = tile_rows(j0 + i, bh, i0);
            float* a_hi = reinterpret_cast<float*>(a_hi_of(st));
            float* a_lo = reinterpret_cast<float*>(a_lo_of(st));

            if (use_tma) {
                if (!wait(&landed[st], i >> 1, kBarProducers, kPvProducers)) break;
            } else {
                // Element loads into the swizzled positions (the stage was
                // last read by the MMAs of tile i - 2): item k of row r at
                // chunk k / 32, 16-byte unit (k % 32 / 4) ^ (r % 8).
                if (i > 1 && !wait(&empty[st], (i - 2) >> 1, kBarProducers, kPvProducers))
                    break;
                const float* prow0 = t.p + (bh * t.Q + i0) * t.p_stride;
                const int kw = 32 * nchunk;
                for (int e = pt; e < kPvM * kw; e += kPvProducers) {
                    const int r = e / kw, k = e - r * kw;
                    const float x = (r < nrows && k < t.K) ? prow0[r * t.p_stride + k] : 0.0f;
                    a_hi[(k >> 5) * (kChunkBytes / 4) + r * 32 +
                         ((((k & 31) >> 2) ^ (r & 7)) << 2) + (k & 3)] = x;
                }
                named_barrier(kBarProducers, kPvProducers);
            }

            // V^T of a new bh, once the MMAs that read the old one (tile
            // i - 1's) have completed.  A thread takes four consecutive
            // columns 4 n4 .. + 3 and an item group g: four 16-byte loads of
            // V rows 4 g .. + 3, transposed in registers into the four
            // columns' 16-byte core-matrix rows, hi and lo.
            if (bh != bh_staged) {
                if (i > 0 && !wait(&empty[(i - 1) & 1], (i - 1) >> 1, kBarProducers,
                                   kPvProducers))
                    break;
                bh_staged = bh;
                const float* vg = t.v + bh * static_cast<int64_t>(t.K) * t.D;
                for (int e = pt; e < (Np / 4) * G4; e += kPvProducers) {
                    const int n4 = e % (Np / 4), g = e / (Np / 4);
                    float w[4][4];
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        const int k = 4 * g + r;
                        float4 row = make_float4(0.f, 0.f, 0.f, 0.f);
                        if (k < t.K && 4 * n4 < t.D)
                            row = __ldg(reinterpret_cast<const float4*>(
                                vg + static_cast<int64_t>(k) * t.D + 4 * n4));
                        w[r][0] = row.x;
                        w[r][1] = row.y;
                        w[r][2] = row.z;
                        w[r][3] = row.w;
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
            }

            // Split in place, 16-byte unit by unit (the layout is the same
            // for both halves); then the stage is full.
#pragma unroll 4
            for (int e = pt; e < L.a_half / 16; e += kPvProducers) {
                const float4 x = reinterpret_cast<const float4*>(a_hi)[e];
                const float4 hi = make_float4(to_tf32(x.x), to_tf32(x.y), to_tf32(x.z),
                                              to_tf32(x.w));
                const float4 lo = make_float4(to_tf32(x.x - hi.x), to_tf32(x.y - hi.y),
                                              to_tf32(x.z - hi.z), to_tf32(x.w - hi.w));
                reinterpret_cast<float4*>(a_hi)[e] = hi;
                reinterpret_cast<float4*>(a_lo)[e] = lo;
            }
            fence_proxy_async_smem();
            mbar_arrive(&full[st]);
        }
    } else if (warp < (kPvProducers + kPvEpilogue) / 32) {
        // ------------------------------------------------------- epilogue
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;
        const int SD = t.D + 4;   // output tile row stride (floats)
        const int et = threadIdx.x - kPvProducers;   // 0 .. 127
        for (int i = 0; i < nt; ++i) {
            const int acc = i & 1;
            int64_t bh;
            int i0;
            const int nrows = tile_rows(j0 + i, bh, i0);
            if (!wait(&acc_full[acc], i >> 1, kBarEpilogue, kPvEpilogue)) break;
            tc_fence_after_sync();
            // Row r of the accumulator into row r of the output tile, 16
            // columns at a time (rows SD apart: the eight rows of a
            // quarter-warp's 16-byte stores fall in different banks).
            const uint32_t tbase = tmem + (static_cast<uint32_t>(quarter * 32) << 16) +
                                   static_cast<uint32_t>(acc * 64);
            for (int c0 = 0; c0 < Np; c0 += 16) {
                float part[16];
                tmem_ld16(tbase + static_cast<uint32_t>(c0), part);
#pragma unroll
                for (int c = 0; c < 16; c += 4)
                    if (c0 + c < t.D)
                        *reinterpret_cast<float4*>(stage + r * SD + c0 + c) =
                            make_float4(part[c], part[c + 1], part[c + 2], part[c + 3]);
            }
            tc_fence_before_sync();
            mbar_arrive(&acc_empty[acc]);
            named_barrier(kBarEpilogue, kPvEpilogue);
            // The tile's rows are contiguous in the output: thread et stores
            // 16-byte unit et % 16 of rows et / 16, et / 16 + 8, ... (a warp
            // two whole rows at D = 64).
            const int u = et & 15;
            if (u < (t.D >> 2)) {
                float* og = t.out + (bh * t.Q + i0) * static_cast<int64_t>(t.D) + 4 * u;
#pragma unroll 4
                for (int rr = et >> 4; rr < nrows; rr += kPvEpilogue / 16)
                    __stcs(reinterpret_cast<float4*>(og + rr * t.D),
                           *reinterpret_cast<const float4*>(stage + rr * SD + 4 * u));
            }
            // The output tile is rewritten only after every epilogue thread
            // has read it.
            named_barrier(kBarEpilogue, kPvEpilogue);
        }
    } else if (warp == kPvMmaWarp) {
        // ---------------------------------------------------- MMA issuer
        const uint32_t idesc = idesc_tf32(kPvM, Np);
        const uint32_t lbo_b = static_cast<uint32_t>(Np / 8) * 128;
        const uint32_t bh0 = smem_addr(b_hi), bl0 = smem_addr(b_lo);
        for (int i = 0; i < nt; ++i) {
            const int st = i & 1, acc = i & 1;
            if (!wait(&full[st], i >> 1, 0u, 32u)) break;
            if (i >= 2 && !wait(&acc_empty[acc], (i >> 1) - 1, 0u, 32u)) break;
            tc_fence_after_sync();
            if (lane == 0) {
                const uint32_t ah0 = smem_addr(a_hi_of(st));
                const uint32_t al0 = smem_addr(a_lo_of(st));
                const uint32_t d = tmem + static_cast<uint32_t>(acc * 64);
                for (int ks = 0; ks < Kp / 8; ++ks) {
                    // A: chunk ks / 4, 32 bytes (8 tf32) per step along the
                    // atom's rows; B: two core matrices per step.
                    const uint32_t ao = (ks >> 2) * kChunkBytes + (ks & 3) * 32;
                    const uint32_t bo = 2u * ks * lbo_b;
                    const uint64_t da_hi = smem_desc_sw128(ah0 + ao, 1024);
                    const uint64_t da_lo = smem_desc_sw128(al0 + ao, 1024);
                    const uint64_t db_hi = smem_desc(bh0 + bo, lbo_b, 128);
                    const uint64_t db_lo = smem_desc(bl0 + bo, lbo_b, 128);
                    mma_tf32(d, da_hi, db_hi, idesc, ks > 0);
                    mma_tf32(d, da_hi, db_lo, idesc, true);
                    mma_tf32(d, da_lo, db_hi, idesc, true);
                }
                mma_commit(&empty[st]);
                mma_commit(&acc_full[acc]);
            }
            __syncwarp();
        }
        // Before the tensor memory is freed, the last MMAs must be done: the
        // epilogue waited for them, unless the CTA aborted; then give them a
        // bounded wait of their own.
        if (*abort_flag && nt > 0) {
            const int last = nt - 1;
            mbar_wait<false>(&acc_full[last & 1], static_cast<uint32_t>((last >> 1) & 1),
                             t.wait_limit_cycles);
        }
    } else if (warp == kPvLoadWarp && use_tma) {
        // --------------------------------------------------------- loader
        int issued = 0;
        for (int i = 0; i < nt; ++i) {
            const int st = i & 1;
            // The stage was last read by the MMAs of tile i - 2.
            if (i > 1 && !wait(&empty[st], (i - 2) >> 1, 0u, 32u)) break;
            int64_t bh;
            int i0;
            tile_rows(j0 + i, bh, i0);
            if (lane == 0) {
                mbar_arrive_expect_tx(&landed[st], static_cast<uint32_t>(L.a_half));
                const int row = static_cast<int>(bh * t.Q + i0);
                for (int c = 0; c < nchunk; ++c)
                    tma_load_2d(a_hi_of(st) + c * kChunkBytes, &tmap, 32 * c, row,
                                &landed[st]);
            }
            ++issued;
            __syncwarp();
        }
        // After an abort a tile's copies may still be in flight: none may
        // land in shared memory after the CTA exits (bounded waits).
        if (*abort_flag) {
            for (int i = (issued > 2 ? issued - 2 : 0); i < issued; ++i)
                mbar_wait<false>(&landed[i & 1], static_cast<uint32_t>((i >> 1) & 1),
                                 t.wait_limit_cycles);
        }
    }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == kPvMmaWarp) tmem_dealloc(tmem, kPvTmemCols);
    if (*abort_flag && threadIdx.x == 0) raise_error(t.err, kBitTimeout);
}

// cuTensorMapEncodeTiled, from the CUDA driver through the runtime (no link
// against the driver library); null if unavailable.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess) {
            cudaGetLastError();
            p = nullptr;
        }
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }();
    return fn;
}

}  // namespace

cudaError_t launch_bienc_pv(const PvTask& task, int sm_count,
                            cudaStream_t stream) {
    const int smem = static_cast<int>(pv_smem_bytes(task.K, task.D));
    cudaError_t e = ensure_smem_attribute(reinterpret_cast<const void*>(bienc_pv_kernel),
                                          27, smem, false);
    if (e != cudaSuccess) return e;
    const int64_t tiles = static_cast<int64_t>(task.BH) * ((task.Q + kPvM - 1) / kPvM);
    const int64_t grid = tiles < sm_count ? tiles : sm_count;
    // P as a 2-D tensor [BH Q rows, K items], rows p_stride floats apart,
    // copied in boxes of 32 items x 128 rows with 128-byte swizzling: needs
    // a 16-byte aligned base and row stride.
    CUtensorMap tmap;
    memset(&tmap, 0, sizeof(tmap));
    int use_tma = 0;
    const int64_t rows = static_cast<int64_t>(task.BH) * task.Q;
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (enc && task.p_stride % 4 == 0 && reinterpret_cast<uintptr_t>(task.p) % 16 == 0 &&
        rows < (int64_t(1) << 31)) {
        const cuuint64_t gdim[2] = {static_cast<cuuint64_t>(task.K),
                                    static_cast<cuuint64_t>(rows)};
        const cuuint64_t gstride[1] = {static_cast<cuuint64_t>(task.p_stride) * 4};
        const cuuint32_t box[2] = {32, static_cast<cuuint32_t>(kPvM)};
        const cuuint32_t estride[2] = {1, 1};
        const CUresult r = enc(&tmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2,
                               const_cast<float*>(task.p), gdim, gstride, box, estride,
                               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                               CU_TENSOR_MAP_L2_PROMOTION_NONE,
                               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        use_tma = r == CUDA_SUCCESS ? 1 : 0;
    }
    bienc_pv_kernel<<<static_cast<unsigned>(grid), kPvThreads, smem, stream>>>(task, tmap,
                                                                                use_tma);
    return cudaGetLastError();
}

}  // namespace cs
