// Internal interface between the C ABI (cs_api.cu) and the kernel
// translation units.  Not installed; the public API is
// include/entropy_bounded_softmax.h.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "entropy_bounded_softmax.h"

namespace cs {

// Bits of the device error word.
constexpr unsigned int kBitNan = 1u << CS_ERR_NAN_INPUT;
constexpr unsigned int kBitInf = 1u << CS_ERR_INF_INPUT;
constexpr unsigned int kBitOverflow = 1u << CS_ERR_ENTROPY_OVERFLOW;
constexpr unsigned int kBitTimeout = 1u << CS_ERR_TIMEOUT;

// Default limit of every bounded device wait, in SM cycles: 2^31 cycles,
// about 1 s at GB300's 2.07 GHz maximum clock.
constexpr uint64_t kWaitLimitCycles = 1ull << 31;

// One launch's worth of work: every row of the matrix with the same
// parameters (the arguments of section 2.1's signature plus t_out and the
// error word).
struct RowTask {
    const void* logits;    // fp32, or bf16 bit patterns when in_bf16
    float* out;
    float* t_out;          // may be null
    unsigned int* err;     // device error word
    int64_t batch;
    int32_t num_classes;
    int32_t max_iter;
    float entropy_bound;
    float t_min;
    float hi0;             // min(1, t_max): upper end of the search
    int32_t strict;        // 1: evaluate every bisection midpoint
    int32_t async_stage;   // cluster kernel: stage with asynchronous copies
    uint64_t wait_limit_cycles;
    int32_t* evals_out;    // may be null: temperatures evaluated per row
    int32_t in_bf16;       // 1: logits are bf16 (promoted exactly to fp32)
    float fan_beta0;       // cluster kernel: the fan's first inverse
                           // temperature (the others 4 and 16 times it),
                           // evaluated with T = 1; 0: no fan
};

// Cluster kernel geometry.
constexpr int kMaxCluster = 16;
// Temperatures the cluster kernel evaluates with T = 1 in few-row launches
// (the fan: beta0, 4 beta0, 16 beta0, so that one exponential and two
// squarings give all three), and the threads an SM the fan instantiations
// keep registers for (__launch_bounds__(256, 2)).
constexpr int kFanPoints = 3;
constexpr int kFanThreadsPerSm = 512;
constexpr int kClusterMaxThreads = 512;
constexpr int kSlotVals = 12;         // floats per exchange slot (48 bytes)

// Byte offsets of the cluster kernel's dynamic shared memory for `warps`
// warps and cluster size n: the exchange slots [2][n * warps][kSlotVals]
// floats (one per warp of the cluster, double-buffered), the two exchange
// mbarriers, then (128-byte aligned) the slice.
struct ClusterSmemLayout {
    int cslot, cbar, row;
};

__host__ __device__ inline ClusterSmemLayout cluster_smem_layout(int warps,
                                                                 int n) {
    ClusterSmemLayout L;
    int p = 0;
    L.cslot = p;
    p += 2 * n * warps * kSlotVals * 4;
    p = ((p + 7) / 8) * 8;
    L.cbar = p;
    p += 2 * 8;
    L.row = ((p + 127) / 128) * 128;
    return L;
}

// Dynamic shared memory of the cluster kernel for a slice of `slice_len`
// classes, `threads` threads and cluster size `n`.
inline int64_t cluster_smem_bytes(int64_t slice_len, int threads, int n) {
    const ClusterSmemLayout L = cluster_smem_layout(threads / 32, n);
    const int64_t row = ((slice_len + 8 + 3) / 4) * 16;  // pad + tail room
    return L.row + row;
}

// Classes per CTA the automatic plan aims for: 64 KB slices, so that
// three CTAs share an SM and one's exchange overlaps the others' passes.
constexpr int64_t kTargetSlice = 16384;

// Automatic threads per CTA: about 40 classes per thread for a launch with
// about one CTA per SM (up to a quarter more CTAs than SMs; all of a CTA's
// time goes to one row), about 72 for larger launches (several CTAs share
// an SM), rounded up to whole pairs of warps; 128-256 threads either way
// (64-256 for many one-CTA rows), where the per-round reductions stay
// short.
inline int cluster_threads_for(int64_t slice_len, int64_t ctas,
                               int64_t sm_count, int n) {
    const bool many = ctas * 4 > sm_count * 5;
    const int64_t per = many ? 72 : 40;
    int64_t t = (slice_len + per - 1) / per;
    // An even number of warps: the sweep's 16000-class slices ran 2.5-3%
    // faster on 192 or 256 threads than on 224 (six sweep points), and 160
    // was between.
    t = ((t + 63) / 64) * 64;
    // At least 128 threads, or 64 for many one-CTA rows: 4096 rows of
    // 1500-4000 classes ran 20-28% faster in 64-thread CTAs than in
    // 128-thread ones (fewer warps wait at every exchange of a short row).
    const int64_t lo = (many && n == 1) ? 64 : 128;
    if (t < lo) t = lo;
    if (t > 256) t = 256;
    return static_cast<int>(t);
}

// One backward launch: grad_in = (1/T) p (g - <g, p>) for every row.
struct BwdTask {
    const float* probs;     // [batch, C] the forward's output p
    const float* grad_out;  // [batch, C] upstream gradient g
    const float* t;         // [batch] the forward's temperatures
    float* grad_in;         // [batch, C]
    int64_t batch;
    int32_t num_classes;
};

// Backward geometry.  Row-group CTAs of 256 threads; cluster CTAs of up to
// 512 threads whose dynamic shared memory is a 512-byte header (the
// exchange slots) followed by the slice of p and, when STAGE_G, of g.
constexpr int kBwdGroupThreads = 256;
constexpr int kBwdMaxThreads = 512;
constexpr int kBwdSmemHeader = 512;
// Classes per CTA the automatic backward plan aims for: 64 KB of p and g,
// so that three CTAs share an SM and one's reduction overlaps the others'
// loads and stores.
constexpr int64_t kBwdTargetSlice = 8192;

inline int64_t backward_smem_bytes(int64_t slice_len, bool stage_g) {
    return kBwdSmemHeader + (slice_len / 4 + 1) * 16 * (stage_g ? 2 : 1);
}

cudaError_t launch_backward_rowgroup(const BwdTask& task, int lanes_per_row,
                                     int elems_per_lane, cudaStream_t stream);
cudaError_t launch_backward_cluster(const BwdTask& task, int cluster_size,
                                    int slice_len, int threads, int smem_bytes,
                                    bool stage_g, int64_t grid_ctas,
                                    cudaStream_t stream);

// One attention_softmax launch: rows = B H S rows of S scores.
struct AttnTask {
    const float* scores;   // [B, H, S, S]
    float* out;            // [B, H, S, S]
    const float* mask;     // [B, S] or null
    unsigned int* err;     // device error word
    int64_t rows;          // B H S
    int32_t heads;
    int32_t seq_len;
    int32_t causal;
};

// attention_softmax geometry: row-group CTAs of 256 threads; row-CTA
// kernel of up to 512 threads with a 512-byte header (reduction slots)
// before the row in shared memory.
constexpr int kAttnGroupThreads = 256;
constexpr int kAttnMaxThreads = 512;
constexpr int kAttnSmemHeader = 512;

inline int64_t attention_smem_bytes(int64_t seq_len) {
    return kAttnSmemHeader + ((seq_len + 6) / 4 + 1) * 16;
}

cudaError_t launch_attention_rowgroup(const AttnTask& task, int lanes_per_row,
                                      int elems_per_lane, cudaStream_t stream);
cudaError_t launch_attention_cta(const AttnTask& task, int threads,
                                 int smem_bytes, int64_t grid_ctas,
                                 cudaStream_t stream);

// One biencoder_attention launch: BH = batch x heads pairs of query
// [Q, D], keys and values [K, D].
struct BiencTask {
    const float* q;
    const float* k;
    const float* v;
    float* out;            // [BH, Q, D]
    float* attn_out;       // [BH, Q, K] or null
    float* t_out;          // [BH, Q] or null
    unsigned int* err;     // device error word
    int32_t BH;
    int32_t Q;
    int32_t K;
    int32_t D;
    float scale;
    float entropy_bound;
    float t_min;
    float hi0;             // min(1, t_max)
    int32_t max_iter;
    float* p_out;          // non-null: steps 1-2 only, weights written here
    int64_t p_stride;      // floats between weight rows in p_out
};

// biencoder_attention geometry: G lanes per query row holding eight or
// sixteen context items each (K <= 8 G or 16 G, G <= 32), in CTAs of 256
// threads, or 512 for G >= 16 (a 256-item context: 16-row tiles instead of
// 8 made 4 x 8 x 1024 x 256 x 64 24% faster; at G = 8 the larger CTAs were
// 3% slower); keys transposed in shared memory with rows of kp (K rounded
// up to 4) floats.
constexpr int kBiencMaxThreads = 512;
__host__ __device__ constexpr int bienc_threads(int G) {
    return G >= 16 ? 512 : 256;
}
constexpr int kBiencMaxContext = 256;
constexpr int kBiencMaxDHead = 256;

__host__ __device__ inline int bienc_kp(int K) { return (K + 3) & ~3; }

// Row stride in floats of a tile's scores (then weights): at least kp, and
// for G < 8 congruent to 4 G modulo 32, so that the 16-byte reads of the
// rows a quarter-warp's lanes search fall in different banks.
__host__ __device__ inline int bienc_ss_stride(int K, int G) {
    const int kp = bienc_kp(K);
    if (G >= 8) return kp + 4;
    return kp + (((4 * G - kp) % 32) + 32) % 32;
}

// Shared memory of the one-kernel path: transposed keys, values, a tile
// of queries and a tile of scores (which become the weights).
inline int64_t bienc_smem_bytes(int K, int D, int G) {
    const int64_t R = bienc_threads(G) / G;
    const int64_t kp = bienc_kp(K);
    return 4 * (D * kp + static_cast<int64_t>(K) * D + R * (D + 4) +
                R * bienc_ss_stride(K, G));
}

// Shared memory of the scores-and-search kernel when step 3 runs on the
// tensor cores: the transposed keys, a tile of queries and its scores.
inline int64_t bienc_search_smem_bytes(int K, int D, int G) {
    const int64_t R = bienc_threads(G) / G;
    const int64_t kp = bienc_kp(K);
    return 4 * (D * kp + R * (D + 4) + R * bienc_ss_stride(K, G));
}

// Query tiles one CTA works through with its staged keys and values:
// about 128 query rows, at most the pair's whole query range.
inline int bienc_tiles_per_cta(int Q, int G) {
    const int R = bienc_threads(G) / G;
    const int tiles = (Q + R - 1) / R;
    int per = (128 + R - 1) / R;
    if (per > tiles) per = tiles;
    return per < 1 ? 1 : per;
}

cudaError_t launch_bienc(const BiencTask& task, int lanes_per_row,
                         int keys_per_lane, int smem_bytes,
                         cudaStream_t stream);

// biencoder_attention's step 3 on the tensor cores (k_bienc_pv.cu): out =
// P . V for every bh, P written before by the scores-and-search kernel
// (into attn_out, or into the first K floats of each output row).
struct PvTask {
    const float* p;        // P rows: p + (bh Q + i) p_stride
    int64_t p_stride;      // floats between P rows (K or D)
    const float* v;        // [BH, K, D]
    float* out;            // [BH, Q, D]
    unsigned int* err;     // device error word
    int32_t BH;
    int32_t Q;
    int32_t K;
    int32_t D;
    uint64_t wait_limit_cycles;
};

constexpr int kPvM = 128;               // query rows per tile (the MMA's M)
constexpr uint32_t kPvTmemCols = 128;   // two fp32 accumulators of N <= 64
constexpr int kPvMaxD = 64;             // head sizes the tensor-core step takes

// N of the MMA: d_head rounded up to 16; its K: the context rounded up to 8
// (the context is at most d_head, so one shared-memory stage holds it).
__host__ __device__ inline int pv_np(int D) { return (D + 15) & ~15; }
__host__ __device__ inline int pv_kp(int K) { return (K + 7) & ~7; }

// Byte offsets of the step-3 kernel's shared memory: two stages of the
// TF32 halves of a tile's P (stage s: hi at 2 s a_half, lo a_half later),
// each half 128 rows x pv_chunks(K) chunks of 32 items in the MMA's 128-byte
// swizzled K-major layout (a chunk is 128 rows of 128 bytes, 16 KB); the
// halves of V^T (Np x Kp, no swizzle); the output tile (128 rows of D + 4
// floats); ten mbarriers (full, empty, acc_full, acc_empty, landed, two of
// each), the abort flag and the word that receives the tensor-memory
// address.
__host__ __device__ inline int pv_chunks(int K) { return (K + 31) / 32; }

struct PvSmemLayout {
    int a_half, b_hi, b_lo, stage, bar, flag, tslot, end;
};

__host__ __device__ inline PvSmemLayout pv_smem_layout(int K, int Np, int D) {
    PvSmemLayout L;
    const int Kp = pv_kp(K);
    L.a_half = pv_chunks(K) * kPvM * 128;
    L.b_hi = 4 * L.a_half;
    L.b_lo = L.b_hi + Np * Kp * 4;
    L.stage = L.b_lo + Np * Kp * 4;
    L.bar = L.stage + kPvM * (D + 4) * 4;
    L.flag = L.bar + 10 * 8;
    L.tslot = L.flag + 4;
    L.end = L.tslot + 4;
    return L;
}

// Bytes to allocate: the layout plus slack to align it to 1024 bytes.
inline int64_t pv_smem_bytes(int K, int D) {
    return pv_smem_layout(K, pv_np(D), D).end + 1024;
}

// Persistent CTAs, one per SM at most, each taking a contiguous run of
// tiles.
cudaError_t launch_bienc_pv(const PvTask& task, int sm_count,
                            cudaStream_t stream);

cudaError_t launch_rowgroup(const RowTask& task, int lanes_per_row,
                            int elems_per_lane, cudaStream_t stream);
cudaError_t launch_cluster(const RowTask& task, int cluster_size,
                           int slice_len, int threads, int smem_bytes,
                           int64_t grid_ctas, cudaStream_t stream);
cudaError_t launch_probe_ex2(float* sink, int iters, int blocks, int threads,
                             cudaStream_t stream);
cudaError_t launch_wait_timeout(unsigned int* err, uint64_t limit_cycles,
                                cudaStream_t stream);
cudaError_t launch_take_error(unsigned int* err, unsigned int* taken,
                              cudaStream_t stream);

// cudaFuncSetAttribute(MaxDynamicSharedMemorySize) once per device and
// kernel, raised only when a launch needs more than was set before.
// slot: one per kernel instantiation; cluster: it is launched in clusters
// (also allows cluster sizes above 8).
cudaError_t ensure_smem_attribute(const void* func, int slot, int bytes,
                                  bool cluster);

}  // namespace cs
