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

// Default limit of every bounded device wait (2 s).
constexpr uint64_t kWaitLimitNs = 2000000000ull;

// One launch's worth of work: every row of the matrix with the same
// parameters (the arguments of section 2.1's signature plus t_out and the
// error word).
struct RowTask {
    const float* logits;
    float* out;
    float* t_out;          // may be null
    unsigned int* err;     // device error word
    int64_t batch;
    int32_t num_classes;
    int32_t max_iter;
    float entropy_bound;
    float t_min;
    float hi0;             // min(1, t_max): upper end of the search
    float prune_k;         // active-set threshold K (0: no pruning)
    uint64_t wait_limit_ns;
};

// Cluster kernel geometry.
constexpr int kMaxCluster = 16;
constexpr int kLoadChunks = 8;        // bulk copies per CTA slice
constexpr int kClusterMaxThreads = 1024;

// Per-warp active-set buffer of the cluster kernel: up to this many floats
// (8 per lane); below kMinWarpBuffer pruning is off.
constexpr int kMaxWarpBuffer = 256;
constexpr int kMinWarpBuffer = 64;

// Dynamic shared memory of the cluster kernel for a slice of `slice_len`
// classes, `threads` threads, cluster size `n` and `cap_w` floats of
// active-set buffer per warp.
inline int64_t cluster_smem_bytes(int64_t slice_len, int threads, int n,
                                  int cap_w) {
    const int64_t warps = threads / 32;
    const int64_t slots = 2 * warps * n * 8;            // exchange buffers
    const int64_t bars = (2 + kLoadChunks) * 8;         // mbarriers
    const int64_t head = ((slots + bars + 127) / 128) * 128;
    const int64_t wbuf = warps * cap_w * 4;
    const int64_t row = ((slice_len + 8 + 3) / 4) * 16;  // pad + tail room
    return head + wbuf + row;
}

inline int cluster_threads_for(int64_t slice_len) {
    // About 16 classes per thread per pass, 128..1024 threads.
    int64_t t = (slice_len + 15) / 16;
    t = ((t + 31) / 32) * 32;
    if (t < 128) t = 128;
    if (t > kClusterMaxThreads) t = kClusterMaxThreads;
    return static_cast<int>(t);
}

// Active-set threshold K for rows of C classes: 36 + ceil(log2 C).
inline float prune_threshold(int64_t C) {
    int lg = 0;
    while ((int64_t{1} << lg) < C) ++lg;
    return static_cast<float>(36 + lg);
}

cudaError_t launch_rowgroup(const RowTask& task, int lanes_per_row,
                            int elems_per_lane, cudaStream_t stream);
cudaError_t launch_cluster(const RowTask& task, int cluster_size,
                           int slice_len, int threads, int cap_w,
                           int smem_bytes, int64_t grid_ctas,
                           cudaStream_t stream);
cudaError_t launch_probe_ex2(float* sink, int iters, int blocks, int threads,
                             cudaStream_t stream);
cudaError_t launch_wait_timeout(unsigned int* err, uint64_t limit_ns,
                                cudaStream_t stream);

}  // namespace cs
