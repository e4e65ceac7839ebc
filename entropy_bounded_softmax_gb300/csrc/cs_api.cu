// C ABI of libcsoftmax: argument checks, launch planning, the device error
// word, and dispatch to the kernels.  See include/entropy_bounded_softmax.h
// for the contract of every function.
#include <float.h>
#include <math.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

#include "cs_internal.h"

// The library's device objects: a bitmask of (1 << code) for the
// asynchronous conditions of "BURT-IMMA CUDA Kernel API Reference",
// section 5.1 (set with atomicOr, so no condition overwrites another), and
// the word cs_get_error exchanges it into before copying it to the host.
__device__ unsigned int g_cs_error_word;
__device__ unsigned int g_cs_error_taken;

namespace cs {
int probe_chains();
}

namespace {

constexpr int kMaxDevices = 64;
constexpr int kProbeThreads = 512;
constexpr int kProbeBlocksPerSm = 4;
// Row-group CTAs of two warps: the block scheduler refills SMs at a fine
// grain, which shortens the launch's tail (rows end at different rounds).
constexpr int kRowgroupThreads = 64;
constexpr int kRowgroupMaxLanes = 32;
constexpr int kRowgroupMaxE4 = 8;      // 32 classes per lane
constexpr int kAutoRowgroupE4 = 4;     // 16 classes per lane
// Widest rows the forward plans on the row-group kernel by default: one
// warp of 32 lanes, 32 classes a lane.  Rows of 513-1024 classes ran
// 1.3-1.4x faster there than in one-CTA clusters with a few rows, and
// 3.1-5.3x faster with 4096-16384 rows (measured at 600, 768, 1000 and
// 1024 classes).  The backward keeps 512 (four float4s of p and of g a
// lane).
constexpr int kAutoRowgroupMaxClassesFwd = 1024;
constexpr int kAutoRowgroupMaxClasses = 512;
constexpr int kMaxIter = 1024;
// Largest t_min accepted: 2^64.  Every temperature a kernel evaluates or
// writes is at most max(1, t_min), so 1/T >= 2^-64 and the floored
// exponent (-2^100) times 1/T stays below -2^36: its term is exactly 0.
constexpr float kMaxTMin = 18446744073709551616.0f;
constexpr int64_t kMaxGridX = 2147483647;
constexpr int64_t kMinWideSlice = 2048;

struct DeviceInfo {
    std::atomic<bool> ready{false};
    int sm_count = 0;
    int smem_optin = 0;
    int smem_per_sm = 0;
    int cc_major = 0;
    int cc_minor = 0;
    int max_cluster = 1;
    unsigned int* err = nullptr;
    unsigned int* err_taken = nullptr;
    std::mutex take_mu;  // one cs_get_error at a time uses err_taken
};

DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

cs_status device_info(DeviceInfo** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return CS_ERR_CUDA;
    }
    if (dev < 0 || dev >= kMaxDevices) return CS_ERR_CUDA;
    DeviceInfo& d = g_dev[dev];
    if (!d.ready.load(std::memory_order_acquire)) {
        std::lock_guard<std::mutex> lock(g_dev_mu);
        if (!d.ready.load(std::memory_order_relaxed)) {
            int v[5] = {0, 0, 0, 0, 0};
            const cudaDeviceAttr attrs[5] = {
                cudaDevAttrMultiProcessorCount,
                cudaDevAttrMaxSharedMemoryPerBlockOptin,
                cudaDevAttrMaxSharedMemoryPerMultiprocessor,
                cudaDevAttrComputeCapabilityMajor,
                cudaDevAttrComputeCapabilityMinor};
            for (int i = 0; i < 5; ++i) {
                if (cudaDeviceGetAttribute(&v[i], attrs[i], dev) != cudaSuccess) {
                    cudaGetLastError();
                    return CS_ERR_CUDA;
                }
            }
            void* p = nullptr;
            void* q = nullptr;
            if (cudaGetSymbolAddress(&p, g_cs_error_word) != cudaSuccess ||
                cudaGetSymbolAddress(&q, g_cs_error_taken) != cudaSuccess) {
                cudaGetLastError();
                return CS_ERR_CUDA;
            }
            d.sm_count = v[0];
            d.smem_optin = v[1];
            d.smem_per_sm = v[2];
            d.cc_major = v[3];
            d.cc_minor = v[4];
            d.max_cluster = v[3] >= 9 ? cs::kMaxCluster : 1;
            d.err = static_cast<unsigned int*>(p);
            d.err_taken = static_cast<unsigned int*>(q);
            d.ready.store(true, std::memory_order_release);
        }
    }
    *out = &d;
    return CS_OK;
}

bool ranges_overlap(const void* a, int64_t a_bytes, const void* b,
                    int64_t b_bytes) {
    if (!a || !b || a_bytes <= 0 || b_bytes <= 0) return false;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a);
    const uintptr_t b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + static_cast<uintptr_t>(b_bytes) &&
           b0 < a0 + static_cast<uintptr_t>(a_bytes);
}

int next_pow2(int64_t x) {
    int p = 1;
    while (p < x) p <<= 1;
    return p;
}

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

cs_status plan_rowgroup(int64_t batch, int32_t C, int32_t param,
                        cs_plan* p) {
    const int64_t q = ceil_div(C, 4);
    int G = 0, e4 = 0;
    if (param == 0) {
        for (int g = 1; g <= kRowgroupMaxLanes; g <<= 1) {
            if (ceil_div(q, g) <= kAutoRowgroupE4) {
                G = g;
                break;
            }
        }
        if (G == 0) G = kRowgroupMaxLanes;
    } else {
        if (param < 1 || param > kRowgroupMaxLanes || (param & (param - 1)))
            return CS_ERR_INVALID_ARG;
        G = param;
    }
    e4 = next_pow2(ceil_div(q, G));
    if (e4 > kRowgroupMaxE4) return CS_ERR_OOM;
    *p = cs_plan{};
    p->variant = CS_VARIANT_ROWGROUP;
    p->lanes_per_row = G;
    p->elems_per_lane = 4 * e4;
    p->threads_per_cta = kRowgroupThreads;
    // Registers bound residency: at most 64 per thread (80 for 32 classes
    // per lane) out of 65536 per SM.
    p->ctas_per_sm = 65536 / ((e4 >= 8 ? 80 : 64) * kRowgroupThreads);
    if (p->ctas_per_sm > 32) p->ctas_per_sm = 32;
    int64_t blocks = ceil_div(batch * G, kRowgroupThreads);
    if (blocks > kMaxGridX) blocks = kMaxGridX;
    p->grid_ctas = blocks;
    return CS_OK;
}

// Cluster plan for n CTAs per row: slice, threads and shared memory.
// Returns false if it does not fit smem_optin.
bool cluster_geometry(int64_t batch, int32_t C, int n, int threads_req,
                      int sm_count, int smem_optin, cs_plan* p) {
    const int64_t L = ceil_div(ceil_div(C, n), 4) * 4;
    const int threads = threads_req
        ? threads_req : cs::cluster_threads_for(L, batch * n, sm_count, n);
    const int64_t smem = cs::cluster_smem_bytes(L, threads, n);
    if (smem > smem_optin) return false;
    p->cluster_size = n;
    p->slice_len = static_cast<int32_t>(L);
    p->threads_per_cta = threads;
    p->smem_bytes = static_cast<int32_t>(smem);
    p->staged_tensors = 1;
    return true;
}

cs_status plan_cluster(int64_t batch, int32_t C, const cs_options& o,
                       int sm_count, int smem_optin, int smem_per_sm,
                       int max_cluster, cs_plan* p) {
    if (o.threads != 0 &&
        (o.threads < 64 || o.threads > cs::kClusterMaxThreads || o.threads % 32))
        return CS_ERR_INVALID_ARG;
    if (o.strict != 0 && o.strict != 1) return CS_ERR_INVALID_ARG;
    *p = cs_plan{};
    p->variant = CS_VARIANT_CLUSTER;
    if (o.param == 0) {
        // Smallest cluster whose slices are at most kTargetSlice classes
        // (and fit), widened while the launch has fewer CTAs than SMs.
        int n0 = static_cast<int>(ceil_div(C, cs::kTargetSlice));
        if (n0 > max_cluster) n0 = max_cluster;
        if (n0 < 1) n0 = 1;
        // Widen only while every CTA keeps at least kMinWideSlice classes.
        // Few rows: two CTAs per SM, rounded up when that oversubscribes
        // the SMs by at most a quarter.  Two CTAs of a latency-bound launch
        // share an SM well: one's exchange overlaps the other's pass, and
        // the slices (hence every pass) are half as long.  32 x 50000 runs in
        // clusters of 10 x 128 threads, 320 CTAs: 15.9 us, against 17.5 us
        // in clusters of 5 x 256 (one CTA per SM) and 19.2 in clusters of 4.
        const int64_t rows = batch > 0 ? batch : 1;
        const int64_t slots = 2 * static_cast<int64_t>(sm_count);
        int64_t widen = slots / rows;
        const int64_t up = ceil_div(slots, rows);
        if (up > widen && rows * up * 4 <= slots * 5) widen = up;
        if (widen > C / kMinWideSlice) widen = C / kMinWideSlice;
        if (widen > max_cluster) widen = max_cluster;
        if (widen > n0) n0 = static_cast<int>(widen);
        bool ok = false;
        for (int c = n0; c <= max_cluster && !ok; ++c)
            ok = cluster_geometry(batch, C, c, o.threads, sm_count,
                                  smem_optin, p);
        if (!ok) return CS_ERR_OOM;
    } else {
        if (o.param < 1 || o.param > cs::kMaxCluster) return CS_ERR_INVALID_ARG;
        if (o.param > max_cluster) return CS_ERR_INVALID_ARG;
        if (!cluster_geometry(batch, C, o.param, o.threads, sm_count,
                              smem_optin, p))
            return CS_ERR_OOM;
    }
    const int n = p->cluster_size;
    const int by_smem = static_cast<int>(smem_per_sm / (p->smem_bytes + 1024));
    const int by_threads = 2048 / p->threads_per_cta;
    p->ctas_per_sm = by_smem < by_threads ? by_smem : by_threads;
    int64_t rows = batch;
    const int64_t max_rows = kMaxGridX / n;
    if (rows > max_rows) rows = max_rows;
    p->grid_ctas = rows * n;
    // Launches of at most one wave are bound by the slowest row's chain of
    // rounds: there the fan, a few more exponentials per class in the T = 1
    // pass, saves rounds.  Wider launches are bound by throughput, where the
    // extra exponentials cost more than the rounds they save.  The fan runs
    // in clusters of CTAs of at most 256 threads, built with registers for
    // 512 threads an SM (cs::kFanThreadsPerSm).
    const int64_t fan_ctas_per_sm = cs::kFanThreadsPerSm / p->threads_per_cta;
    const int64_t resident =
        fan_ctas_per_sm < p->ctas_per_sm ? fan_ctas_per_sm : p->ctas_per_sm;
    const bool one_wave = p->grid_ctas <= static_cast<int64_t>(sm_count) * resident;
    p->fan_points = (o.strict == 0 && n > 1 && p->threads_per_cta <= 256 && one_wave)
        ? cs::kFanPoints : 0;
    if (p->fan_points > 0 && o.param == 0 && o.threads == 0 &&
        p->grid_ctas > 2 * static_cast<int64_t>(sm_count)) {
        // With the fan the T = 1 pass is about twice as long, and a CTA
        // that shares its SM with two others holds up its whole cluster's
        // first exchange: when the widening above rounded up past two CTAs
        // an SM, take instead the largest power-of-two cluster that keeps
        // at most two on every SM (32 x 50000: clusters of 8 x 128, 14.5 us,
        // against 15.3 us in the clusters of 10).
        int nf = 1;
        while (nf * 2 <= max_cluster && nf * 2 <= C / kMinWideSlice &&
               rows * nf * 2 <= 2 * static_cast<int64_t>(sm_count))
            nf *= 2;
        cs_plan q = *p;
        if (nf > 1 && nf != n && ceil_div(C, nf) <= cs::kTargetSlice &&
            cluster_geometry(batch, C, nf, 0, sm_count, smem_optin, &q) &&
            q.threads_per_cta <= 256) {
            const int bs = static_cast<int>(smem_per_sm / (q.smem_bytes + 1024));
            const int bt = 2048 / q.threads_per_cta;
            q.ctas_per_sm = bs < bt ? bs : bt;
            q.grid_ctas = rows * nf;
            *p = q;
        }
    }
    return CS_OK;
}

// ------------------------------------------------------------------ backward
// Row-group backward: G lanes per row, the smallest power of two that leaves
// at most four float4s of p (and of g) per lane; float4s counted for the
// worst alignment of a row start (pad 3), since rows of a num_classes that
// is not a multiple of 4 start at every alignment.
cs_status plan_backward_rowgroup(int64_t batch, int32_t C, int32_t param,
                                 cs_plan* p) {
    const int64_t q = (static_cast<int64_t>(C) + 6) / 4;
    int G = 0;
    if (param == 0) {
        for (int g = 1; g <= kRowgroupMaxLanes; g <<= 1) {
            if (ceil_div(q, g) <= kAutoRowgroupE4) {
                G = g;
                break;
            }
        }
        if (G == 0) G = kRowgroupMaxLanes;
    } else {
        if (param < 1 || param > kRowgroupMaxLanes || (param & (param - 1)))
            return CS_ERR_INVALID_ARG;
        G = param;
    }
    const int e4 = next_pow2(ceil_div(q, G));
    if (e4 > kRowgroupMaxE4) return CS_ERR_OOM;
    const int64_t blocks = ceil_div(batch * G, cs::kBwdGroupThreads);
    if (blocks > kMaxGridX) return CS_ERR_DIM_MISMATCH;
    *p = cs_plan{};
    p->variant = CS_VARIANT_ROWGROUP;
    p->lanes_per_row = G;
    p->elems_per_lane = 4 * e4;
    p->threads_per_cta = cs::kBwdGroupThreads;
    // Registers bound residency: 2 x 4 e4 for the row plus about 28
    // (ptxas: 32, 38, 60 and 90 for e4 = 1, 2, 4, 8).
    int regs = ((8 * e4 + 28 + 7) / 8) * 8;
    if (regs < 32) regs = 32;
    p->ctas_per_sm = 65536 / (regs * cs::kBwdGroupThreads);
    if (p->ctas_per_sm > 2048 / cs::kBwdGroupThreads)
        p->ctas_per_sm = 2048 / cs::kBwdGroupThreads;
    p->grid_ctas = blocks;
    return CS_OK;
}

// Cluster backward geometry for n CTAs per row: p and g staged when both
// fit, else p alone (stage_both = false); false if neither fits.  per: the
// float4s of each staged tensor per thread the automatic thread count aims
// for.
bool backward_geometry(int32_t C, int n, int threads_req, int smem_optin,
                       bool stage_both, int per, cs_plan* p) {
    const int64_t L = ceil_div(ceil_div(C, n), 4) * 4;
    const int64_t smem = cs::backward_smem_bytes(L, stage_both);
    if (smem > smem_optin) return false;
    int threads = threads_req;
    if (threads == 0) {
        int64_t t = ceil_div(ceil_div(L, 4), per);
        t = ceil_div(t, 32) * 32;
        if (t < 64) t = 64;
        if (t > cs::kBwdMaxThreads) t = cs::kBwdMaxThreads;
        threads = static_cast<int>(t);
    }
    p->cluster_size = n;
    p->slice_len = static_cast<int32_t>(L);
    p->threads_per_cta = threads;
    p->smem_bytes = static_cast<int32_t>(smem);
    p->staged_tensors = stage_both ? 2 : 1;
    return true;
}

cs_status plan_backward_cluster(int64_t batch, int32_t C, const cs_options& o,
                                int sm_count, int smem_optin, int smem_per_sm,
                                int max_cluster, cs_plan* p) {
    if (o.threads != 0 &&
        (o.threads < 64 || o.threads > cs::kBwdMaxThreads || o.threads % 32))
        return CS_ERR_INVALID_ARG;
    *p = cs_plan{};
    p->variant = CS_VARIANT_CLUSTER;
    bool ok = false;
    if (o.param == 0) {
        // Smallest cluster whose slices are at most kBwdTargetSlice classes,
        // widened to about two CTAs per SM for few rows while slices keep
        // kMinWideSlice classes (32 x 50000: clusters of 10, 5000-class
        // slices).
        int n0 = static_cast<int>(ceil_div(C, cs::kBwdTargetSlice));
        if (n0 > max_cluster) n0 = max_cluster;
        if (n0 < 1) n0 = 1;
        const int64_t rows = batch > 0 ? batch : 1;
        int64_t widen = ceil_div(2 * static_cast<int64_t>(sm_count), rows);
        if (widen > C / kMinWideSlice) widen = C / kMinWideSlice;
        if (widen > max_cluster) widen = max_cluster;
        // Launches of few CTAs are latency-bound: fewer float4s per thread
        // (32 x 50000 in clusters of 10: 6.9 us on 160 threads, 6.6 on
        // 256); larger ones aim for eight, enough in flight per SM.
        const int per = widen > n0 ? 5 : 8;
        if (widen > n0) n0 = static_cast<int>(widen);
        for (int c = n0; c <= max_cluster && !ok; ++c)
            ok = backward_geometry(C, c, o.threads, smem_optin, true, per, p);
        if (!ok)
            ok = backward_geometry(C, max_cluster, o.threads, smem_optin,
                                   false, per, p);
    } else {
        if (o.param < 1 || o.param > cs::kMaxCluster) return CS_ERR_INVALID_ARG;
        if (o.param > max_cluster) return CS_ERR_INVALID_ARG;
        ok = backward_geometry(C, o.param, o.threads, smem_optin, true, 8, p) ||
             backward_geometry(C, o.param, o.threads, smem_optin, false, 8, p);
    }
    if (!ok) return CS_ERR_OOM;
    const int n = p->cluster_size;
    const int by_smem = static_cast<int>(smem_per_sm / (p->smem_bytes + 1024));
    const int by_threads = 2048 / p->threads_per_cta;
    p->ctas_per_sm = by_smem < by_threads ? by_smem : by_threads;
    int64_t rows = batch;
    const int64_t max_rows = kMaxGridX / n;
    if (rows > max_rows) rows = max_rows;
    p->grid_ctas = rows * n;
    return CS_OK;
}

// ------------------------------------------------------------------ attention
cs_status plan_attention(int32_t batch, int32_t heads, int32_t S,
                         int32_t aligned, const cs_options& o, int sm_count,
                         int smem_optin, int smem_per_sm, cs_plan* p) {
    (void)sm_count;
    if (o.strict != 0 || o.evals_out) return CS_ERR_INVALID_ARG;
    const int64_t rows = static_cast<int64_t>(batch) * heads * S;
    // Float4s a row spans: exact for aligned rows, else at the worst
    // alignment of a row start.
    int64_t q = aligned ? ceil_div(S, 4) : (static_cast<int64_t>(S) + 6) / 4;
    if (q < 1) q = 1;
    int variant = o.variant;
    if (variant == CS_VARIANT_AUTO) {
        if (o.param != 0 || o.threads != 0) return CS_ERR_INVALID_ARG;
        variant = q <= kRowgroupMaxLanes * kRowgroupMaxE4 ? CS_VARIANT_ROWGROUP
                                                          : CS_VARIANT_CLUSTER;
    }
    *p = cs_plan{};
    if (variant == CS_VARIANT_ROWGROUP) {
        if (o.threads != 0) return CS_ERR_INVALID_ARG;
        int G = 0;
        if (o.param == 0) {
            for (int g = 1; g <= kRowgroupMaxLanes; g <<= 1) {
                if (ceil_div(q, g) <= kAutoRowgroupE4) {
                    G = g;
                    break;
                }
            }
            if (G == 0) G = kRowgroupMaxLanes;
        } else {
            if (o.param < 1 || o.param > kRowgroupMaxLanes || (o.param & (o.param - 1)))
                return CS_ERR_INVALID_ARG;
            G = o.param;
        }
        const int e4 = next_pow2(ceil_div(q, G));
        if (e4 > kRowgroupMaxE4) return CS_ERR_OOM;
        const int64_t blocks = ceil_div(rows * G, cs::kAttnGroupThreads);
        if (blocks > kMaxGridX) return CS_ERR_DIM_MISMATCH;
        p->variant = CS_VARIANT_ROWGROUP;
        p->lanes_per_row = G;
        p->elems_per_lane = 4 * e4;
        p->threads_per_cta = cs::kAttnGroupThreads;
        int regs = ((4 * e4 + 30 + 7) / 8) * 8;
        p->ctas_per_sm = 65536 / (regs * cs::kAttnGroupThreads);
        if (p->ctas_per_sm > 2048 / cs::kAttnGroupThreads)
            p->ctas_per_sm = 2048 / cs::kAttnGroupThreads;
        p->grid_ctas = blocks;
        return CS_OK;
    }
    if (variant != CS_VARIANT_CLUSTER) return CS_ERR_INVALID_ARG;
    if (o.param != 0 && o.param != 1) return CS_ERR_INVALID_ARG;
    if (o.threads != 0 &&
        (o.threads < 64 || o.threads > cs::kAttnMaxThreads || o.threads % 32))
        return CS_ERR_INVALID_ARG;
    const int64_t smem = cs::attention_smem_bytes(S);
    if (smem > smem_optin) return CS_ERR_OOM;
    int threads = o.threads;
    if (threads == 0) {
        // About eight float4s per thread.
        int64_t t = ceil_div(ceil_div(q, 8), 32) * 32;
        if (t < 64) t = 64;
        if (t > cs::kAttnMaxThreads) t = cs::kAttnMaxThreads;
        threads = static_cast<int>(t);
    }
    p->variant = CS_VARIANT_CLUSTER;
    p->cluster_size = 1;
    p->slice_len = S;
    p->threads_per_cta = threads;
    p->smem_bytes = static_cast<int32_t>(smem);
    p->staged_tensors = 1;
    const int by_smem = static_cast<int>(smem_per_sm / (smem + 1024));
    const int by_threads = 2048 / threads;
    p->ctas_per_sm = by_smem < by_threads ? by_smem : by_threads;
    p->grid_ctas = rows < kMaxGridX ? rows : kMaxGridX;
    return CS_OK;
}

}  // namespace

namespace {

// Argument check of the forward for logits of in_bytes (4: fp32, 2: bf16)
// per element.
cs_status check_forward_args(const void* logits, const float* out,
                             int64_t batch, int32_t num_classes,
                             float entropy_bound, float t_min, float t_max,
                             int32_t max_iter, const float* t_out,
                             int in_bytes) {
    if (batch < 0 || num_classes < 1) return CS_ERR_DIM_MISMATCH;
    if (num_classes > CS_MAX_NUM_CLASSES) return CS_ERR_OOM;
    if (batch > INT64_MAX / 4 / num_classes) return CS_ERR_DIM_MISMATCH;
    if (isnan(entropy_bound)) return CS_ERR_INVALID_ARG;
    if (!(t_min >= FLT_MIN) || !(t_min <= kMaxTMin)) return CS_ERR_INVALID_ARG;
    if (isnan(t_max) || t_max < t_min) return CS_ERR_INVALID_ARG;
    if (max_iter < 0 || max_iter > kMaxIter) return CS_ERR_INVALID_ARG;
    if (batch == 0) return CS_OK;
    if (!logits || !out) return CS_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(logits) % in_bytes) return CS_ERR_INVALID_ARG;
    const int64_t in_size = batch * num_classes * in_bytes;
    const int64_t bytes = batch * num_classes * 4;
    if (ranges_overlap(logits, in_size, out, bytes)) return CS_ERR_INVALID_ARG;
    if (t_out && (ranges_overlap(t_out, batch * 4, logits, in_size) ||
                  ranges_overlap(t_out, batch * 4, out, bytes)))
        return CS_ERR_INVALID_ARG;
    return CS_OK;
}

// The forward for fp32 (in_bf16 = false) or bf16 logits.
cs_status forward(const void* logits, bool in_bf16, float* out, int64_t batch,
                  int32_t num_classes, float entropy_bound, float t_min,
                  float t_max, int32_t max_iter, float* t_out,
                  const cs_options* options, void* stream) {
    const int in_bytes = in_bf16 ? 2 : 4;
    cs_status st = check_forward_args(logits, out, batch, num_classes,
                                      entropy_bound, t_min, t_max, max_iter,
                                      t_out, in_bytes);
    if (st != CS_OK) return st;
    if (batch == 0) return CS_OK;
    if (options && options->evals_out) {
        const int64_t bytes = batch * num_classes * 4;
        const void* e = options->evals_out;
        if (ranges_overlap(e, batch * 4, logits, batch * num_classes * in_bytes) ||
            ranges_overlap(e, batch * 4, out, bytes) ||
            (t_out && ranges_overlap(e, batch * 4, t_out, batch * 4)))
            return CS_ERR_INVALID_ARG;
    }
    DeviceInfo* d = nullptr;
    st = device_info(&d);
    if (st != CS_OK) return st;
    cs_plan p;
    st = cs_plan_host(batch, num_classes, options, d->sm_count, d->smem_optin,
                      d->smem_per_sm, d->max_cluster, &p);
    if (st != CS_OK) return st;

    cs::RowTask task;
    task.logits = logits;
    task.out = out;
    task.t_out = t_out;
    task.err = d->err;
    task.batch = batch;
    task.num_classes = num_classes;
    task.max_iter = max_iter;
    task.entropy_bound = entropy_bound;
    task.t_min = t_min;
    task.hi0 = t_max < 1.0f ? t_max : 1.0f;
    task.strict = options ? options->strict : 0;
    // Asynchronous staging pays when several CTAs share an SM (the same
    // threshold as the per-thread work rule of the thread count).
    task.async_stage = p.grid_ctas * 4 > static_cast<int64_t>(d->sm_count) * 5;
    task.wait_limit_cycles = cs::kWaitLimitCycles;
    task.evals_out = options ? options->evals_out : nullptr;
    task.in_bf16 = in_bf16 ? 1 : 0;
    // The fan's inverse temperatures sqrt(1 / (hi0 t_min)) times 1/4, 1 and
    // 4: the middle of the search's range in log beta and a factor 4 on
    // either side; only when that range spans a factor 64 or more.
    task.fan_beta0 = 0.0f;
    if (p.variant == CS_VARIANT_CLUSTER && p.fan_points > 0 &&
        entropy_bound > 0.0f && 64.0 * t_min <= task.hi0)
        task.fan_beta0 = static_cast<float>(
            0.25 / sqrt(static_cast<double>(task.hi0) * t_min));

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (p.variant == CS_VARIANT_ROWGROUP) {
        e = cs::launch_rowgroup(task, p.lanes_per_row, p.elems_per_lane, s);
    } else {
        e = cs::launch_cluster(task, p.cluster_size, p.slice_len,
                               p.threads_per_cta, p.smem_bytes, p.grid_ctas, s);
    }
    if (e != cudaSuccess) {
        cudaGetLastError();
        return CS_ERR_CUDA;
    }
    return CS_OK;
}

}  // namespace

extern "C" {

cs_status cs_check_args(const float* logits, const float* out, int64_t batch,
                        int32_t num_classes, float entropy_bound, float t_min,
                        float t_max, int32_t max_iter, const float* t_out) {
    return check_forward_args(logits, out, batch, num_classes, entropy_bound,
                              t_min, t_max, max_iter, t_out, 4);
}

cs_status cs_check_args_bf16(const uint16_t* logits, const float* out,
                             int64_t batch, int32_t num_classes,
                             float entropy_bound, float t_min, float t_max,
                             int32_t max_iter, const float* t_out) {
    return check_forward_args(logits, out, batch, num_classes, entropy_bound,
                              t_min, t_max, max_iter, t_out, 2);
}

cs_status cs_plan_host(int64_t batch, int32_t num_classes,
                       const cs_options* options, int32_t sm_count,
                       int32_t smem_per_block_optin, int32_t smem_per_sm,
                       int32_t max_cluster, cs_plan* plan) {
    if (!plan) return CS_ERR_INVALID_ARG;
    if (batch < 0 || num_classes < 1) return CS_ERR_DIM_MISMATCH;
    if (num_classes > CS_MAX_NUM_CLASSES) return CS_ERR_OOM;
    if (sm_count < 1 || smem_per_block_optin < 1 || smem_per_sm < 1 ||
        max_cluster < 1)
        return CS_ERR_INVALID_ARG;
    if (max_cluster > cs::kMaxCluster) max_cluster = cs::kMaxCluster;
    cs_options o = options ? *options : cs_options{};
    if (o.variant == CS_VARIANT_AUTO) {
        if (o.param != 0) return CS_ERR_INVALID_ARG;
        o.variant = num_classes <= kAutoRowgroupMaxClassesFwd ? CS_VARIANT_ROWGROUP
                                                              : CS_VARIANT_CLUSTER;
    }
    if (o.variant == CS_VARIANT_ROWGROUP) {
        if (o.threads != 0 || (o.strict != 0 && o.strict != 1))
            return CS_ERR_INVALID_ARG;
        return plan_rowgroup(batch, num_classes, o.param, plan);
    }
    if (o.variant == CS_VARIANT_CLUSTER)
        return plan_cluster(batch, num_classes, o, sm_count,
                            smem_per_block_optin, smem_per_sm, max_cluster,
                            plan);
    return CS_ERR_INVALID_ARG;
}

cs_status cs_plan_launch(int64_t batch, int32_t num_classes,
                         const cs_options* options, cs_plan* plan) {
    DeviceInfo* d = nullptr;
    const cs_status st = device_info(&d);
    if (st != CS_OK) return st;
    return cs_plan_host(batch, num_classes, options, d->sm_count,
                        d->smem_optin, d->smem_per_sm, d->max_cluster, plan);
}

cs_status cs_constrained_softmax_ex(const float* logits, float* out,
                                    int64_t batch, int32_t num_classes,
                                    float entropy_bound, float t_min,
                                    float t_max, int32_t max_iter,
                                    float* t_out, const cs_options* options,
                                    void* stream) {
    return forward(logits, false, out, batch, num_classes, entropy_bound,
                   t_min, t_max, max_iter, t_out, options, stream);
}

cs_status cs_constrained_softmax(const float* logits, float* out,
                                 int64_t batch, int32_t num_classes,
                                 float entropy_bound, float t_min, float t_max,
                                 int32_t max_iter, float* t_out, void* stream) {
    return forward(logits, false, out, batch, num_classes, entropy_bound,
                   t_min, t_max, max_iter, t_out, nullptr, stream);
}

cs_status cs_constrained_softmax_bf16_ex(const uint16_t* logits, float* out,
                                         int64_t batch, int32_t num_classes,
                                         float entropy_bound, float t_min,
                                         float t_max, int32_t max_iter,
                                         float* t_out,
                                         const cs_options* options,
                                         void* stream) {
    return forward(logits, true, out, batch, num_classes, entropy_bound,
                   t_min, t_max, max_iter, t_out, options, stream);
}

cs_status cs_constrained_softmax_bf16(const uint16_t* logits, float* out,
                                      int64_t batch, int32_t num_classes,
                                      float entropy_bound, float t_min,
                                      float t_max, int32_t max_iter,
                                      float* t_out, void* stream) {
    return forward(logits, true, out, batch, num_classes, entropy_bound,
                   t_min, t_max, max_iter, t_out, nullptr, stream);
}

cs_status cs_get_error(int32_t* code_mask, void* stream) {
    if (!code_mask) return CS_ERR_INVALID_ARG;
    DeviceInfo* d = nullptr;
    const cs_status st = device_info(&d);
    if (st != CS_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    unsigned int h = 0;
    // Read and clear in one atomic exchange on the device, so that a bit a
    // launch on another stream sets at the same time is never dropped.
    std::lock_guard<std::mutex> lock(d->take_mu);
    if (cs::launch_take_error(d->err, d->err_taken, s) != cudaSuccess ||
        cudaMemcpyAsync(&h, d->err_taken, sizeof(h), cudaMemcpyDeviceToHost,
                        s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess) {
        cudaGetLastError();
        return CS_ERR_CUDA;
    }
    *code_mask = static_cast<int32_t>(h);
    return CS_OK;
}

cs_status cs_check_backward_args(const float* probs, const float* grad_out,
                                 const float* t, const float* grad_in,
                                 int64_t batch, int32_t num_classes) {
    if (batch < 0 || num_classes < 1) return CS_ERR_DIM_MISMATCH;
    if (num_classes > CS_MAX_NUM_CLASSES) return CS_ERR_OOM;
    if (batch > INT64_MAX / 4 / num_classes) return CS_ERR_DIM_MISMATCH;
    if (batch == 0) return CS_OK;
    if (!probs || !grad_out || !t || !grad_in) return CS_ERR_INVALID_ARG;
    const int64_t bytes = batch * num_classes * 4;
    if (grad_in != probs && ranges_overlap(grad_in, bytes, probs, bytes))
        return CS_ERR_INVALID_ARG;
    if (grad_in != grad_out && ranges_overlap(grad_in, bytes, grad_out, bytes))
        return CS_ERR_INVALID_ARG;
    if (ranges_overlap(t, batch * 4, grad_in, bytes)) return CS_ERR_INVALID_ARG;
    return CS_OK;
}

cs_status cs_plan_backward_host(int64_t batch, int32_t num_classes,
                                const cs_options* options, int32_t sm_count,
                                int32_t smem_per_block_optin,
                                int32_t smem_per_sm, int32_t max_cluster,
                                cs_plan* plan) {
    if (!plan) return CS_ERR_INVALID_ARG;
    if (batch < 0 || num_classes < 1) return CS_ERR_DIM_MISMATCH;
    if (num_classes > CS_MAX_NUM_CLASSES) return CS_ERR_OOM;
    if (sm_count < 1 || smem_per_block_optin < 1 || smem_per_sm < 1 ||
        max_cluster < 1)
        return CS_ERR_INVALID_ARG;
    if (max_cluster > cs::kMaxCluster) max_cluster = cs::kMaxCluster;
    cs_options o = options ? *options : cs_options{};
    if (o.strict != 0 || o.evals_out) return CS_ERR_INVALID_ARG;
    if (o.variant == CS_VARIANT_AUTO) {
        if (o.param != 0 || o.threads != 0) return CS_ERR_INVALID_ARG;
        o.variant = num_classes <= kAutoRowgroupMaxClasses ? CS_VARIANT_ROWGROUP
                                                           : CS_VARIANT_CLUSTER;
    }
    if (o.variant == CS_VARIANT_ROWGROUP) {
        if (o.threads != 0) return CS_ERR_INVALID_ARG;
        return plan_backward_rowgroup(batch, num_classes, o.param, plan);
    }
    if (o.variant == CS_VARIANT_CLUSTER)
        return plan_backward_cluster(batch, num_classes, o, sm_count,
                                     smem_per_block_optin, smem_per_sm,
                                     max_cluster, plan);
    return CS_ERR_INVALID_ARG;
}

cs_status cs_plan_backward_launch(int64_t batch, int32_t num_classes,
                                  const cs_options* options, cs_plan* plan) {
    DeviceInfo* d = nullptr;
    const cs_status st = device_info(&d);
    if (st != CS_OK) return st;
    return cs_plan_backward_host(batch, num_classes, options, d->sm_count,
                                 d->smem_optin, d->smem_per_sm,
                                 d->max_cluster, plan);
}

cs_status cs_constrained_softmax_backward_ex(const float* probs,
                                             const float* grad_out,
                                             const float* t, float* grad_in,
                                             int64_t batch,
                                             int32_t num_classes,
                                             const cs_options* options,
                                             void* stream) {
    cs_status st = cs_check_backward_args(probs, grad_out, t, grad_in, batch,
                                          num_classes);
    if (st != CS_OK) return st;
    if (batch == 0) return CS_OK;
    DeviceInfo* d = nullptr;
    st = device_info(&d);
    if (st != CS_OK) return st;
    cs_plan p;
    st = cs_plan_backward_host(batch, num_classes, options, d->sm_count,
                               d->smem_optin, d->smem_per_sm, d->max_cluster,
                               &p);
    if (st != CS_OK) return st;
    cs::BwdTask task;
    task.probs = probs;
    task.grad_out = grad_out;
    task.t = t;
    task.grad_in = grad_in;
    task.batch = batch;
    task.num_classes = num_classes;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (p.variant == CS_VARIANT_ROWGROUP) {
        e = cs::launch_backward_rowgroup(task, p.lanes_per_row,
                                         p.elems_per_lane, s);
    } else {
        e = cs::launch_backward_cluster(task, p.cluster_size, p.slice_len,
                                        p.threads_per_cta, p.smem_bytes,
                                        p.staged_tensors == 2, p.grid_ctas, s);
    }
    if (e != cudaSuccess) {
        cudaGetLastError();
        return CS_ERR_CUDA;
    }
    return CS_OK;
}

cs_status cs_constrained_softmax_backward(const float* probs,
                                          const float* grad_out,
                                          const float* t, float* grad_in,
                                          int64_t batch, int32_t num_classes,
                                          void* stream) {
    return cs_constrained_softmax_backward_ex(probs, grad_out, t, grad_in,
                                              batch, num_classes, nullptr,
                                              stream);
}

cs_status cs_check_attention_args(const float* scores, const float* out,
                                  const float* mask, int32_t batch,
                                  int32_t heads, int32_t seq_len,
                                  int32_t causal) {
    if (batch < 0 || heads < 0 || seq_len < 0) return CS_ERR_DIM_MISMATCH;
    if (causal != 0 && causal != 1) return CS_ERR_INVALID_ARG;
    if (seq_len > CS_MAX_SEQ_LEN) return CS_ERR_OOM;
    const int64_t rows = static_cast<int64_t>(batch) * heads * seq_len;
    if (rows == 0) return CS_OK;
    if (rows > INT64_MAX / 4 / seq_len) return CS_ERR_DIM_MISMATCH;
    if (!scores || !out) return CS_ERR_INVALID_ARG;
    const int64_t bytes = rows * seq_len * 4;
    if (out != scores && ranges_overlap(out, bytes, scores, bytes))
        return CS_ERR_INVALID_ARG;
    if (mask && ranges_overlap(mask, static_cast<int64_t>(batch) * seq_len * 4,
                               out, bytes))
        return CS_ERR_INVALID_ARG;
    return CS_OK;
}

cs_status cs_plan_attention_host(int32_t batch, int32_t heads,
                                 int32_t seq_len, int32_t aligned,
                                 const cs_options* options, int32_t sm_count,
                                 int32_t smem_per_block_optin,
                                 int32_t smem_per_sm, cs_plan* plan) {
    if (!plan) return CS_ERR_INVALID_ARG;
    if (batch < 0 || heads < 0 || seq_len < 1) return CS_ERR_DIM_MISMATCH;
    if (seq_len > CS_MAX_SEQ_LEN) return CS_ERR_OOM;
    if (aligned != 0 && aligned != 1) return CS_ERR_INVALID_ARG;
    if (sm_count < 1 || smem_per_block_optin < 1 || smem_per_sm < 1)
        return CS_ERR_INVALID_ARG;
    const cs_options o = options ? *options : cs_options{};
    return plan_attention(batch, heads, seq_len, aligned, o, sm_count,
                          smem_per_block_optin, smem_per_sm, plan);
}

cs_status cs_plan_attention_launch(int32_t batch, int32_t heads,
                                   int32_t seq_len, int32_t aligned,
                                   const cs_options* options, cs_plan* plan) {
    DeviceInfo* d = nullptr;
    const cs_status st = device_info(&d);
    if (st != CS_OK) return st;
    return cs_plan_attention_host(batch, heads, seq_len, aligned, options,
                                  d->sm_count, d->smem_optin, d->smem_per_sm,
                                  plan);
}

cs_status cs_attention_softmax_ex(const float* scores, float* out,
                                  const float* mask, int32_t batch,
                                  int32_t heads, int32_t seq_len,
                                  int32_t causal, const cs_options* options,
                                  void* stream) {
    cs_status st = cs_check_attention_args(scores, out, mask, batch, heads,
                                           seq_len, causal);
    if (st != CS_OK) return st;
    const int64_t rows = static_cast<int64_t>(batch) * heads * seq_len;
    if (rows == 0) return CS_OK;
    DeviceInfo* d = nullptr;
    st = device_info(&d);
    if (st != CS_OK) return st;
    const bool aligned = seq_len % 4 == 0 &&
                         (reinterpret_cast<uintptr_t>(scores) & 15) == 0 &&
                         (reinterpret_cast<uintptr_t>(out) & 15) == 0;
    cs_plan p;
    st = cs_plan_attention_host(batch, heads, seq_len, aligned ? 1 : 0,
                                options, d->sm_count, d->smem_optin,
                                d->smem_per_sm, &p);
    if (st != CS_OK) return st;
    cs::AttnTask task;
    task.scores = scores;
    task.out = out;
    task.mask = mask;
    task.err = d->err;
    task.rows = rows;
    task.heads = heads;
    task.seq_len = seq_len;
    task.causal = causal;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (p.variant == CS_VARIANT_ROWGROUP)
        e = cs::launch_attention_rowgroup(task, p.lanes_per_row,
                                          p.elems_per_lane, s);
    else
        e = cs::launch_attention_cta(task, p.threads_per_cta, p.smem_bytes,
                                     p.grid_ctas, s);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return CS_ERR_CUDA;
    }
    return CS_OK;
}

cs_status cs_attention_softmax(const float* scores, float* out,
                               const float* mask, int32_t batch,
                               int32_t heads, int32_t seq_len,
                               int32_t causal, void* stream) {
    return cs_attention_softmax_ex(scores, out, mask, batch, heads, seq_len,
                                   causal, nullptr, stream);
}

cs_status cs_check_biencoder_args(const float* query,
                                  const float* context_keys,
                                  const float* context_values,
                                  const float* output, int32_t batch_size,
                                  int32_t query_len, int32_t context_len,
                                  int32_t d_head, int32_t num_heads,
                                  float scale, float entropy_bound,
                                  float t_min, float t_max, int32_t max_iter,
                                  const float* attn_out, const float* t_out) {
    if (batch_size < 0 || query_len < 0 || num_heads < 0 || context_len < 1 ||
        d_head < 1)
        return CS_ERR_DIM_MISMATCH;
    if (context_len > cs::kBiencMaxContext || d_head > cs::kBiencMaxDHead)
        return CS_ERR_OOM;
    if (d_head % 4 != 0) return CS_ERR_INVALID_ARG;
    if (!isfinite(scale)) return CS_ERR_INVALID_ARG;
    // The search parameters, as for cs_constrained_softmax.
    const cs_status st = cs_check_args(nullptr, nullptr, 0, context_len,
                                       entropy_bound, t_min, t_max, max_iter,
                                       nullptr);
    if (st != CS_OK) return st;
    const int64_t bh = static_cast<int64_t>(batch_size) * num_heads;
    const int64_t rows = bh * query_len;
    if (rows == 0) return CS_OK;
    if (!query || !context_keys || !context_values || !output)
        return CS_ERR_INVALID_ARG;
    const void* ptrs[4] = {query, context_keys, context_values, output};
    for (const void* ptr : ptrs)
        if (reinterpret_cast<uintptr_t>(ptr) & 15) return CS_ERR_INVALID_ARG;
    const int64_t qb = rows * d_head * 4;
    const int64_t kb = bh * context_len * d_head * 4;
    if (ranges_overlap(output, qb, query, qb) ||
        ranges_overlap(output, qb, context_keys, kb) ||
        ranges_overlap(output, qb, context_values, kb))
        return CS_ERR_INVALID_ARG;
    const int64_t ab = rows * context_len * 4;
    if (attn_out && (ranges_overlap(attn_out, ab, output, qb) ||
                     ranges_overlap(attn_out, ab, query, qb) ||
                     ranges_overlap(attn_out, ab, context_keys, kb) ||
                     ranges_overlap(attn_out, ab, context_values, kb)))
        return CS_ERR_INVALID_ARG;
    if (t_out && (ranges_overlap(t_out, rows * 4, output, qb) ||
                  ranges_overlap(t_out, rows * 4, query, qb) ||
                  ranges_overlap(t_out, rows * 4, context_keys, kb) ||
                  ranges_overlap(t_out, rows * 4, context_values, kb) ||
                  (attn_out && ranges_overlap(t_out, rows * 4, attn_out, ab))))
        return CS_ERR_INVALID_ARG;
    return CS_OK;
}

cs_status cs_plan_biencoder_host(int32_t batch_size, int32_t query_len,
                                 int32_t context_len, int32_t d_head,
                                 int32_t num_heads, const cs_options* options,
                                 int32_t smem_per_block_optin, cs_plan* plan) {
    if (!plan) return CS_ERR_INVALID_ARG;
    if (batch_size < 0 || query_len < 0 || num_heads < 0 || context_len < 1 ||
        d_head < 1)
        return CS_ERR_DIM_MISMATCH;
    if (context_len > cs::kBiencMaxContext || d_head > cs::kBiencMaxDHead)
        return CS_ERR_OOM;
    if (d_head % 4 != 0) return CS_ERR_INVALID_ARG;
    const cs_options o = options ? *options : cs_options{};
    if (o.threads != 0 || o.strict != 0 || o.evals_out) return CS_ERR_INVALID_ARG;
    // G lanes a query row, each holding `keys` context items: by default
    // sixteen (the fewest lanes, so the fewest copies of each row's search
    // bookkeeping); a forced G holds eight when that covers the context.
    int G = 0;
    if (o.variant == CS_VARIANT_AUTO ||
        (o.variant == CS_VARIANT_FUSED && o.param == 0)) {
        if (o.param != 0) return CS_ERR_INVALID_ARG;
        G = 1;
        while (16 * G < context_len) G <<= 1;
    } else if (o.variant == CS_VARIANT_ROWGROUP || o.variant == CS_VARIANT_FUSED) {
        G = o.param;
        if (G < 1 || G > kRowgroupMaxLanes || (G & (G - 1)))
            return CS_ERR_INVALID_ARG;
        if (16 * G < context_len) return CS_ERR_OOM;
    } else {
        return CS_ERR_INVALID_ARG;
    }
    const int keys = (o.variant == CS_VARIANT_AUTO ||
                      (o.variant == CS_VARIANT_FUSED && o.param == 0) ||
                      8 * G < context_len) ? 16 : 8;
    // Step 3 on the tensor cores (a second kernel) unless forced fused:
    // for head sizes up to kPvMaxD and contexts no longer than the head, so
    // that the weights fit in the output's own rows when attn_out is not
    // requested.
    const bool tc = o.variant != CS_VARIANT_FUSED && d_head <= cs::kPvMaxD &&
                    context_len <= d_head &&
                    cs::pv_smem_bytes(context_len, d_head) <= smem_per_block_optin;
    const int64_t smem = tc ? cs::bienc_search_smem_bytes(context_len, d_head, G)
                            : cs::bienc_smem_bytes(context_len, d_head, G);
    if (smem > smem_per_block_optin) return CS_ERR_OOM;
    const int64_t rows_per_tile = cs::bienc_threads(G) / G;
    const int64_t tiles = ceil_div(query_len, rows_per_tile);
    const int64_t per = cs::bienc_tiles_per_cta(query_len, G);
    const int64_t grid = static_cast<int64_t>(batch_size) * num_heads *
                         ceil_div(tiles, per);
    if (grid > kMaxGridX) return CS_ERR_DIM_MISMATCH;
    *plan = cs_plan{};
    plan->variant = CS_VARIANT_ROWGROUP;
    plan->lanes_per_row = G;
    plan->elems_per_lane = keys;
    plan->threads_per_cta = cs::bienc_threads(G);
    plan->smem_bytes = static_cast<int32_t>(smem);
    plan->grid_ctas = grid;
    plan->staged_tensors = tc ? 2 : 3;
    plan->tensor_cores = tc ? 1 : 0;
    return CS_OK;
}

cs_status cs_biencoder_attention_ex(const float* query,
                                    const float* context_keys,
                                    const float* context_values,
                                    float* output, int32_t batch_size,
                                    int32_t query_len, int32_t context_len,
                                    int32_t d_head, int32_t num_heads,
                                    float scale, float entropy_bound,
                                    float t_min, float t_max,
                                    int32_t max_iter, float* attn_out,
                                    float* t_out, const cs_options* options,
                                    void* stream) {
    cs_status st = cs_check_biencoder_args(
        query, context_keys, context_values, output, batch_size, query_len,
        context_len, d_head, num_heads, scale, entropy_bound, t_min, t_max,
        max_iter, attn_out, t_out);
    if (st != CS_OK) return st;
    const int64_t bh = static_cast<int64_t>(batch_size) * num_heads;
    if (bh * query_len == 0) return CS_OK;
    DeviceInfo* d = nullptr;
    st = device_info(&d);
    if (st != CS_OK) return st;
    cs_plan p;
    st = cs_plan_biencoder_host(batch_size, query_len, context_len, d_head,
                                num_heads, options, d->smem_optin, &p);
    if (st != CS_OK) return st;
    cs::BiencTask task;
    task.q = query;
    task.k = context_keys;
    task.v = context_values;
    task.out = output;
    task.attn_out = attn_out;
    task.t_out = t_out;
    task.err = d->err;
    task.BH = static_cast<int32_t>(bh);
    task.Q = query_len;
    task.K = context_len;
    task.D = d_head;
    task.scale = scale;
    task.entropy_bound = entropy_bound;
    task.t_min = t_min;
    task.hi0 = t_max < 1.0f ? t_max : 1.0f;
    task.max_iter = max_iter;
    task.p_out = nullptr;
    task.p_stride = 0;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (p.tensor_cores) {
        // Steps 1-2 write the weights (to attn_out, or to the first
        // context_len floats of each output row), then the tensor-core
        // kernel turns them into the output on the same stream.
        task.p_out = attn_out ? attn_out : output;
        task.p_stride = attn_out ? context_len : d_head;
        e = cs::launch_bienc(task, p.lanes_per_row, p.elems_per_lane, p.smem_bytes, s);
        if (e == cudaSuccess) {
            cs::PvTask pv;
            pv.p = task.p_out;
            pv.p_stride = task.p_stride;
            pv.v = context_values;
            pv.out = output;
            pv.err = d->err;
            pv.BH = task.BH;
            pv.Q = query_len;
            pv.K = context_len;
            pv.D = d_head;
            pv.wait_limit_cycles = cs::kWaitLimitCycles;
            e = cs::launch_bienc_pv(pv, d->sm_count, s);
        }
    } else {
        e = cs::launch_bienc(task, p.lanes_per_row, p.elems_per_lane, p.smem_bytes, s);
    }
    if (e != cudaSuccess) {
        cudaGetLastError();
        return CS_ERR_CUDA;
    }
    return CS_OK;
}

cs_status cs_biencoder_attention(const float* query,
                                 const float* context_keys,
                                 const float* context_values, float* output,
                                 int32_t batch_size, int32_t query_len,
                                 int32_t context_len, int32_t d_head,
                                 int32_t num_heads, float scale,
                                 float entropy_bound, void* stream) {
    return cs_biencoder_attention_ex(query, context_keys, context_values,
                                     output, batch_size, query_len,
                                     context_len, d_head, num_heads, scale,
                                     entropy_bound, 0.01f, 10.0f, 20, nullptr,
                                     nullptr, nullptr, stream);
}

int32_t cs_probe_ex2_sink_floats(void) {
    DeviceInfo* d = nullptr;
    if (device_info(&d) != CS_OK) return -1;
    return d->sm_count * kProbeBlocksPerSm * kProbeThreads;
}

cs_status cs_probe_ex2(float* sink, int32_t iters, int64_t* ex2_count,
                       void* stream) {
    if (!sink || !ex2_count || iters < 1) return CS_ERR_INVALID_ARG;
    DeviceInfo* d = nullptr;
    const cs_status st = device_info(&d);
    if (st != CS_OK) return st;
    const int blocks = d->sm_count * kProbeBlocksPerSm;
    const cudaError_t e = cs::launch_probe_ex2(
        sink, iters, blocks, kProbeThreads, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) {
        cudaGetLastError();
        return CS_ERR_CUDA;
    }
    *ex2_count = static_cast<int64_t>(blocks) * kProbeThreads * iters *
                 cs::probe_chains();
    return CS_OK;
}

cs_status cs_test_wait_timeout(int64_t limit_ns, void* stream) {
    if (limit_ns < 1 || limit_ns > 10000000000ll) return CS_ERR_INVALID_ARG;
    DeviceInfo* d = nullptr;
    const cs_status st = device_info(&d);
    if (st != CS_OK) return st;
    // The wait is bounded in SM cycles; 2.07 cycles per ns at GB300's
    // maximum clock (a lower clock only lengthens the wait).
    const uint64_t cycles = static_cast<uint64_t>(limit_ns) * 207 / 100;
    const cudaError_t e = cs::launch_wait_timeout(
        d->err, cycles, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) {
        cudaGetLastError();
        return CS_ERR_CUDA;
    }
    return CS_OK;
}

const char* cs_version(void) { return "1.0.0 sm_103a"; }

const char* cs_status_string(cs_status status) {
    switch (status) {
        case CS_OK: return "success";
        case CS_ERR_NAN_INPUT: return "NaN in input";
        case CS_ERR_INF_INPUT: return "Inf in input";
        case CS_ERR_ENTROPY_OVERFLOW: return "entropy bound unsatisfiable";
        case CS_ERR_DIM_MISMATCH: return "dimension mismatch";
        case CS_ERR_OOM: return "row does not fit the shared-memory plan";
        case CS_ERR_INVALID_ARG: return "invalid argument";
        case CS_ERR_CUDA: return "CUDA error";
        case CS_ERR_TIMEOUT: return "device wait timed out";
        default: return "unknown status";
    }
}

}  // extern "C"
