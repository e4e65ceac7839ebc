// Auxiliary kernels: the ex2 throughput probe that sets the roofline of the
// constrained softmax (its hot loop is one ex2 per class per bisection step),
// the atomic read-and-clear of the error word and the bounded-wait timeout
// exercise; plus the per-device cache of kernel shared-memory attributes.
#include <atomic>
#include <mutex>

#include "cs_device.cuh"

namespace cs {
namespace {

using namespace csd;

constexpr int kProbeChains = 8;

// Every thread runs kProbeChains independent chains x <- 2^x - 1, which
// stays in [-1, 0] for x in [-1, 0]; one FADD per ex2.
__global__ void probe_ex2_kernel(float* sink, int iters) {
    float x[kProbeChains];
#pragma unroll
    for (int c = 0; c < kProbeChains; ++c)
        x[c] = -0.001f * static_cast<float>((threadIdx.x + 37 * c) & 511);
    for (int i = 0; i < iters; ++i) {
#pragma unroll
        for (int c = 0; c < kProbeChains; ++c) x[c] = ex2(x[c]) - 1.0f;
    }
    float acc = 0.0f;
#pragma unroll
    for (int c = 0; c < kProbeChains; ++c) acc += x[c];
    sink[blockIdx.x * blockDim.x + threadIdx.x] = acc;
}

// One CTA waits on an mbarrier that nothing ever completes; the bounded
// wait gives up after limit_cycles and the timeout is recorded.
__global__ void wait_timeout_kernel(unsigned int* err, uint64_t limit_cycles) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1u);
        fence_mbar_init();
    }
    __syncthreads();
    const bool ok = mbar_wait<false>(&bar, 0u, limit_cycles);
    if (!ok && threadIdx.x == 0) raise_error(err, kBitTimeout);
}

// Reads and clears the error word in one atomic step, into the word the
// host then copies back: a bit set by a launch on another stream lands
// either in this read or in the word after it, never between the two.
__global__ void take_error_kernel(unsigned int* err, unsigned int* taken) {
    *taken = atomicExch(err, 0u);
}

}  // namespace

int probe_chains() { return kProbeChains; }

cudaError_t launch_take_error(unsigned int* err, unsigned int* taken,
                              cudaStream_t stream) {
    take_error_kernel<<<1, 1, 0, stream>>>(err, taken);
    return cudaGetLastError();
}

cudaError_t launch_probe_ex2(float* sink, int iters, int blocks, int threads,
                             cudaStream_t stream) {
    probe_ex2_kernel<<<blocks, threads, 0, stream>>>(sink, iters);
    return cudaGetLastError();
}

cudaError_t launch_wait_timeout(unsigned int* err, uint64_t limit_cycles,
                                cudaStream_t stream) {
    wait_timeout_kernel<<<1, 32, 0, stream>>>(err, limit_cycles);
    return cudaGetLastError();
}

namespace {
constexpr int kMaxDevices = 64;
constexpr int kSlots = 56;
// Largest MaxDynamicSharedMemorySize set so far, per device and kernel.
std::atomic<int> g_smem_set[kMaxDevices][kSlots];
std::mutex g_smem_mu;
}  // namespace

cudaError_t ensure_smem_attribute(const void* func, int slot, int bytes,
                                  bool cluster) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices || slot < 0 || slot >= kSlots)
        return cudaErrorInvalidValue;
    if (g_smem_set[dev][slot].load(std::memory_order_acquire) >= bytes)
        return cudaSuccess;
    std::lock_guard<std::mutex> lock(g_smem_mu);
    if (g_smem_set[dev][slot].load(std::memory_order_relaxed) >= bytes)
        return cudaSuccess;
    e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             bytes);
    if (e != cudaSuccess) return e;
    if (cluster) {
        e = cudaFuncSetAttribute(
            func, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
    }
    g_smem_set[dev][slot].store(bytes, std::memory_order_release);
    return cudaSuccess;
}

}  // namespace cs
