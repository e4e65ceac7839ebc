// Auxiliary kernels: the ex2 throughput probe that sets the roofline of the
// constrained softmax (its hot loop is one ex2 per class per bisection step),
// and the bounded-wait timeout exercise.
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
// wait gives up after limit_ns and the timeout is recorded.
__global__ void wait_timeout_kernel(unsigned int* err, uint64_t limit_ns) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1u);
        fence_mbar_init();
    }
    __syncthreads();
    const bool ok = mbar_wait(&bar, 0u, limit_ns);
    if (!ok && threadIdx.x == 0) raise_error(err, kBitTimeout);
}

}  // namespace

int probe_chains() { return kProbeChains; }

cudaError_t launch_probe_ex2(float* sink, int iters, int blocks, int threads,
                             cudaStream_t stream) {
    probe_ex2_kernel<<<blocks, threads, 0, stream>>>(sink, iters);
    return cudaGetLastError();
}

cudaError_t launch_wait_timeout(unsigned int* err, uint64_t limit_ns,
                                cudaStream_t stream) {
    wait_timeout_kernel<<<1, 32, 0, stream>>>(err, limit_ns);
    return cudaGetLastError();
}

}  // namespace cs
