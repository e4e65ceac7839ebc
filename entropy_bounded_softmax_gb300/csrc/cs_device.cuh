// Device helpers shared by the kernels of libcsoftmax: the ex2/lg2 units,
// mbarriers with bounded waits, DSMEM pushes and
// warp/group reductions.  sm_103a only; inline PTX where CUDA has no
// intrinsic.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "cs_internal.h"

namespace csd {

constexpr float kLog2e = 1.44269504088896341f;
constexpr float kLn2 = 0.693147180559945309f;
// Floor for y = (l - max) * log2(e).  The floor keeps 0 * y finite when
// l - max overflows to -inf.  A floored y contributes exactly 0 to every sum
// and output at every temperature the kernels use: those are at most
// max(1, t_min), the argument check caps t_min at 2^64, so beta >= 2^-64
// and beta * y <= -2^36, whose ex2 is +0 (and so is the exact term).
constexpr float kYFloor = -1.2676506002282294e30f;  // -2^100

// ---------------------------------------------------------------- math units
// 2^x on the MUFU ex2 unit; subnormal results flush to +0.
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// log2(x) on the MUFU lg2 unit.
__device__ __forceinline__ float lg2_approx(float x) {
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// 1/x on the MUFU rcp unit.
__device__ __forceinline__ float rcp_approx(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Packed fp32x2 arithmetic (one instruction for two lanes of data).
__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
    float2 d;
    asm("{\n .reg .b64 ra, rb, rd;\n mov.b64 ra, {%2, %3};\n"
        " mov.b64 rb, {%4, %5};\n mul.rn.f32x2 rd, ra, rb;\n"
        " mov.b64 {%0, %1}, rd;\n}"
        : "=f"(d.x), "=f"(d.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}

__device__ __forceinline__ float2 add2(float2 a, float2 b) {
    float2 d;
    asm("{\n .reg .b64 ra, rb, rd;\n mov.b64 ra, {%2, %3};\n"
        " mov.b64 rb, {%4, %5};\n add.rn.f32x2 rd, ra, rb;\n"
        " mov.b64 {%0, %1}, rd;\n}"
        : "=f"(d.x), "=f"(d.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}

__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
    float2 d;
    asm("{\n .reg .b64 ra, rb, rc, rd;\n mov.b64 ra, {%2, %3};\n"
        " mov.b64 rb, {%4, %5};\n mov.b64 rc, {%6, %7};\n"
        " fma.rn.f32x2 rd, ra, rb, rc;\n mov.b64 {%0, %1}, rd;\n}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}

// Accumulators of S = sum 2^(beta y) and V = sum y 2^(beta y), four lanes
// each as two packed pairs.
struct SV4 {
    float2 s01, s23, v01, v23;
    __device__ __forceinline__ void zero() {
        s01 = s23 = v01 = v23 = make_float2(0.f, 0.f);
    }
    // Adds the four classes of y at inverse temperature beta (b2 = {beta,
    // beta}).
    __device__ __forceinline__ void add(float4 y, float2 b2) {
        const float2 y01 = make_float2(y.x, y.y);
        const float2 y23 = make_float2(y.z, y.w);
        const float2 x01 = mul2(y01, b2);
        const float2 x23 = mul2(y23, b2);
        const float2 e01 = make_float2(ex2(x01.x), ex2(x01.y));
        const float2 e23 = make_float2(ex2(x23.x), ex2(x23.y));
        s01 = add2(s01, e01);
        s23 = add2(s23, e23);
        v01 = fma2(e01, y01, v01);
        v23 = fma2(e23, y23, v23);
    }
    __device__ __forceinline__ float2 total() const {
        const float2 s = add2(s01, s23);
        const float2 v = add2(v01, v23);
        return make_float2(s.x + s.y, v.x + v.y);
    }
};

// Entropy test without a division: with H = ln 2 (log2 S - beta V / S) and
// S > 0, H > bound  <=>  S (log2 S - bound log2 e) - beta V > 0.
// bound_bits = bound * log2(e).
__device__ __forceinline__ bool entropy_above(float2 sv, float beta,
                                              float bound_bits) {
    const float t = fmaf(sv.x, lg2_approx(sv.x) - bound_bits, -beta * sv.y);
    return t > 0.0f;
}

// ------------------------------------------------------------ shared memory
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 16-byte asynchronous copy global -> shared (L1 bypassed); both addresses
// 16-byte aligned.  Completes, visible to the issuing thread, at its
// cp_async_wait_all().
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;"
                 :: "r"(smem_addr(dst)), "l"(src) : "memory");
}

// As cp_async16, but only the first src_bytes (0..16) bytes are read and
// the rest of the 16 destination bytes are zero-filled (src_bytes = 0
// reads nothing).
__device__ __forceinline__ void cp_async16_zfill(void* dst, const void* src,
                                                 uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;"
                 :: "r"(smem_addr(dst)), "l"(src), "r"(src_bytes) : "memory");
}

// 8-byte asynchronous copy global -> shared (through L1); both addresses
// 8-byte aligned.
__device__ __forceinline__ void cp_async8(void* dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;"
                 :: "r"(smem_addr(dst)), "l"(src) : "memory");
}

__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.wait_all;" ::: "memory");
}

// Barrier among the `count` threads (whole warps) that use barrier `id`
// (1..15; 0 is __syncthreads).
__device__ __forceinline__ void named_barrier(uint32_t id, uint32_t count) {
    asm volatile("bar.sync %0, %1;" :: "r"(id), "r"(count) : "memory");
}

// The same barrier, returning in every participating thread whether v was
// true in all of them.
__device__ __forceinline__ bool named_barrier_and(uint32_t id, uint32_t count,
                                                  bool v) {
    uint32_t r;
    asm volatile(
        "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n"
        " bar.red.and.pred q, %2, %3, p;\n selp.u32 %0, 1, 0, q;\n}"
        : "=r"(r) : "r"(v ? 1u : 0u), "r"(id), "r"(count) : "memory");
    return r != 0;
}

// ------------------------------------------------------------------- inputs
// Logit element types.  fp32 logits are read as they are; bf16 logits (their
// 16-bit patterns) are promoted to fp32 on load, which is exact (a bf16 is
// the top half of the fp32 with the same value), so everything after the
// load is the fp32 operation on the promoted logits.  Loads are streaming
// (read once).  get4 reads 4 consecutive elements from an address aligned
// to 4 elements (16 bytes for fp32, 8 for bf16).
struct InF32 {
    using T = float;
    static constexpr int kBytes = 4;
    static __device__ __forceinline__ float get(const T* p) { return *p; }
    static __device__ __forceinline__ float get_cs(const T* p) { return __ldcs(p); }
    static __device__ __forceinline__ float4 get4(const T* p) {
        return __ldcs(reinterpret_cast<const float4*>(p));
    }
    // Asynchronous copy of 4 elements into a 16-byte shared slot, and the
    // slot's fp32 values once it landed.
    static __device__ __forceinline__ void copy4_async(float4* dst, const T* p) {
        cp_async16(dst, p);
    }
    static __device__ __forceinline__ float4 widen(float4 slot) { return slot; }
};

struct InBF16 {
    using T = unsigned short;
    static constexpr int kBytes = 2;
    static __device__ __forceinline__ float lo(uint32_t u) { return __uint_as_float(u << 16); }
    static __device__ __forceinline__ float hi(uint32_t u) {
        return __uint_as_float(u & 0xffff0000u);
    }
    static __device__ __forceinline__ float get(const T* p) {
        return lo(static_cast<uint32_t>(*p));
    }
    static __device__ __forceinline__ float get_cs(const T* p) {
        return lo(static_cast<uint32_t>(__ldcs(p)));
    }
    static __device__ __forceinline__ float4 get4(const T* p) {
        const uint2 v = __ldcs(reinterpret_cast<const uint2*>(p));
        return make_float4(lo(v.x), hi(v.x), lo(v.y), hi(v.y));
    }
    // The 8 bytes of 4 bf16 go to the first half of the slot; widen()
    // expands them to the slot's four fp32 values.
    static __device__ __forceinline__ void copy4_async(float4* dst, const T* p) {
        cp_async8(dst, p);
    }
    static __device__ __forceinline__ float4 widen(float4 slot) {
        const uint32_t a = __float_as_uint(slot.x), b = __float_as_uint(slot.y);
        return make_float4(lo(a), hi(a), lo(b), hi(b));
    }
};

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;"
                 :: "r"(smem_addr(bar)), "r"(count) : "memory");
}

// Makes mbarrier initialisation visible to the cluster and the async proxy.
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar,
                                                      uint32_t bytes) {
    asm volatile(
        "mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;"
        :: "r"(smem_addr(bar)), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];"
                 :: "r"(smem_addr(bar)) : "memory");
}

// One test of the phase (a thread may be suspended briefly by the hardware
// while the phase is incomplete).  CLUSTER_SCOPE: acquire at cluster scope
// (remote st.async writes); otherwise at CTA scope.
template <bool CLUSTER_SCOPE>
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    if (CLUSTER_SCOPE) {
        asm volatile(
            "{\n .reg .pred p;\n"
            " mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
            " selp.u32 %0, 1, 0, p;\n}"
            : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
    } else {
        asm volatile(
            "{\n .reg .pred p;\n"
            " mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n"
            " selp.u32 %0, 1, 0, p;\n}"
            : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
    }
    return ok != 0;
}

// Waits for the phase with the given parity to complete, for at most
// limit_cycles SM clock cycles (measured with clock64, which costs a few
// cycles to read) and at most 2^31 polls.  Returns false on timeout.
template <bool CLUSTER_SCOPE>
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity,
                                          uint64_t limit_cycles) {
    const uint32_t a = smem_addr(bar);
    if (mbar_try_wait<CLUSTER_SCOPE>(a, parity)) return true;
    const long long c0 = clock64();
    for (uint32_t i = 1; i < (1u << 31); ++i) {
        if (mbar_try_wait<CLUSTER_SCOPE>(a, parity)) return true;
        if (clock64() - c0 > static_cast<long long>(limit_cycles)) return false;
    }
    return false;
}

// ------------------------------------------------------------------ cluster
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// The two halves of cluster_sync(), for work in between: after
// cluster_arrive() and cluster_wait(), every thread of the cluster has
// passed its cluster_arrive() (release / acquire at cluster scope).
__device__ __forceinline__ void cluster_arrive() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_wait() {
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;"
                 : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}

// Writes {a, b} into (possibly remote) shared memory and counts 8
// transaction bytes on the (same CTA's) mbarrier when the write lands.
__device__ __forceinline__ void push_pair(uint32_t dst, float a, float b,
                                          uint32_t bar) {
    asm volatile(
        "st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.f32 "
        "[%0], {%1, %2}, [%3];"
        :: "r"(dst), "f"(a), "f"(b), "r"(bar) : "memory");
}

// --------------------------------------------------------------- reductions
__device__ __forceinline__ float2 warp_sum2(float2 v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        v.x += __shfl_xor_sync(0xffffffffu, v.x, o);
        v.y += __shfl_xor_sync(0xffffffffu, v.y, o);
    }
    return v;
}

__device__ __forceinline__ float2 warp_max2(float2 v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        v.x = fmaxf(v.x, __shfl_xor_sync(0xffffffffu, v.x, o));
        v.y = fmaxf(v.y, __shfl_xor_sync(0xffffffffu, v.y, o));
    }
    return v;
}

// Sets bits in the library's device error word (rare path).
__device__ __forceinline__ void raise_error(unsigned int* err,
                                            unsigned int bits) {
    if (bits) atomicOr(err, bits);
}

}  // namespace csd
