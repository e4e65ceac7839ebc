// Inline-PTX wrappers for the 5th-generation tensor cores of sm_103a
// (tcgen05): tensor-memory allocation, the MMA with operands in shared
// memory and the accumulator in tensor memory, its completion on an
// mbarrier, loads of the accumulator into registers, and tensor copies
// from global into shared memory.  Used by the attn . V step of
// biencoder_attention (k_bienc_pv.cu).
#pragma once

#include <stdint.h>

#include "cs_device.cuh"

namespace csd {

// Allocates ncols (a power of two, 32..512) columns of tensor memory for
// the CTA; executed by one whole warp.  The tensor-memory address is
// written to the shared word at dst.
__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 :: "r"(smem_addr(dst)), "r"(ncols) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

// Frees what tmem_alloc allocated; executed by the same warp.
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;"
                 :: "r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before_sync() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after_sync() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Makes this thread's ordinary shared-memory stores visible to the tensor
// cores (the async proxy).
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Rounds an fp32 to the nearest TF32 (10 stored mantissa bits), returned as
// the fp32 with the low 13 bits zero.
__device__ __forceinline__ float to_tf32(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return __uint_as_float(r);
}

// Shared-memory matrix descriptor, no swizzle (the canonical "interleaved"
// layout of 8-row x 16-byte core matrices): start address, the byte offset
// between core matrices adjacent along K (leading) and along M or N
// (stride), and the descriptor version of this architecture.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo,
                                              uint32_t sbo) {
    return static_cast<uint64_t>((saddr >> 4) & 0x3FFFu) |
           (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16) |
           (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) |
           (1ull << 46);
}

// Instruction descriptor of a dense kind::tf32 MMA with an fp32
// accumulator, both operands TF32 and K-major, M x N.
__host__ __device__ constexpr uint32_t idesc_tf32(int M, int N) {
    return (1u << 4)                                   // D: fp32
         | (2u << 7)                                   // A: TF32
         | (2u << 10)                                  // B: TF32
         | (static_cast<uint32_t>(N >> 3) << 17)
         | (static_cast<uint32_t>(M >> 4) << 24);
}

// D[tmem] (+)= A[smem] . B[smem]^T, issued by one thread.
__device__ __forceinline__ void mma_tf32(uint32_t d_tmem, uint64_t a_desc,
                                         uint64_t b_desc, uint32_t idesc,
                                         bool accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n}"
        :: "r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc),
           "r"(accumulate ? 1u : 0u) : "memory");
}

// The mbarrier at bar receives one arrival when every tcgen05 operation
// this thread issued before has completed.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
        :: "r"(smem_addr(bar)) : "memory");
}

// 16 consecutive 32-bit columns of this thread's tensor-memory lane (the
// warp's quarter of the lanes: lane base 32 (warp % 4)).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    // The load and its wait in one statement, so that no use of the
    // registers can be scheduled between them.
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];\n"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
          "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]),
          "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr) : "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// 2-D tiled copy by the tensor-memory-access unit: the box of the tensor
// map at element coordinates (x, y) into shared memory at sdst (laid out
// and swizzled as the map says), counted in bytes on the mbarrier at bar.
__device__ __forceinline__ void tma_load_2d(void* sdst, const void* tmap, int x,
                                            int y, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];"
        :: "r"(smem_addr(sdst)), "l"(tmap), "r"(x), "r"(y), "r"(smem_addr(bar))
        : "memory");
}

// Shared-memory matrix descriptor of a K-major operand in the 128-byte
// swizzled layout: 8-row groups of 128-byte rows (1024-byte atoms, each
// row's 16-byte units permuted by the row index mod 8), atoms stacked
// along M or N every sbo bytes; the start address may step through an
// atom's row in 32-byte (one K = 8 tf32) increments.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr, uint32_t sbo) {
    return static_cast<uint64_t>((saddr >> 4) & 0x3FFFu) |
           (static_cast<uint64_t>(1u) << 16) |
           (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) |
           (1ull << 46) |
           (2ull << 61);
}

}  // namespace csd
