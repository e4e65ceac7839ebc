// Row-group kernel for narrow rows (mixture-of-experts router widths):
// G lanes of a warp share one row and each lane keeps its 4*E4 classes in
// registers for the whole search, so the row is read from HBM once (128-bit
// streaming loads) and written once (128-bit streaming stores).
//
// Method: "BURT-IMMA CUDA Kernel API Reference", section 2.1
// `constrained_softmax`, Description steps 1-4, with sections 5.3 and 5.4;
// max once, y = (l - m) log2 e, then the bisection itself on the grid of
// cs_search.cuh, one register pass per halving giving S = sum 2^(beta y)
// and V = sum y 2^(beta y),
// H = ln 2 (log2 S - beta V/S).  The per-step reduction is a butterfly over
// the G lanes (all lanes end with bit-identical sums, so they take the same
// decision); H > bound is decided without a division as
// S (log2 S - bound log2 e) - beta V > 0, with log2 on the MUFU lg2 unit.
#include <math.h>

#include "cs_rowgroup.cuh"

namespace cs {
namespace {

using namespace csd;

// At most 64 registers a thread (32 warps per SM, which the latency of each
// row's dependent reduce-and-decide chain needs), or 80 when a lane holds
// 32 classes.
template <int G, int E4, class In>
__global__ void __launch_bounds__(64, E4 >= 8 ? 12 : 16)
rowgroup_kernel(RowTask t, int vec) {
    const int lane = threadIdx.x & 31;
    const int sub = lane & (G - 1);
    const unsigned gmask =
        G == 32 ? 0xffffffffu : (((1u << G) - 1u) << (lane & ~(G - 1)));
    const int C = t.num_classes;
    const int Q = (C + 3) >> 2;  // float4 slots per row
    const float bound_bits = t.entropy_bound * kLog2e;
    const SearchCfg cfg{t.t_min, t.hi0, t.entropy_bound, bound_bits,
                        t.entropy_bound > 0.0f ? lg2_approx(t.entropy_bound) : 0.0f,
                        make_grid(t.t_min, fmaxf(t.hi0, t.t_min), t.max_iter)};
    const int64_t groups_per_grid =
        (static_cast<int64_t>(gridDim.x) * blockDim.x) / G;

    for (int64_t row = (static_cast<int64_t>(blockIdx.x) * blockDim.x +
                        threadIdx.x) / G;
         row < t.batch; row += groups_per_grid) {
        const typename In::T* src = static_cast<const typename In::T*>(t.logits) + row * C;
        float* dst = t.out + row * C;
        float4 y[E4];
        float m = -INFINITY;
        float bad = 0.0f;
        if (vec) {
            // bad becomes NaN if any element is NaN or infinite (x * 0).
            float2 bad2 = make_float2(0.f, 0.f);
            const float2 zero2 = make_float2(0.f, 0.f);
#pragma unroll
            for (int i = 0; i < E4; ++i) {
                const int q = i * G + sub;
                if (q < Q) {
                    y[i] = In::get4(src + 4 * q);
                    m = fmaxf(m, fmaxf(fmaxf(y[i].x, y[i].y),
                                       fmaxf(y[i].z, y[i].w)));
                    bad2 = fma2(make_float2(y[i].x, y[i].y), zero2, bad2);
                    bad2 = fma2(make_float2(y[i].z, y[i].w), zero2, bad2);
                } else {
                    y[i] = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
                }
            }
            bad = bad2.x + bad2.y;
        } else {
#pragma unroll
            for (int i = 0; i < E4; ++i) {
                const int j0 = 4 * (i * G + sub);
                float e[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int j = j0 + k;
                    e[k] = -INFINITY;
                    if (j < C) {
                        e[k] = In::get_cs(src + j);
                        m = fmaxf(m, e[k]);
                        bad = fmaf(e[k], 0.f, bad);
                    }
                }
                y[i] = make_float4(e[0], e[1], e[2], e[3]);
            }
        }
        const RowSolution sol = solve_row<G, E4, (E4 < 8)>(y, m, bad, cfg, bound_bits,
                                                          t.strict != 0, gmask);
        const unsigned int bits = sol.bits;
        const float T_row = sol.T_row;
        const float beta_out = sol.beta_out, inv_s = sol.inv_s;
        const bool zero = sol.zero;
        if (vec) {
            float4* d4 = reinterpret_cast<float4*>(dst);
#pragma unroll
            for (int i = 0; i < E4; ++i) {
                const int q = i * G + sub;
                if (q < Q) {
                    float4 p = make_float4(0.f, 0.f, 0.f, 0.f);
                    if (!zero) {
                        const float2 b2 = make_float2(beta_out, beta_out);
                        const float2 i2 = make_float2(inv_s, inv_s);
                        const float2 x01 = mul2(make_float2(y[i].x, y[i].y), b2);
                        const float2 x23 = mul2(make_float2(y[i].z, y[i].w), b2);
                        const float2 p01 = mul2(make_float2(ex2(x01.x), ex2(x01.y)), i2);
                        const float2 p23 = mul2(make_float2(ex2(x23.x), ex2(x23.y)), i2);
                        p = make_float4(p01.x, p01.y, p23.x, p23.y);
                    }
                    __stcs(d4 + q, p);
                }
            }
        } else {
#pragma unroll
            for (int i = 0; i < E4; ++i) {
                const int j0 = 4 * (i * G + sub);
                const float yy[4] = {y[i].x, y[i].y, y[i].z, y[i].w};
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int j = j0 + k;
                    if (j < C)
                        __stcs(dst + j, zero ? 0.0f : ex2(yy[k] * beta_out) * inv_s);
                }
            }
        }
        if (sub == 0) {
            if (t.t_out) t.t_out[row] = T_row;
            if (t.evals_out) t.evals_out[row] = sol.evals + (zero ? 0 : 1);
            raise_error(t.err, bits);
        }
    }
}

template <int G, class In>
cudaError_t launch_g(const RowTask& t, int e4, int vec, dim3 grid, dim3 block,
                     cudaStream_t s) {
    switch (e4) {
        case 1: rowgroup_kernel<G, 1, In><<<grid, block, 0, s>>>(t, vec); break;
        case 2: rowgroup_kernel<G, 2, In><<<grid, block, 0, s>>>(t, vec); break;
        case 4: rowgroup_kernel<G, 4, In><<<grid, block, 0, s>>>(t, vec); break;
        case 8: rowgroup_kernel<G, 8, In><<<grid, block, 0, s>>>(t, vec); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

template <class In>
cudaError_t launch_in(const RowTask& t, int lanes_per_row, int e4, int vec,
                      dim3 grid, dim3 block, cudaStream_t stream) {
    switch (lanes_per_row) {
        case 1: return launch_g<1, In>(t, e4, vec, grid, block, stream);
        case 2: return launch_g<2, In>(t, e4, vec, grid, block, stream);
        case 4: return launch_g<4, In>(t, e4, vec, grid, block, stream);
        case 8: return launch_g<8, In>(t, e4, vec, grid, block, stream);
        case 16: return launch_g<16, In>(t, e4, vec, grid, block, stream);
        case 32: return launch_g<32, In>(t, e4, vec, grid, block, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

constexpr int kRowgroupThreads = 64;  // as the planner in cs_api.cu
constexpr int64_t kMaxGridX = 2147483647;

cudaError_t launch_rowgroup(const RowTask& t, int lanes_per_row,
                            int elems_per_lane, cudaStream_t stream) {
    const int e4 = elems_per_lane / 4;
    const int C = t.num_classes;
    // Whole float4s of output, and of input (four elements: 16 bytes of
    // fp32, 8 of bf16), when every row starts aligned.
    const uintptr_t in_align = t.in_bf16 ? 8 : 16;
    const bool aligned =
        (C % 4 == 0) && (reinterpret_cast<uintptr_t>(t.logits) % in_align == 0) &&
        (reinterpret_cast<uintptr_t>(t.out) % 16 == 0);
    const int64_t rows_per_block = kRowgroupThreads / lanes_per_row;
    int64_t blocks = (t.batch + rows_per_block - 1) / rows_per_block;
    if (blocks > kMaxGridX) blocks = kMaxGridX;
    const dim3 grid(static_cast<unsigned>(blocks));
    const dim3 block(kRowgroupThreads);
    const int vec = aligned ? 1 : 0;
    return t.in_bf16
        ? launch_in<InBF16>(t, lanes_per_row, e4, vec, grid, block, stream)
        : launch_in<InF32>(t, lanes_per_row, e4, vec, grid, block, stream);
}

}  // namespace cs
