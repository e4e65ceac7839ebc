// Row-group kernel for narrow rows (mixture-of-experts router widths):
// G lanes of a warp share one row and each lane keeps its 4*E4 classes in
// registers for the whole search, so the row is read from HBM once (128-bit
// streaming loads) and written once (128-bit streaming stores).
//
// Method: "BURT-IMMA CUDA Kernel API Reference", section 2.1
// `constrained_softmax`, Description steps 1-4, with sections 5.3 and 5.4;
// the steps are the same as in the cluster kernel: max once, y = (l - m)
// log2 e, then the temperature search of cs_search.cuh, whose rounds are
// register passes giving S = sum 2^(beta y), V = sum y 2^(beta y) and
// W = sum y^2 2^(beta y) at 1-3 temperatures.  The per-round reduction is a
// butterfly over the G lanes (all lanes end with bit-identical sums, so
// they take the same decisions).
#include <math.h>

#include "cs_search.cuh"

namespace cs {
namespace {

using namespace csd;

template <int G>
__device__ __forceinline__ float2 group_max2(float2 v, unsigned mask) {
#pragma unroll
    for (int o = G / 2; o > 0; o >>= 1) {
        v.x = fmaxf(v.x, __shfl_xor_sync(mask, v.x, o));
        v.y = fmaxf(v.y, __shfl_xor_sync(mask, v.y, o));
    }
    return v;
}

// (S, V, W) of this lane's classes at P inverse temperatures, into
// out = {S_0, V_0, W_0, S_1, ...}.
template <int E4, int P>
__device__ __forceinline__ void reg_eval(const float4 (&y)[E4],
                                         const float (&beta)[kMaxPoints],
                                         float (&out)[3 * P]) {
#pragma unroll
    for (int p = 0; p < P; ++p) {
        const float2 b2 = make_float2(beta[p], beta[p]);
        float2 s = make_float2(0.f, 0.f), v = s, w = s;
#pragma unroll
        for (int i = 0; i < E4; ++i) {
            const float2 y01 = make_float2(y[i].x, y[i].y);
            const float2 y23 = make_float2(y[i].z, y[i].w);
            const float2 x01 = mul2(y01, b2);
            const float2 x23 = mul2(y23, b2);
            const float2 e01 = make_float2(ex2(x01.x), ex2(x01.y));
            const float2 e23 = make_float2(ex2(x23.x), ex2(x23.y));
            const float2 ey01 = mul2(e01, y01);
            const float2 ey23 = mul2(e23, y23);
            s = add2(s, add2(e01, e23));
            v = add2(v, add2(ey01, ey23));
            w = fma2(ey01, y01, w);
            w = fma2(ey23, y23, w);
        }
        out[3 * p] = s.x + s.y;
        out[3 * p + 1] = v.x + v.y;
        out[3 * p + 2] = w.x + w.y;
    }
}

template <int G, int NV>
__device__ __forceinline__ void group_sum(float (&a)[NV], unsigned mask) {
#pragma unroll
    for (int o = G / 2; o > 0; o >>= 1) {
#pragma unroll
        for (int i = 0; i < NV; ++i) a[i] += __shfl_xor_sync(mask, a[i], o);
    }
}

// One search round of the row with P temperatures (all lanes of the group).
template <int G, int E4, int P>
__device__ __forceinline__ void group_round(Search& st, const SearchCfg& cfg,
                                            const float (&T)[kMaxPoints],
                                            const float4 (&y)[E4],
                                            unsigned gmask, int np) {
    float beta[kMaxPoints];
#pragma unroll
    for (int p = 0; p < kMaxPoints; ++p) beta[p] = p < P ? rcp_approx(T[p]) : 1.0f;
    float a[3 * P];
    reg_eval<E4, P>(y, beta, a);
    group_sum<G, 3 * P>(a, gmask);
    float S[kMaxPoints], V[kMaxPoints], W[kMaxPoints];
#pragma unroll
    for (int p = 0; p < kMaxPoints; ++p) {
        const int q = p < P ? p : 0;
        S[p] = p < P ? a[3 * q] : 1.0f;
        V[p] = p < P ? a[3 * q + 1] : 0.0f;
        W[p] = p < P ? a[3 * q + 2] : 0.0f;
    }
    search_update(st, cfg, np, T, beta, S, V, W);
}

template <int G, int E4>
__global__ void __launch_bounds__(256, E4 <= 2 ? 4 : (E4 <= 4 ? 3 : 2))
rowgroup_kernel(RowTask t, int vec) {
    const int lane = threadIdx.x & 31;
    const int sub = lane & (G - 1);
    const unsigned gmask =
        G == 32 ? 0xffffffffu : (((1u << G) - 1u) << (lane & ~(G - 1)));
    const int C = t.num_classes;
    const int Q = (C + 3) >> 2;  // float4 slots per row
    const SearchCfg cfg{t.t_min, t.hi0, t.entropy_bound,
                        t.entropy_bound * kLog2e, t.max_iter};
    const int64_t groups_per_grid =
        (static_cast<int64_t>(gridDim.x) * blockDim.x) / G;

    for (int64_t row = (static_cast<int64_t>(blockIdx.x) * blockDim.x +
                        threadIdx.x) / G;
         row < t.batch; row += groups_per_grid) {
        const float* src = t.logits + row * C;
        float* dst = t.out + row * C;
        float4 y[E4];
        float m = -INFINITY;
        float bad = 0.0f;
        if (vec) {
            const float4* s4 = reinterpret_cast<const float4*>(src);
#pragma unroll
            for (int i = 0; i < E4; ++i) {
                const int q = i * G + sub;
                if (q < Q) {
                    y[i] = __ldcs(s4 + q);
                    m = fmaxf(m, fmaxf(fmaxf(y[i].x, y[i].y),
                                       fmaxf(y[i].z, y[i].w)));
                    bad = fmaf(y[i].x, 0.f, bad);
                    bad = fmaf(y[i].y, 0.f, bad);
                    bad = fmaf(y[i].z, 0.f, bad);
                    bad = fmaf(y[i].w, 0.f, bad);
                } else {
                    y[i] = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
                }
            }
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
                        e[k] = __ldcs(src + j);
                        m = fmaxf(m, e[k]);
                        bad = fmaf(e[k], 0.f, bad);
                    }
                }
                y[i] = make_float4(e[0], e[1], e[2], e[3]);
            }
        }
        float code = 0.0f;
        if (bad != bad) {
            code = 1.0f;
#pragma unroll
            for (int i = 0; i < E4; ++i) {
                if (isnan(y[i].x) || isnan(y[i].y) || isnan(y[i].z) ||
                    isnan(y[i].w))
                    code = 2.0f;
            }
        }
        const float2 mc = group_max2<G>(make_float2(m, code), gmask);
        m = mc.x;
        const int row_code = static_cast<int>(mc.y);

        unsigned int bits = 0;
        float T_row = NAN;
        float beta_out = 0.0f, inv_s = 0.0f;
        if (row_code != 0) {
            bits = row_code == 2 ? kBitNan : kBitInf;
        } else {
#pragma unroll
            for (int i = 0; i < E4; ++i) {
                y[i].x = fmaxf((y[i].x - m) * kLog2e, kYFloor);
                y[i].y = fmaxf((y[i].y - m) * kLog2e, kYFloor);
                y[i].z = fmaxf((y[i].z - m) * kLog2e, kYFloor);
                y[i].w = fmaxf((y[i].w - m) * kLog2e, kYFloor);
            }
            float s1[3];
            {
                const float one[kMaxPoints] = {1.0f, 1.0f, 1.0f};
                reg_eval<E4, 1>(y, one, s1);
            }
            group_sum<G, 3>(s1, gmask);
            if (!entropy_above(make_float2(s1[0], s1[1]), 1.0f, cfg.bound_bits)) {
                T_row = 1.0f;
                beta_out = 1.0f;
                inv_s = 1.0f / s1[0];
            } else {
                Search st = search_begin(cfg, s1[0], s1[1], s1[2], t.strict != 0);
                if (!(cfg.t_min < cfg.hi0)) {
                    // No interval to halve: T = t_min (section 5.4 check).
                    st.final_round = true;
                    st.final_check = true;
                    st.T_out = cfg.t_min;
                    const float T1[kMaxPoints] = {cfg.t_min, 0.f, 0.f};
                    group_round<G, E4, 1>(st, cfg, T1, y, gmask, 1);
                }
                // The rows of a warp run their rounds together with the
                // warp's largest point count (padding repeats a point), so
                // the warp never executes several round shapes one after
                // the other.
                const unsigned active = __activemask();
                bool running = true;
                while (__any_sync(active, running)) {
                    float T[kMaxPoints];
                    int np = 0;
                    if (running) {
                        np = search_plan(st, cfg, T);
                        if (np == 0) running = false;
                    }
                    const int npw = __reduce_max_sync(active, np);
                    if (npw == 0) break;
                    if (running) {
                        for (int i = np; i < kMaxPoints; ++i) T[i] = T[0];
                        if (npw == 1)
                            group_round<G, E4, 1>(st, cfg, T, y, gmask, np);
                        else if (npw == 2)
                            group_round<G, E4, 2>(st, cfg, T, y, gmask, np);
                        else
                            group_round<G, E4, 3>(st, cfg, T, y, gmask, np);
                        if (st.done) running = false;
                    }
                }
                if (st.overflow) bits |= kBitOverflow;
                T_row = st.T_out;
                beta_out = rcp_approx(st.T_out);
                inv_s = 1.0f / st.S_out;
            }
        }
        const bool zero = row_code != 0;
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
            raise_error(t.err, bits);
        }
    }
}

template <int G>
cudaError_t launch_g(const RowTask& t, int e4, int vec, dim3 grid, dim3 block,
                     cudaStream_t s) {
    switch (e4) {
        case 1: rowgroup_kernel<G, 1><<<grid, block, 0, s>>>(t, vec); break;
        case 2: rowgroup_kernel<G, 2><<<grid, block, 0, s>>>(t, vec); break;
        case 4: rowgroup_kernel<G, 4><<<grid, block, 0, s>>>(t, vec); break;
        case 8: rowgroup_kernel<G, 8><<<grid, block, 0, s>>>(t, vec); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace

constexpr int kRowgroupThreads = 256;
constexpr int64_t kMaxGridX = 2147483647;

cudaError_t launch_rowgroup(const RowTask& t, int lanes_per_row,
                            int elems_per_lane, cudaStream_t stream) {
    const int e4 = elems_per_lane / 4;
    const int C = t.num_classes;
    const bool aligned =
        (C % 4 == 0) && (reinterpret_cast<uintptr_t>(t.logits) % 16 == 0) &&
        (reinterpret_cast<uintptr_t>(t.out) % 16 == 0);
    const int64_t rows_per_block = kRowgroupThreads / lanes_per_row;
    int64_t blocks = (t.batch + rows_per_block - 1) / rows_per_block;
    if (blocks > kMaxGridX) blocks = kMaxGridX;
    const dim3 grid(static_cast<unsigned>(blocks));
    const dim3 block(kRowgroupThreads);
    const int vec = aligned ? 1 : 0;
    switch (lanes_per_row) {
        case 1: return launch_g<1>(t, e4, vec, grid, block, stream);
        case 2: return launch_g<2>(t, e4, vec, grid, block, stream);
        case 4: return launch_g<4>(t, e4, vec, grid, block, stream);
        case 8: return launch_g<8>(t, e4, vec, grid, block, stream);
        case 16: return launch_g<16>(t, e4, vec, grid, block, stream);
        case 32: return launch_g<32>(t, e4, vec, grid, block, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace cs
