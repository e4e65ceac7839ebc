// Row-group machinery shared by the kernels that keep a short row in the
// registers of G lanes of a warp (the constrained softmax's row-group
// kernel and the fused biencoder_attention kernel): butterfly reductions
// over the group, the register passes of the search, and the whole
// per-row decision ("BURT-IMMA CUDA Kernel API Reference", section 2.1
// Description steps 1-4 with sections 5.3 and 5.4): the row max, the
// NaN/Inf policy, T = 1, and the grid search of cs_search.cuh.
#pragma once

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

template <int G>
__device__ __forceinline__ float2 group_sum2(float2 v, unsigned mask) {
#pragma unroll
    for (int o = G / 2; o > 0; o >>= 1) {
        v.x += __shfl_xor_sync(mask, v.x, o);
        v.y += __shfl_xor_sync(mask, v.y, o);
    }
    return v;
}

// (S, V) of this lane's classes at inverse temperature beta.
template <int E4>
__device__ __forceinline__ float2 reg_pass(const float4 (&y)[E4], float beta) {
    SV4 acc;
    acc.zero();
    const float2 b2 = make_float2(beta, beta);
#pragma unroll
    for (int i = 0; i < E4; ++i) acc.add(y[i], b2);
    return acc.total();
}

template <int G>
__device__ __forceinline__ float3 group_sum3(float3 v, unsigned mask) {
#pragma unroll
    for (int o = G / 2; o > 0; o >>= 1) {
        v.x += __shfl_xor_sync(mask, v.x, o);
        v.y += __shfl_xor_sync(mask, v.y, o);
        v.z += __shfl_xor_sync(mask, v.z, o);
    }
    return v;
}

// (S, V, W) of this lane's classes at inverse temperature beta, with
// W = sum y^2 2^(beta y) for the Newton slope.  S and V take exactly the
// arithmetic of reg_pass, so a grid point gets the same decision whichever
// pass evaluates it.  UNIT: beta = 1, whose product y * 1 = y is skipped.
template <int E4, bool UNIT = false>
__device__ __forceinline__ float3 reg_pass3(const float4 (&y)[E4], float beta) {
    SV4 acc;
    acc.zero();
    float2 w = make_float2(0.f, 0.f);
    const float2 b2 = make_float2(beta, beta);
#pragma unroll
    for (int i = 0; i < E4; ++i) {
        const float2 y01 = make_float2(y[i].x, y[i].y);
        const float2 y23 = make_float2(y[i].z, y[i].w);
        const float2 x01 = UNIT ? y01 : mul2(y01, b2);
        const float2 x23 = UNIT ? y23 : mul2(y23, b2);
        const float2 e01 = make_float2(ex2(x01.x), ex2(x01.y));
        const float2 e23 = make_float2(ex2(x23.x), ex2(x23.y));
        acc.s01 = add2(acc.s01, e01);
        acc.s23 = add2(acc.s23, e23);
        acc.v01 = fma2(e01, y01, acc.v01);
        acc.v23 = fma2(e23, y23, acc.v23);
        w = fma2(mul2(e01, y01), y01, w);
        w = fma2(mul2(e23, y23), y23, w);
    }
    const float2 sv = acc.total();
    return make_float3(sv.x, sv.y, w.x + w.y);
}

// What a row's search settled on.
struct RowSolution {
    float T_row;      // reported temperature (NaN for a NaN/Inf row)
    float beta_out;   // 1/T of the output
    float inv_s;      // 1/S at that temperature
    unsigned int bits;
    int evals;        // temperatures evaluated (T = 1 and the search)
    bool zero;        // NaN/Inf row: output zeros
};

// The per-row decision for a row held in y[E4] by the G lanes of `gmask`:
// y holds the raw logits (lanes past the row hold -inf), m the lane's max,
// bad the lane's finiteness check (NaN when a logit is NaN or infinite).
// On return y holds (l - max) log2 e (floored), ready for the output pass
// 2^(beta_out y) inv_s.  Every lane of the group returns the same values.
// SPLIT_GRID: two copies of the search, one per grid kind (fewer
// instructions a round, more registers: the row-group instantiations with
// 32 classes a lane keep one copy, where the split spilled; the biencoder
// kernel splits, a few bytes of spills and all, 0.8% faster).
template <int G, int E4, bool SPLIT_GRID = true>
__device__ __forceinline__ RowSolution solve_row(float4 (&y)[E4], float m,
                                                 float bad,
                                                 const SearchCfg& cfg,
                                                 float bound_bits,
                                                 bool strict,
                                                 unsigned gmask) {
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
    int evals = 0;
    float T_row = NAN;
    float beta_out = 0.0f, inv_s = 0.0f;
    if (row_code != 0) {
        bits = row_code == 2 ? kBitNan : kBitInf;
    } else {
        // (l - m) log2 e, floored, two lanes per packed operation (the
        // same roundings as the scalar subtract and multiply).
        const float2 neg_m = make_float2(-m, -m);
        const float2 l2e = make_float2(kLog2e, kLog2e);
#pragma unroll
        for (int i = 0; i < E4; ++i) {
            const float2 a = mul2(add2(make_float2(y[i].x, y[i].y), neg_m), l2e);
            const float2 b = mul2(add2(make_float2(y[i].z, y[i].w), neg_m), l2e);
            y[i] = make_float4(fmaxf(a.x, kYFloor), fmaxf(a.y, kYFloor),
                               fmaxf(b.x, kYFloor), fmaxf(b.y, kYFloor));
        }
        const float3 r1 = group_sum3<G>(reg_pass3<E4, true>(y, 1.0f), gmask);
        evals = 1;
        float2 sv = make_float2(r1.x, r1.y);
        if (!entropy_above(sv, 1.0f, bound_bits)) {
            T_row = 1.0f;
            beta_out = 1.0f;
            inv_s = 1.0f / sv.x;
        } else {
            bool over = false;
            int n_search = 0;
            auto eval3 = [&](float b) { return group_sum3<G>(reg_pass3<E4>(y, b), gmask); };
            auto eval2 = [&](float b) { return group_sum2<G>(reg_pass<E4>(y, b), gmask); };
            if (SPLIT_GRID) {
                // One search instance per grid kind (max_iter above 24 or
                // not), so that its loops carry no branch on the kind.
                if (cfg.g.fine)
                    narrow_search<kGridFine>(cfg, r1.x, r1.y, r1.z, strict, eval3,
                                             eval2, T_row, beta_out, inv_s, over,
                                             n_search);
                else
                    narrow_search<kGridExact>(cfg, r1.x, r1.y, r1.z, strict, eval3,
                                              eval2, T_row, beta_out, inv_s, over,
                                              n_search);
            } else {
                narrow_search<kGridAny>(cfg, r1.x, r1.y, r1.z, strict, eval3, eval2,
                                        T_row, beta_out, inv_s, over, n_search);
            }
            evals += n_search;
            if (over) bits |= kBitOverflow;
        }
    }
    RowSolution r;
    r.T_row = T_row;
    r.beta_out = beta_out;
    r.inv_s = inv_s;
    r.bits = bits;
    r.evals = evals;
    r.zero = row_code != 0;
    return r;
}

}  // namespace
}  // namespace cs
