// The temperature search shared by the kernels: the result of the page's
// bisection ("BURT-IMMA CUDA Kernel API Reference", section 2.1 Description
// step 3: max_iter halvings of [t_min, min(1, t_max)], hi moves to an
// infeasible midpoint, lo to a feasible one) computed with few evaluations.
//
// H(T) is nondecreasing in T (section 2.1 step 4), so once evaluations have
// found a feasible A and an infeasible B, every midpoint m <= A is feasible
// and every m >= B infeasible without being evaluated.  The search keeps that
// bracket and replays the bisection's midpoint sequence (same fp32
// arithmetic, same early stop) with the decisions it settles; only
// midpoints inside (A, B) are unknown.  To shrink the bracket it evaluates
// safeguarded Newton points for log H(beta) = log bound (beta = 1/T), the
// bracket's geometric midpoint when Newton leaves it, t_min when the root
// approaches it, and, once Newton has converged, the two ends of the
// bisection path predicted from the Newton point.  When every midpoint is
// settled, the bisection's final lo is known; its S (for the output) comes
// from the evaluation at lo, made in one last round if lo was not evaluated
// already.  The result is the bisection's: each of its decisions is either
// evaluated or implied by evaluations and the monotonicity of H.  A strict
// mode evaluates every unsettled midpoint one at a time instead.
//
// One evaluation at inverse temperature beta yields, over the row's
// y = (l - max) log2 e:  S = sum 2^(beta y),  V = sum y 2^(beta y),
// W = sum y^2 2^(beta y).  Then H = ln2 (log2 S - beta V / S) nats and
// dH/dbeta = -beta ln2^2 (W/S - (V/S)^2).
#pragma once

#include <math.h>

#include "cs_device.cuh"

namespace csd {

constexpr int kMaxPoints = 3;       // temperatures evaluated per round
constexpr int kMaxNewtonRounds = 40;  // then evaluate midpoints one by one

struct SearchCfg {
    float t_min;
    float hi0;          // min(1, t_max)
    float bound;        // nats
    float bound_bits;   // bound * log2 e
    int max_iter;
};

// Midpoint of the bisection, in the fp32 arithmetic every variant uses.
__device__ __forceinline__ float midpoint(float lo, float hi) {
    return 0.5f * (lo + hi);
}

struct BisectPath {
    float lo, hi;
    bool lo_eval;      // lo was set by a (settled) feasible decision
    bool settled;      // every decision was settled
    float unsettled;   // first unsettled midpoint (when !settled)
};

// Replays the bisection.  Decisions: m >= B infeasible, m <= A feasible
// (A = 0: none known); otherwise [m > Tp] when use_pred, else stop.
__device__ __forceinline__ BisectPath replay(const SearchCfg& c, float A,
                                             float B, bool use_pred,
                                             float Tp) {
    BisectPath p{c.t_min, c.hi0, false, true, 0.0f};
    bool hi_eval = c.hi0 == 1.0f;
    for (int k = 0; k < c.max_iter; ++k) {
        const float m = midpoint(p.lo, p.hi);
        if ((m == p.lo && p.lo_eval) || (m == p.hi && hi_eval)) break;
        bool inf;
        if (m >= B) {
            inf = true;
        } else if (A > 0.0f && m <= A) {
            inf = false;
        } else if (use_pred) {
            inf = m > Tp;
        } else {
            p.settled = false;
            p.unsettled = m;
            return p;
        }
        if (inf) {
            p.hi = m;
            hi_eval = true;
        } else {
            p.lo = m;
            p.lo_eval = true;
        }
    }
    return p;
}

// Per-row search state; identical in every thread working on the row.
struct Search {
    float A, SA;        // largest feasible T evaluated, its S (A = 0: none)
    float B;            // smallest infeasible T evaluated
    float bc, Hc, dHc;  // Newton anchor: beta, H (nats), dH/dbeta
    float S_tmin;       // S at t_min, if evaluated
    bool tmin_done, tmin_inf;
    bool final_round;   // this round evaluates the final lo
    bool final_check;   // ... which is t_min, never moved: flag if infeasible
    bool done;
    bool strict;        // evaluate unsettled midpoints one by one
    int rounds;
    float T_out, S_out;
    bool overflow;      // section 5.4: even t_min violates the bound
};

__device__ __forceinline__ float entropy_nats(float S, float V, float beta) {
    return kLn2 * (lg2_approx(S) - beta * V * rcp_approx(S));
}

__device__ __forceinline__ float entropy_slope(float S, float V, float W,
                                               float beta) {
    const float is = rcp_approx(S);
    const float ey = V * is;
    return -beta * (kLn2 * kLn2) * fmaxf(W * is - ey * ey, 0.0f);
}

// Starts the search after the T = 1 evaluation (S1, V1, W1), which found
// H(1) > bound.
__device__ __forceinline__ Search search_begin(float S1, float V1, float W1,
                                               bool strict) {
    Search s;
    s.A = 0.0f;
    s.SA = 0.0f;
    s.B = 1.0f;
    s.bc = 1.0f;
    s.Hc = entropy_nats(S1, V1, 1.0f);
    s.dHc = entropy_slope(S1, V1, W1, 1.0f);
    s.S_tmin = 0.0f;
    s.tmin_done = false;
    s.tmin_inf = false;
    s.final_round = false;
    s.final_check = false;
    s.done = false;
    s.strict = strict;
    s.rounds = 0;
    s.T_out = 0.0f;
    s.S_out = 0.0f;
    s.overflow = false;
    return s;
}

// Chooses the temperatures of the next round; returns how many (0: done,
// with T_out, S_out and overflow set).
__device__ __forceinline__ int search_plan(Search& s, const SearchCfg& c,
                                           float (&T)[kMaxPoints]) {
    const BisectPath path = replay(c, s.A, s.B, false, 0.0f);
    if (path.settled) {
        const float lo = path.lo;
        s.T_out = lo;
        if (!path.lo_eval) {
            // lo never moved: it is t_min, whose own evaluation decides the
            // degradation flag (section 5.4).
            if (s.tmin_done) {
                s.S_out = s.S_tmin;
                s.overflow = s.tmin_inf;
                s.done = true;
                return 0;
            }
        } else if (s.A > 0.0f && lo == s.A) {
            s.S_out = s.SA;
            s.done = true;
            return 0;
        } else if (s.tmin_done && lo == c.t_min) {
            s.S_out = s.S_tmin;
            s.done = true;
            return 0;
        }
        s.final_round = true;
        s.final_check = !path.lo_eval;
        T[0] = lo;
        return 1;
    }
    if (s.strict || s.rounds >= kMaxNewtonRounds) {
        T[0] = path.unsettled;
        return 1;
    }
    // Safeguarded Newton for log H = log bound in beta (plain Newton on H
    // when the bound is not positive), kept inside the bracket in beta,
    // (1/B, 1/A) or (1/B, 1/t_min) while no feasible point is known.
    const float b_inf = rcp_approx(s.B);
    const float b_feas = rcp_approx(s.A > 0.0f ? s.A : c.t_min);
    float bn;
    if (c.bound > 0.0f && s.Hc > 0.0f) {
        const float g = lg2_approx(s.Hc) - lg2_approx(c.bound);   // log2 units
        const float gp = s.dHc * rcp_approx(s.Hc) * kLog2e;
        bn = gp < 0.0f ? s.bc - g / gp : NAN;
    } else {
        bn = s.dHc < 0.0f ? s.bc - (s.Hc - c.bound) / s.dHc : NAN;
    }
    if (!(bn > b_inf && bn < b_feas)) bn = sqrtf(b_inf * b_feas);
    float Tn = rcp_approx(bn);
    const float Tlo = s.A > 0.0f ? s.A : c.t_min;
    if (!(Tn > Tlo && Tn < s.B)) {
        // Rounding put the point on an end: take the bracket's midpoint.
        Tn = midpoint(Tlo, s.B);
        if (!(Tn > Tlo && Tn < s.B)) Tn = path.unsettled;
    }
    int np = 0;
    T[np++] = Tn;
    if (!s.tmin_done && s.A == 0.0f && Tn <= 4.0f * c.t_min && Tn != c.t_min &&
        c.t_min < s.B)
        T[np++] = c.t_min;
    if (np == 1 && fabsf(bn - s.bc) <= 1e-3f * s.bc) {
        // Newton has converged: also evaluate the ends of the bisection path
        // it predicts, so the next replay can settle every decision.
        const BisectPath pred = replay(c, s.A, s.B, true, Tn);
        if (pred.lo > s.A && pred.lo < s.B && pred.lo != Tn &&
            pred.lo >= c.t_min)
            T[np++] = pred.lo;
        if (pred.hi > s.A && pred.hi < s.B && pred.hi != Tn && np < kMaxPoints)
            T[np++] = pred.hi;
    }
    return np;
}

// Records the round's evaluations: T[i] at beta[i] = rcp_approx(T[i]) gave
// the row sums S, V, W (arrays of length np).
__device__ __forceinline__ void search_update(Search& s, const SearchCfg& c,
                                              int np,
                                              const float (&T)[kMaxPoints],
                                              const float (&beta)[kMaxPoints],
                                              const float* S, const float* V,
                                              const float* W) {
#pragma unroll
    for (int i = 0; i < kMaxPoints; ++i) {
        if (i >= np) break;
        const bool inf = entropy_above(make_float2(S[i], V[i]), beta[i],
                                       c.bound_bits);
        if (T[i] == c.t_min) {
            s.tmin_done = true;
            s.tmin_inf = inf;
            s.S_tmin = S[i];
        }
        if (inf) {
            if (T[i] < s.B) s.B = T[i];
        } else if (T[i] > s.A) {
            s.A = T[i];
            s.SA = S[i];
        }
    }
    if (s.final_round) {
        s.S_out = S[0];
        s.overflow = s.final_check &&
                     entropy_above(make_float2(S[0], V[0]), beta[0],
                                   c.bound_bits);
        s.done = true;
        return;
    }
    // The Newton anchor moves to the round's first point.
    s.bc = beta[0];
    s.Hc = entropy_nats(S[0], V[0], beta[0]);
    s.dHc = entropy_slope(S[0], V[0], W[0], beta[0]);
    ++s.rounds;
}

}  // namespace csd
