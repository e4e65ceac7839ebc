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
// bisection path predicted from the Newton point.  Midpoints that remain
// unsettled after that (they lie where fp32 evaluations of H are within
// rounding of the bound) are evaluated directly, each together with both
// of its possible successors, two bisection levels per round.  The replay
// keeps a cursor, so every decision is taken once.  When every midpoint is
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

// Position of the replayed bisection: its lo and hi, whether each has been
// decided (for the fp32 early stop) and the steps taken.
struct Cursor {
    float lo, hi;
    bool lo_eval, hi_eval;
    int k;
};

__device__ __forceinline__ Cursor cursor_begin(const SearchCfg& c) {
    return Cursor{c.t_min, c.hi0, false, c.hi0 == 1.0f, 0};
}

// Advances the replay while its decisions are settled: m >= B infeasible,
// m <= A feasible (A = 0: none known); with use_pred, the rest by
// [m > Tp].  Returns true and the midpoint in *um if it stopped at an
// unsettled midpoint, false when the bisection is complete.
__device__ __forceinline__ bool advance(Cursor& cu, const SearchCfg& c,
                                        float A, float B, bool use_pred,
                                        float Tp, float* um) {
    while (cu.k < c.max_iter) {
        const float m = midpoint(cu.lo, cu.hi);
        if ((m == cu.lo && cu.lo_eval) || (m == cu.hi && cu.hi_eval)) {
            // The fp32 midpoint repeats a decided end: every further step
            // would repeat that decision.
            cu.k = c.max_iter;
            break;
        }
        bool inf;
        if (m >= B) {
            inf = true;
        } else if (A > 0.0f && m <= A) {
            inf = false;
        } else if (use_pred) {
            inf = m > Tp;
        } else {
            *um = m;
            return true;
        }
        if (inf) {
            cu.hi = m;
            cu.hi_eval = true;
        } else {
            cu.lo = m;
            cu.lo_eval = true;
        }
        ++cu.k;
    }
    return false;
}

// Per-row search state; identical in every thread working on the row.
struct Search {
    Cursor cur;         // the replayed bisection
    float A, SA;        // largest feasible T evaluated, its S (A = 0: none)
    float B;            // smallest infeasible T evaluated
    float bc, Hc, dHc;  // Newton anchor: beta, H (nats), dH/dbeta
    float S_tmin;       // S at t_min, if evaluated
    bool tmin_done, tmin_inf;
    bool final_round;   // this round evaluates the final lo
    bool final_check;   // ... which is t_min, never moved: flag if infeasible
    bool done;
    bool strict;        // evaluate unsettled midpoints one by one
    bool endgame;       // Newton has converged: bisect the unsettled rest
    bool pred_valid;    // pred holds the path predicted at convergence
    Cursor pred;        // ... whose ends are being evaluated this round
    float S_plo;        // S at pred.lo, once evaluated (0: not yet)
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
__device__ __forceinline__ Search search_begin(const SearchCfg& c, float S1,
                                               float V1, float W1,
                                               bool strict) {
    Search s;
    s.cur = cursor_begin(c);
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
    s.endgame = false;
    s.pred_valid = false;
    s.pred = s.cur;
    s.S_plo = 0.0f;
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
    float um = 0.0f;
    if (s.pred_valid) {
        // The path predicted at convergence is the bisection's if its ends
        // were evaluated on the predicted sides: every predicted-feasible
        // midpoint is then <= A and every predicted-infeasible one >= B, so
        // the replay would take exactly the predicted decisions.
        s.pred_valid = false;
        if ((!s.pred.lo_eval || s.A >= s.pred.lo) &&
            (!s.pred.hi_eval || s.B <= s.pred.hi))
            s.cur = s.pred;
    }
    if (!advance(s.cur, c, s.A, s.B, false, 0.0f, &um)) {
        const float lo = s.cur.lo;
        s.T_out = lo;
        if (!s.cur.lo_eval) {
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
        } else if (s.S_plo > 0.0f && lo == s.pred.lo) {
            s.S_out = s.S_plo;
            s.done = true;
            return 0;
        }
        s.final_round = true;
        s.final_check = !s.cur.lo_eval;
        T[0] = lo;
        return 1;
    }
    if (s.strict || s.rounds >= kMaxNewtonRounds) {
        T[0] = um;
        return 1;
    }
    if (s.endgame) {
        // The unsettled midpoint and both midpoints that can follow it.
        int np = 0;
        T[np++] = um;
        const float m_inf = midpoint(s.cur.lo, um);   // if um is infeasible
        const float m_feas = midpoint(um, s.cur.hi);  // if um is feasible
        const float Tlo = s.A > 0.0f ? s.A : 0.0f;
        if (m_inf > Tlo && m_inf < s.B && m_inf != um) T[np++] = m_inf;
        if (m_feas > Tlo && m_feas < s.B && m_feas != um) T[np++] = m_feas;
        return np;
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
        bn = gp < 0.0f ? s.bc - g * rcp_approx(gp) : NAN;
    } else {
        bn = s.dHc < 0.0f ? s.bc - (s.Hc - c.bound) * rcp_approx(s.dHc) : NAN;
    }
    if (!(bn > b_inf && bn < b_feas)) bn = sqrtf(b_inf * b_feas);
    float Tn = rcp_approx(bn);
    const float Tlo = s.A > 0.0f ? s.A : c.t_min;
    if (!(Tn > Tlo && Tn < s.B)) {
        // Rounding put the point on an end: take the bracket's midpoint.
        Tn = midpoint(Tlo, s.B);
        if (!(Tn > Tlo && Tn < s.B)) Tn = um;
    }
    int np = 0;
    T[np++] = Tn;
    if (!s.tmin_done && s.A == 0.0f && Tn <= 4.0f * c.t_min && Tn != c.t_min &&
        c.t_min < s.B)
        T[np++] = c.t_min;
    if (np == 1 && fabsf(bn - s.bc) <= 1e-3f * s.bc) {
        // Newton has converged: also evaluate the ends of the bisection path
        // it predicts, so the next replay can settle every decision.
        Cursor pred = s.cur;
        float dummy;
        advance(pred, c, s.A, s.B, true, Tn, &dummy);
        s.pred = pred;
        s.pred_valid = true;
        if (pred.lo > s.A && pred.lo < s.B && pred.lo != Tn &&
            pred.lo >= c.t_min)
            T[np++] = pred.lo;
        if (pred.hi > s.A && pred.hi < s.B && pred.hi != Tn && np < kMaxPoints)
            T[np++] = pred.hi;
        s.endgame = true;
    }
    return np;
}

// Whether the round just planned is followed by a Newton step, which needs
// the slope (hence W) at the round's first point.
__device__ __forceinline__ bool newton_next(const Search& s) {
    return !s.final_round && !s.strict && !s.endgame &&
           s.rounds + 1 < kMaxNewtonRounds;
}

// Records the round's evaluations: T[i] at beta[i] = rcp_approx(T[i]) gave
// the row sums S, V (arrays of length np) and, when has_w, W[0] at T[0].
__device__ __forceinline__ void search_update(Search& s, const SearchCfg& c,
                                              int np,
                                              const float (&T)[kMaxPoints],
                                              const float (&beta)[kMaxPoints],
                                              const float* S, const float* V,
                                              const float* W, bool has_w) {
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
        if (s.pred_valid && T[i] == s.pred.lo) s.S_plo = S[i];
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
    // The Newton anchor moves to the round's first point (only used when
    // a Newton step follows, which is when W was accumulated).
    if (has_w) {
        s.bc = beta[0];
        s.Hc = entropy_nats(S[0], V[0], beta[0]);
        s.dHc = entropy_slope(S[0], V[0], W[0], beta[0]);
    }
    ++s.rounds;
}

}  // namespace csd
