// The temperature search shared by the kernels: the result of the page's
// bisection ("BURT-IMMA CUDA Kernel API Reference", section 2.1 Description
// step 3: max_iter halvings of [t_min, min(1, t_max)], hi moves to an
// infeasible midpoint, lo to a feasible one).
//
// The grid.  After K = max_iter halvings every point the bisection can
// reach is lo0 + j (hi0 - lo0) / 2^K for an integer j in [0, 2^K]
// (lo0 = t_min, hi0 = min(1, t_max)); the kernels use those exact dyadic
// points, rounded once to fp32, rather than repeated fp32 halving (the
// page gives no precision for mid; an fp64 bisection's midpoints are the
// same dyadic points).  For K > 24 the points are closer together than
// fp32 resolves over most of the range, and the grid is the fp32 numbers
// of [lo0, hi0] themselves (index = bit-pattern offset from lo0).  A
// halving is then an integer midpoint of a bracket of indices [jl, jh]:
// jl feasible (or 0, t_min, not evaluated), jh infeasible (or the top,
// hi0, which the bisection never evaluates).
//
// The result.  H(T) is nondecreasing in T (section 2.1 step 4), so the
// bisection's final lo is the largest grid point whose H is within the
// bound (t_min if none): the bracket can be closed from evaluations inside
// it in any order, and once jh = jl + 1 the result is G(jl).  The default
// search therefore evaluates safeguarded Newton points for
// log H(beta) = log bound (beta = 1/T) placed on the grid, t_min when the
// root approaches it, then, once Newton has converged, the grid points on
// both sides of the Newton point; if the bracket is still open
// (evaluations of H in fp32 are within rounding of the bound there) it
// gallops away from the end the last round moved, when only one moved,
// with strides growing eightfold, else splits the bracket into quarters,
// two halvings per round.  The cluster kernel's few-row launches take the
// first point instead from a fan of temperatures evaluated with T = 1
// (search_fan).  With one
// point per round (narrow rows, where a pass costs little next to
// divergent bookkeeping) the Newton point is evaluated alone and the
// neighbours follow one by one, with doubling strides.  The strict mode
// evaluates the bracket's midpoint, one halving per round.  The output
// needs S at the result, kept from the evaluation that set jl (or taken in
// one last round at t_min, which also decides the section 5.4 flag).
//
// One evaluation at inverse temperature beta yields, over the row's
// y = (l - max) log2 e:  S = sum 2^(beta y),  V = sum y 2^(beta y),
// W = sum y^2 2^(beta y).  Then H = ln2 (log2 S - beta V / S) nats and
// dH/dbeta = -beta ln2^2 (W/S - (V/S)^2).
#pragma once

#include <math.h>

#include "cs_device.cuh"

namespace csd {

constexpr int kMaxPoints = 3;         // temperatures evaluated per round
constexpr int kMaxNewtonRounds = 40;  // then halve the bracket round by round
constexpr int kMaxExactLevels = 24;   // grid indices exact in fp32 up to 2^24
// Grid kinds for code that fixes the kind at compile time (Grid::at_t).
constexpr int kGridAny = 0;    // branch on Grid::fine
constexpr int kGridExact = 1;  // fine == false
constexpr int kGridFine = 2;   // fine == true

// The bisection's grid (see the file comment).
struct Grid {
    float lo0;       // index 0: t_min
    float step_hi;   // (hi0 - lo0) / 2^K = step_hi + step_lo exactly
    float step_lo;
    float inv_step;  // 1 / step_hi, to place a temperature on the grid
    int lo_bits;     // fine grid: bit pattern of lo0
    int top;         // index of hi0
    bool fine;       // K > 24: every fp32 value of [lo0, hi0] is a point

    // Grid point j, 0 <= j <= top; nondecreasing in j.
    __device__ __forceinline__ float at(int j) const {
        if (fine) return __int_as_float(lo_bits + j);
        const float fj = static_cast<float>(j);
        return fmaf(fj, step_hi, fmaf(fj, step_lo, lo0));
    }
    // An index whose point is within about one step of T (lo0 < T).
    __device__ __forceinline__ int near(float T) const {
        if (fine) return __float_as_int(T) - lo_bits;
        return __float2int_rd(fminf((T - lo0) * inv_step, 2.0e9f));
    }
    // The same for a grid kind chosen at compile time: K = kGridExact or
    // kGridFine (which must equal fine) spares a search loop the branch on
    // every call; kGridAny branches on fine.
    template <int K>
    __device__ __forceinline__ float at_t(int j) const {
        if (K == kGridAny) return at(j);
        if (K == kGridFine) return __int_as_float(lo_bits + j);
        const float fj = static_cast<float>(j);
        return fmaf(fj, step_hi, fmaf(fj, step_lo, lo0));
    }
    template <int K>
    __device__ __forceinline__ int near_t(float T) const {
        if (K == kGridAny) return near(T);
        if (K == kGridFine) return __float_as_int(T) - lo_bits;
        return __float2int_rd(fminf((T - lo0) * inv_step, 2.0e9f));
    }
};

// Grid of max_iter halvings of [lo0, hi0]; requires 0 < lo0 < hi0.
__device__ __forceinline__ Grid make_grid(float lo0, float hi0, int max_iter) {
    Grid g;
    g.lo0 = lo0;
    g.lo_bits = __float_as_int(lo0);
    g.fine = max_iter > kMaxExactLevels;
    if (g.fine) {
        g.top = __float_as_int(hi0) - g.lo_bits;
        g.step_hi = g.step_lo = g.inv_step = 0.0f;
    } else {
        // hi0 - lo0 = s + e exactly (two-sum), scaled by 2^-K exactly.
        const float s = hi0 - lo0;
        const float bv = s - hi0;
        const float e = (hi0 - (s - bv)) + (-lo0 - bv);
        const float scale = __int_as_float((127 - max_iter) << 23);
        g.step_hi = s * scale;
        g.step_lo = e * scale;
        g.inv_step = 1.0f / g.step_hi;
        g.top = 1 << max_iter;
    }
    return g;
}

struct SearchCfg {
    float t_min;
    float hi0;          // min(1, t_max)
    float bound;        // nats
    float bound_bits;   // bound * log2 e
    float lg2_bound;    // log2(bound) when bound > 0
    Grid g;
};

// Per-row state of the bracket search (the cluster kernel); identical in
// every thread that plans for the row.  Kept small: every thread of the
// cluster holds it in registers through the whole search.
struct Search {
    int jl, jh;         // bracket of grid indices
    int jl_prev, jh_prev;  // the bracket when the last round was planned
    int stride;         // the next galloping step
    int rounds;
    uint32_t f;         // kJlEval | kTminInf | ... below
    float SA;           // S at G(jl) when jl was evaluated; S at t_min when
                        // t_min was found infeasible or in the final round
    float b_jl, b_jh;   // beta of the bracket's ends (t_min while unevaluated)
    float bc, Hc, dHc;  // Newton anchor: beta, H (nats), dH/dbeta; with
                        // kFirst, bc is the next round's point instead
};

constexpr uint32_t kJlEval = 1u;     // G(jl) was evaluated feasible
constexpr uint32_t kTminInf = 2u;    // t_min was evaluated infeasible (5.4)
constexpr uint32_t kFinal = 4u;      // this round evaluates t_min for the result
constexpr uint32_t kDone = 8u;
constexpr uint32_t kStrict = 16u;    // halve the bracket one point per round
constexpr uint32_t kEndgame = 32u;   // Newton has converged
constexpr uint32_t kOverflow = 64u;  // section 5.4: even t_min violates the bound
constexpr uint32_t kFirst = 128u;    // the next round evaluates 1/bc (after a fan)

// H (nats) and dH/dbeta at beta from the sums, given ls = log2 S and
// is = 1 / S.
__device__ __forceinline__ float entropy_nats(float ls, float is, float V,
                                              float beta) {
    return kLn2 * (ls - beta * V * is);
}

__device__ __forceinline__ float entropy_slope(float is, float V, float W,
                                               float beta) {
    const float ey = V * is;
    return -beta * (kLn2 * kLn2) * fmaxf(W * is - ey * ey, 0.0f);
}

// Starts the search after the T = 1 evaluation (S1, V1, W1), which found
// H(1) > bound.
__device__ __forceinline__ Search search_begin(const SearchCfg& c, float S1,
                                               float V1, float W1,
                                               bool strict) {
    Search s;
    s.jl = 0;
    s.jh = c.g.top;
    s.jl_prev = s.jl;
    s.jh_prev = s.jh;
    s.stride = 1;
    s.rounds = 0;
    s.f = strict ? kStrict : 0u;
    s.SA = 0.0f;
    s.b_jl = rcp_approx(c.t_min);
    s.b_jh = rcp_approx(c.hi0);
    const float is = rcp_approx(S1);
    s.bc = 1.0f;
    s.Hc = entropy_nats(lg2_approx(S1), is, V1, 1.0f);
    s.dHc = entropy_slope(is, V1, W1, 1.0f);
    return s;
}

// Appends grid index v to the round's points (constant register indices,
// no local memory).
__device__ __forceinline__ void put_point(int (&J)[kMaxPoints], int& np,
                                          int v) {
    if (np == 0) J[0] = v;
    else if (np == 1) J[1] = v;
    else J[2] = v;
    ++np;
}

// Chooses the grid points of the next round (indices J); returns how many
// (0: done; the result is then search_result()).
__device__ __forceinline__ int search_plan(Search& s, const SearchCfg& c,
                                           int (&J)[kMaxPoints]) {
    const Grid& g = c.g;
    if (s.f & kTminInf) {
        // Every grid point is infeasible: lo never moves (section 5.4).
        s.f |= kOverflow | kDone;
        return 0;
    }
    if (s.jh - s.jl <= 1) {
        if (s.f & kJlEval) {
            s.f |= kDone;
            return 0;
        }
        // lo stayed at t_min without an evaluation there: one more for its
        // S and the section 5.4 check.
        s.f |= kFinal;
        J[0] = 0;
        return 1;
    }
    if ((s.f & kStrict) || s.rounds >= kMaxNewtonRounds) {
        J[0] = s.jl + ((s.jh - s.jl) >> 1);
        return 1;
    }
    int np = 0;
    if (s.f & kFirst) {
        // The point the fan placed (search_fan), t_min with it when it
        // comes within 4 t_min and no feasible point is known.
        s.f &= ~kFirst;
        const float Tn = rcp_approx(s.bc);
        int jn = Tn > g.lo0 ? g.near(Tn) : 0;
        jn = min(max(jn, s.jl + 1), s.jh - 1);
        s.jl_prev = s.jl;
        s.jh_prev = s.jh;
        put_point(J, np, jn);
        if (!(s.f & kJlEval) && Tn <= 4.0f * g.lo0) put_point(J, np, 0);
        return np;
    }
    if (s.f & kEndgame) {
        const bool lo_moved = s.jl != s.jl_prev, hi_moved = s.jh != s.jh_prev;
        s.jl_prev = s.jl;
        s.jh_prev = s.jh;
        const int d = s.jh - s.jl;
        if (lo_moved != hi_moved) {
            // Only one end moved last round: the crossing is most likely
            // just past that end (fp32 evaluations of H next to the bound
            // can put a converged Newton point a few points off, and on the
            // fine grid, where every fp32 value is a point, a converged
            // Newton point is still many points off).  Gallop from it
            // towards the other end, 1, 2 and 4 strides out (the stride
            // starting at 1 on the exact grid, 2 on the fine one) and
            // growing eightfold per round; when the bracket is shorter than
            // a stride, quarter it instead.  Quartering the whole bracket
            // instead cost rows whose crossing sat next to the moved end
            // up to eight extra rounds.
            s.stride = max(s.stride, g.fine ? 2 : 1);
#pragma unroll
            for (int k = 0; k < kMaxPoints; ++k) {
                const int off = s.stride << k;
                if (off < d) put_point(J, np, lo_moved ? s.jl + off : s.jh - off);
            }
            if (s.stride < (1 << 26)) s.stride <<= 3;
            if (np > 0) return np;
        }
        // The bracket's midpoint and quarter points: two halvings per round.
        const int m = s.jl + (d >> 1);
        put_point(J, np, m);
        const int a = s.jl + (d >> 2);
        const int b = m + ((s.jh - m) >> 1);
        if (a > s.jl && a < m) put_point(J, np, a);
        if (b > m && b < s.jh) put_point(J, np, b);
        return np;
    }
    // Safeguarded Newton for log H = log bound in beta (plain Newton on H
    // when the bound is not positive), kept inside the bracket in beta.
    const float b_inf = s.b_jh;
    const float b_feas = s.b_jl;
    float bn;
    if (c.bound > 0.0f && s.Hc > 0.0f) {
        // log2 H - log2 bound over its slope, in one reciprocal:
        // bn = bc - (lg2 H - lg2 bound) H / (dH log2 e).
        const float gl = lg2_approx(s.Hc) - c.lg2_bound;  // log2 units
        bn = s.dHc < 0.0f ? s.bc - gl * s.Hc * rcp_approx(s.dHc * kLog2e) : NAN;
    } else {
        bn = s.dHc < 0.0f ? s.bc - (s.Hc - c.bound) * rcp_approx(s.dHc) : NAN;
    }
    // A step that leaves the bracket is replaced by the bracket's geometric
    // midpoint, unless it points back past the bracket end the anchor is
    // (H there equal to the bound in fp32, or on the wrong side of it by a
    // rounding): that step is kept, and the clamp below takes that end's
    // inner neighbour.
    if (!(bn > b_inf && bn < b_feas)) {
        const bool back = s.rounds > 0 &&
                          (bn >= b_feas ? s.bc >= b_feas : (bn <= b_inf && s.bc <= b_inf));
        if (!back) bn = sqrtf(b_inf * b_feas);
    }
    const float Tn = rcp_approx(bn);
    // The grid point at or just below Tn, strictly inside the bracket.
    int jn = Tn > g.lo0 ? g.near(Tn) : 0;
    jn = min(max(jn, s.jl + 1), s.jh - 1);
    s.jl_prev = s.jl;
    s.jh_prev = s.jh;
    const bool probe = !(s.f & kJlEval) && Tn <= 4.0f * g.lo0;  // t_min probe
    put_point(J, np, jn);
    if (probe) put_point(J, np, 0);
    if (!probe && fabsf(bn - s.bc) <= 1e-3f * s.bc) {
        // Newton has converged: also evaluate the neighbours, which close
        // the bracket when the crossing lies next to jn.
        if (jn + 1 < s.jh) put_point(J, np, jn + 1);
        if (jn - 1 > s.jl) put_point(J, np, jn - 1);
        s.f |= kEndgame;
    }
    return np;
}

// Whether the round just planned is followed by a Newton step, which needs
// the slope (hence W) at the round's first point.
__device__ __forceinline__ bool newton_next(const Search& s) {
    return !(s.f & (kFinal | kStrict | kEndgame)) &&
           s.rounds + 1 < kMaxNewtonRounds;
}

// Moves the bracket's ends with the decisions inf[i] at grid points J[i]
// (inverse temperatures beta[i], sums S[i]), i < np: feasible points raise
// jl, then infeasible ones lower jh; a point the bracket no longer contains
// is already decided and skipped.
__device__ __forceinline__ void bracket_update(Search& s, int np,
                                               const int (&J)[kMaxPoints],
                                               const float (&beta)[kMaxPoints],
                                               const float (&S)[kMaxPoints],
                                               const bool (&inf)[kMaxPoints]) {
#pragma unroll
    for (int i = 0; i < kMaxPoints; ++i) {
        if (i >= np || inf[i]) continue;
        const bool inside = J[i] > s.jl || (J[i] == 0 && !(s.f & kJlEval));
        if (inside && J[i] < s.jh) {
            s.jl = J[i];
            s.f |= kJlEval;
            s.SA = S[i];
            s.b_jl = beta[i];
        }
    }
#pragma unroll
    for (int i = 0; i < kMaxPoints; ++i) {
        if (i >= np || !inf[i]) continue;
        if (J[i] == 0 && !(s.f & kJlEval)) {
            s.f |= kTminInf;
            s.SA = S[i];
        } else if (J[i] > s.jl && J[i] < s.jh) {
            s.jh = J[i];
            s.b_jh = beta[i];
        }
    }
}

// Temperatures evaluated alongside T = 1 by the few-row launches of the
// cluster kernel (the "fan"): they place the search's first point.
constexpr int kFanPoints = cs::kFanPoints;

// Takes in the fan evaluated with the T = 1 pass: (S[k], V[k]) at inverse
// temperatures beta[k] (increasing; not grid points, and their decisions
// do not move the bracket), with H(1) > bound from (S1, V1).  The next
// round evaluates the point where log H, interpolated linearly in log beta
// between the two of {1, beta[0..]} that straddle the bound, meets it (the
// line through the last two when the whole fan lies above the bound), and
// the Newton steps start from there (its round accumulates W).
__device__ __forceinline__ void search_fan(Search& s, const SearchCfg& c,
                                           const float (&beta)[kFanPoints],
                                           const float (&S)[kFanPoints],
                                           const float (&V)[kFanPoints],
                                           float S1, float V1) {
    // (log2 beta, log2 H in bits) of T = 1 and the fan.
    float x[kFanPoints + 1], y[kFanPoints + 1];
    x[0] = 0.0f;
    y[0] = lg2_approx(lg2_approx(S1) - V1 * rcp_approx(S1));
#pragma unroll
    for (int i = 0; i < kFanPoints; ++i) {
        x[i + 1] = lg2_approx(beta[i]);
        y[i + 1] = lg2_approx(lg2_approx(S[i]) - beta[i] * V[i] * rcp_approx(S[i]));
    }
    const float ly = c.lg2_bound - lg2_approx(kLn2);  // log2 of the bound in bits
    // The first point at or below the bound, and the one before it.
    int i1 = kFanPoints;
#pragma unroll
    for (int i = kFanPoints; i >= 1; --i)
        if (y[i] <= ly) i1 = i;
    float xa = x[0], ya = y[0], xb = x[1], yb = y[1];
#pragma unroll
    for (int i = 1; i <= kFanPoints; ++i) {
        if (i == i1) {
            xa = x[i - 1];
            ya = y[i - 1];
            xb = x[i];
            yb = y[i];
        }
    }
    // A point beyond an end of the bracket (an extended line overshoots
    // where H falls steeply) is moved to that end: the clamp to the
    // bracket's inner points follows in search_plan.
    float b0 = ex2(xa + (ly - ya) * (xb - xa) * rcp_approx(yb - ya));
    b0 = b0 == b0 ? fminf(fmaxf(b0, s.b_jh), s.b_jl) : sqrtf(s.b_jh * s.b_jl);
    s.bc = b0;
    s.f |= kFirst;
}

// Records the round's evaluations: grid point J[i] (at inverse temperature
// beta[i]) gave the row sums S[i], V[i], and, when has_w, W[0].  Feasible
// points raise jl, then infeasible ones lower jh; a point the bracket no
// longer contains is already decided and skipped, so fp32 evaluations that
// disagree with monotonicity at the crossing cannot invert the bracket.
__device__ __forceinline__ void search_update(Search& s, const SearchCfg& c,
                                              int np,
                                              const int (&J)[kMaxPoints],
                                              const float (&beta)[kMaxPoints],
                                              const float (&S)[kMaxPoints],
                                              const float (&V)[kMaxPoints],
                                              const float (&W)[kMaxPoints],
                                              bool has_w) {
    bool inf[kMaxPoints];
#pragma unroll
    for (int i = 0; i < kMaxPoints; ++i)
        inf[i] = i < np && entropy_above(make_float2(S[i], V[i]), beta[i],
                                         c.bound_bits);
    if (s.f & kFinal) {
        s.SA = S[0];
        s.f |= kDone | (inf[0] ? kOverflow : 0u);
        return;
    }
    bracket_update(s, np, J, beta, S, inf);
    // The Newton anchor moves to the round's first point (only used when
    // a Newton step follows, which is when W was accumulated).
    if (has_w) {
        const float is = rcp_approx(S[0]);
        s.bc = beta[0];
        s.Hc = entropy_nats(lg2_approx(S[0]), is, V[0], beta[0]);
        s.dHc = entropy_slope(is, V[0], W[0], beta[0]);
    }
    ++s.rounds;
}

// The search's result once search_plan returned 0: the temperature, S there
// and the section 5.4 flag.
__device__ __forceinline__ float search_result_T(const Search& s,
                                                 const SearchCfg& c) {
    return (s.f & (kTminInf | kFinal)) ? c.g.lo0 : c.g.at(s.jl);
}

// Newton rounds a searching narrow row may take before the fallback.
constexpr int kNarrowNewtonRounds = 7;
// The narrow search probes t_min instead of the Newton point when no
// feasible point is known and the Newton point lies within this factor of
// t_min: generously after the first step (from T = 1, whose Newton point
// can be off by a factor of three either way), tightly later (a probe
// costs a round whenever the root lies above t_min).
constexpr float kNarrowProbeFirst = 4.0f;
constexpr float kNarrowProbeLater = 1.5f;
// A Newton point within this fraction of the bracket's far end (in beta,
// measured from the end it steps from) is replaced by the bracket's
// geometric midpoint: log H is far from linear over such a step, and a row
// can otherwise oscillate between the two ends.
constexpr float kNarrowFarEnd = 0.1f;

// The search for narrow rows, one grid point per round (the row-group
// kernel, whose rows are a few registers per lane; a multi-point pass there
// costs more than the rounds it saves).  Called
// after H(1) > bound with S1, V1, W1 at beta = 1; eval3(beta) returns the
// row's (S, V, W) at beta and eval2(beta) its (S, V).  Strict: the
// bisection, one evaluation per halving.  Otherwise up to
// kNarrowNewtonRounds Newton steps on log H(beta) from the last point
// evaluated, kept inside the bracket in beta (its geometric midpoint when
// the step leaves it across the far end or lands next to that end; the
// inner neighbour of the near end when it points back past that end) and
// placed on the grid point at or below (t_min when the step comes near t_min and no feasible
// point is known; when t_min then proves feasible, the next step is taken
// from whichever of t_min and the point before it has H nearer the bound
// in log terms), then, only while the bracket is open, points stepping
// from the end moved last with doubling strides.  One lg2 and one
// reciprocal of S serve both the decision and the next step.  Returns T,
// 1/T, 1/S(T), the section 5.4 flag and the number of evaluations made.
template <int K, class Eval3, class Eval2>
__device__ __forceinline__ void narrow_search(const SearchCfg& cfg, float S1,
                                              float V1, float W1, bool strict,
                                              Eval3 eval3, Eval2 eval2,
                                              float& T_out, float& beta_out,
                                              float& inv_s, bool& overflow,
                                              int& evals) {
    const Grid& g = cfg.g;
    evals = 0;
    int jl = 0, jh = g.top;
    bool jl_eval = false;   // G(jl) evaluated feasible
    bool tmin_inf = false;  // t_min evaluated infeasible
    float s_lo = 0.0f;
    if (cfg.t_min < cfg.hi0 && strict) {
        while (jh - jl > 1) {
            const int jm = jl + ((jh - jl) >> 1);
            const float b = rcp_approx(g.template at_t<K>(jm));
            const float2 sv = eval2(b);
            ++evals;
            if (entropy_above(sv, b, cfg.bound_bits)) {
                jh = jm;
            } else {
                jl = jm;
                jl_eval = true;
                s_lo = sv.x;
            }
        }
    } else if (cfg.t_min < cfg.hi0) {
        float b = 1.0f, S = S1, V = V1, W = W1;
        float ls = lg2_approx(S);  // log2 S, shared by the decision and the step
        // The point evaluated before a t_min probe (its beta and sums).
        float pb = 1.0f, pS = S1, pV = V1, pW = W1;
        // The side of the point the next step starts from, and whether the
        // far-end guard applies to that step (not right after stepping
        // back to the point before a probe).
        bool anchor_feas = false;
        bool far_guard = false;
        float b_inf = rcp_approx(cfg.hi0);
        float b_feas = rcp_approx(cfg.t_min);
        const bool log_newton = cfg.bound > 0.0f;
        int jlast = -1;
        // The round's bookkeeping is written as selects rather than
        // branches: the lane groups of a warp take different sides at
        // every round, and each branch would be run for both.
        for (int k = 0; k < kNarrowNewtonRounds && jh - jl > 1 && !tmin_inf; ++k) {
            const bool at_end = k > 0;  // the step starts from a bracket end
            const float is = rcp_approx(S);
            const float ey = V * is;
            const float H = kLn2 * (ls - b * ey);
            const float dH = -b * (kLn2 * kLn2) * fmaxf(fmaf(W, is, -ey * ey), 0.0f);
            // Newton on log H (log2 H - log2 bound over its slope) when the
            // bound is positive, else on H itself.
            const bool on_log = log_newton && H > 0.0f;
            const float num = on_log ? (lg2_approx(H) - cfg.lg2_bound) * H : H - cfg.bound;
            const float den = on_log ? dH * kLog2e : dH;
            float bn = b - num * rcp_approx(den);
            // A step that points back past the end it starts from (H there
            // equal to the bound in fp32, or on the wrong side of it by a
            // rounding) is kept: the clamp below then takes that end's
            // inner neighbour, which closes the bracket when the crossing
            // is next to it.  A step that leaves the bracket otherwise, or
            // lands next to its far end, takes the geometric midpoint.
            const bool outside = !(bn > b_inf && bn < b_feas);
            const bool back = at_end && (anchor_feas ? bn >= b_feas : bn <= b_inf);
            const float far = anchor_feas ? b_inf : b_feas;
            const bool by_far = far_guard && fabsf(far - bn) < kNarrowFarEnd * fabsf(far - b);
            if (outside ? !back : by_far) bn = sqrtf(b_inf * b_feas);
            const float Tn = rcp_approx(bn);
            const float pf = k == 0 ? kNarrowProbeFirst : kNarrowProbeLater;
            const bool probe = !jl_eval && Tn <= pf * cfg.t_min;
            int jn = Tn > cfg.t_min ? g.template near_t<K>(Tn) : 0;
            jn = probe ? 0 : min(max(jn, jl + 1), jh - 1);
            pb = probe ? b : pb;
            pS = probe ? S : pS;
            pV = probe ? V : pV;
            pW = probe ? W : pW;
            b = rcp_approx(probe ? cfg.t_min : g.template at_t<K>(jn));
            const float3 r = eval3(b);
            ++evals;
            S = r.x;
            V = r.y;
            W = r.z;
            // entropy_above's test, with log2 S kept for the next step.
            ls = lg2_approx(S);
            const bool inf = fmaf(S, ls - cfg.bound_bits, -b * V) > 0.0f;
            const bool feas = !inf;
            jlast = jn;
            s_lo = (probe || feas) ? S : s_lo;
            tmin_inf = tmin_inf || (probe && inf);
            jl_eval = jl_eval || feas;
            b_feas = feas ? b : b_feas;
            const bool move_hi = !probe && inf;
            const bool move_lo = !probe && feas;
            jh = move_hi ? jn : jh;
            b_inf = move_hi ? b : b_inf;
            jl = move_lo ? jn : jl;
            anchor_feas = feas;
            far_guard = true;
            if (probe && feas) {
                // t_min is feasible: the next step starts from whichever of
                // t_min and the point before the probe has H nearer the
                // bound (in log terms).
                const float h_t = kLn2 * (ls - b * V * rcp_approx(S));
                const float h_p = kLn2 * (lg2_approx(pS) - pb * pV * rcp_approx(pS));
                const float lb = log_newton ? cfg.lg2_bound : 0.0f;
                if (!(h_t > 0.0f) ||
                    fabsf(lg2_approx(h_p) - lb) < fabsf(lg2_approx(h_t) - lb)) {
                    // The point before the probe: infeasible, since no
                    // feasible point was known when the probe was chosen.
                    b = pb;
                    S = pS;
                    V = pV;
                    W = pW;
                    ls = lg2_approx(pS);
                    anchor_feas = false;
                    far_guard = false;
                }
            }
        }
        int stride = 1;
        while (jh - jl > 1 && !tmin_inf) {
            const int d = jh - jl;
            const int step = max(min(stride, d >> 1), 1);
            const int jm = jl == jlast ? jl + step : jh == jlast ? jh - step : jl + (d >> 1);
            stride *= 2;
            jlast = jm;
            const float bm = rcp_approx(g.template at_t<K>(jm));
            const float2 sv = eval2(bm);
            ++evals;
            if (entropy_above(sv, bm, cfg.bound_bits)) {
                jh = jm;
            } else {
                jl = jm;
                jl_eval = true;
                s_lo = sv.x;
            }
        }
    }
    const float lo = jl_eval ? g.template at_t<K>(jl) : cfg.t_min;
    const float b_lo = rcp_approx(lo);
    overflow = tmin_inf;
    if (!tmin_inf && !jl_eval) {
        // lo is still t_min: evaluate it (section 5.4 check).
        const float2 sv = eval2(b_lo);
        ++evals;
        s_lo = sv.x;
        overflow = entropy_above(sv, b_lo, cfg.bound_bits);
    }
    T_out = lo;
    beta_out = b_lo;
    inv_s = 1.0f / s_lo;
}

}  // namespace csd
