// Search control for the global lambda: the fixed 40-step bisection, walked
// with as few rounds of evaluations as possible.
//
// The problem ("Rate-adaptive KV-cache quantizer", "Mathematical statement")
// is separable given lambda, and the total rate R(lambda) = sum_r d_r H_r of
// the per-block minimisers is non-increasing in lambda.  The lambda that the
// bisection returns is fixed by the predicate P(lambda) = [R(lambda) <= B] at
// the midpoints it visits:
//   R(0) <= B  -> lambda = 0;
//   hi = hi0 * 2^t, t the first of 0..30 with P true (none: infeasible);
//   40 times: mid = 0.5 (lo + hi); P(mid) ? hi = mid : lo = mid;
//   lambda = hi.
// Each round evaluates R at up to 32 lambdas at once (one per lane of the
// DP).  Every evaluated lambda tightens a window (xa, xb): xa the largest
// lambda known infeasible, xb the smallest known feasible.  Because R is
// monotone, a midpoint at or above xb is feasible and one at or below xa is
// not, so the walk only stops at midpoints strictly inside the window; the
// next round evaluates those, breadth first over the walk's possible paths.
// Round 0 probes lambda = 0, the first doublings of hi0 and a geometric grid
// below hi0, which brackets the answer within a factor 2^1.5 at once.
//
// Rates are sums of per-block d_r H_r in fixed point (integers in units of
// 2^-20 bit) and the budget is compared as floor(B 2^20), so R <= B is an
// integer comparison with the same outcome as the real one.  The walk's
// midpoints 0.5 (lo + hi) are one binary64 add of exactly halved operands
// (half_sum), and lambdas are compared through order-preserving integer keys:
// the control runs on a GPU whose double-precision unit has a long latency,
// and every one of these steps is on the search's critical path.
//
// Plain C++ usable on the host (tests) and the device (last CTA of a round).
#pragma once
#include <math.h>
#include <stdint.h>
#include <string.h>

#ifndef KVQ_HD
#ifdef __CUDACC__
#define KVQ_HD __host__ __device__
#else
#define KVQ_HD
#endif
#endif

// Out of line: a rarely taken branch whose arithmetic (binary64, on a GPU
// with a slow double-precision unit) must not be evaluated speculatively on
// the common path.
#ifndef KVQ_COLD
#ifdef __CUDA_ARCH__
#define KVQ_COLD __noinline__
#else
#define KVQ_COLD __attribute__((noinline))
#endif
#endif

namespace kvq {

constexpr int kSearchProbes = 32;
constexpr int kSearchSteps = 40;
constexpr int kSearchMaxDoublings = 30;
constexpr int kSearchFirstDoublings = 3;       // hi0 * 2^0 .. 2^2 in round 0

enum SearchPhase : int32_t {
    kSearchPilot = 4,     // a sample of the blocks at the round-0 probes (estimate only)
    kSearchBracket = 0,   // round 0: 0, hi0 * 2^{0,1,2}, geometric grid
    kSearchDouble = 1,    // hi0 * 2^3 .. 2^30 (only if round 0 found no feasible hi)
    kSearchWalk = 2,      // bisection walk
    kSearchDone = 3,
};

struct alignas(16) SearchState {
    double hi0;           // max_r (c_max - c_min)^2
    double lo, hi;        // bisection interval
    double xa, xb;        // known infeasible (largest) / feasible (smallest)
    double lambda;        // the answer once done
    long long R_xb;       // R at xb (fixed point)
    double probe[kSearchProbes];   // lambdas of the next round (walk phase)
    int32_t phase;
    int32_t step;         // bisection steps taken
    int32_t nprobe;       // probes in use this round
    int32_t xa_probe;     // probe of the last round that became xa, or -1
    int32_t xb_probe;     // probe of the last round that became xb, or -1
    int32_t infeasible;
    int32_t rounds;
    int32_t pilot_stride;     // pilot round: every pilot_stride-th block (0: no pilot)
    int32_t pilot_blocks;     // blocks the pilot evaluated
    int32_t have_grid;        // round 0 uses probe[4..31] (set by the pilot)
    int32_t f32_lambda;       // R depends on lambda only through its binary32 rounding
};

// ------------------------------------------------------- binary64 helpers
KVQ_HD inline uint64_t dbits(double x) {
    uint64_t u;
    memcpy(&u, &x, 8);
    return u;
}
KVQ_HD inline double dfrom(uint64_t u) {
    double x;
    memcpy(&x, &u, 8);
    return x;
}

// Order-preserving key: okey(a) < okey(b) iff a < b (finite or infinite, not
// NaN; -0 sorts just below +0, which no caller distinguishes).
KVQ_HD inline uint64_t okey(double x) {
    const uint64_t u = dbits(x);
    return (u >> 63) ? ~u : (u | 0x8000000000000000ull);
}

// 0.5 * (a + b), bit for bit as binary64 arithmetic computes it, for finite
// a, b >= 0.  Same exponent field (the late steps of every bisection): the
// raw bits are a fixed-point significand, so the midpoint is their integer
// mean rounded half to even.  Otherwise halving is exact for normal numbers
// and commutes with rounding, so RN(a + b) / 2 = RN(a/2 + b/2); each half is
// an exponent decrement (integer) and one binary64 add remains instead of an
// add and a multiply.  Zero or near-subnormal operands in different binades
// take the expression itself.
KVQ_HD inline uint64_t mean_bits_same_exponent(uint64_t ua, uint64_t ub) {
    const uint64_t t = ua + ub, h = t >> 1;   // no overflow: both below 2^63
    return h + (t & h & 1u);                  // a tie goes to the even neighbour
}
KVQ_HD inline double half_sum(double a, double b) {
    const uint64_t ua = dbits(a), ub = dbits(b);
    if ((ua >> 52) == (ub >> 52) && (ua >> 52) < 2047) return dfrom(mean_bits_same_exponent(ua, ub));
    const uint32_t ea = (uint32_t)(ua >> 52), eb = (uint32_t)(ub >> 52);   // sign bit 0
    const bool na = ea >= 3 && ea <= 2046, nbb = eb >= 3 && eb <= 2046;
    if ((na || ua == 0) && (nbb || ub == 0) && (na || nbb)) {
        const double ah = ua == 0 ? 0.0 : dfrom(ua - (1ull << 52));
        const double bh = ub == 0 ? 0.0 : dfrom(ub - (1ull << 52));
        return ah + bh;
    }
    return 0.5 * (a + b);
}

// Raw bits of the smallest binary64 value that rounds (to nearest, ties to
// even) to the binary32 value f, for f > 0 (+inf included), and of the
// largest one, for finite f >= 0: the midpoints between f and its neighbours,
// exact in binary64, or the next double inward when the tie goes to the
// neighbour.  For a normal f the binary64 bits of f are its binary32 bits
// shifted left by 29 with the exponent rebiased, a binary32 half-ulp is 2^28
// binary64 ulps of the same binade (of the binade below, for the midpoint
// under a power of two), and +inf continues the pattern (2^128 - 2^103 is the
// smallest value that overflows); subnormal neighbours take the arithmetic
// itself.
KVQ_HD inline uint64_t f32_as_f64_bits(uint32_t fb) {
    return ((uint64_t)fb << 29) + (896ull << 52);   // exponent bias 1023 - 127
}
KVQ_HD inline KVQ_COLD uint64_t f32_low_bits_sub(float f) {
    uint32_t fb;
    memcpy(&fb, &f, 4);
    const uint32_t pb = fb - 1u;
    float p;
    memcpy(&p, &pb, 4);
    const double m = ((double)p + (double)f) * 0.5;
    return (fb & 1u) ? dbits(m) + 1u : dbits(m);
}
KVQ_HD inline KVQ_COLD uint64_t f32_high_bits_sub(float f) {
    uint32_t fb;
    memcpy(&fb, &f, 4);
    const uint32_t nb = fb + 1u;
    float n;
    memcpy(&n, &nb, 4);
    const double m = ((double)f + (double)n) * 0.5;
    return (fb & 1u) ? dbits(m) - 1u : dbits(m);
}
KVQ_HD inline uint64_t f32_low_bits(float f) {
    uint32_t fb;
    memcpy(&fb, &f, 4);
    if (fb > 0x00800000u) return f32_as_f64_bits(fb) - (1ull << 28) + (fb & 1u);
    return f32_low_bits_sub(f);
}
KVQ_HD inline uint64_t f32_high_bits(float f) {
    uint32_t fb;
    memcpy(&fb, &f, 4);
    if (fb >= 0x00800000u) return f32_as_f64_bits(fb) + (1ull << 28) - (fb & 1u);
    return f32_high_bits_sub(f);
}

// x * 2^t for x = 0 or normal x > 0 whose result stays normal (exponent
// arithmetic); anything else goes through ldexp.
KVQ_HD inline double pow2_scale(double x, int t) {
    const uint64_t u = dbits(x);
    const int e = (int)(u >> 52);
    if (u == 0) return 0.0;
    if ((u >> 63) || e == 0 || e + t < 1 || e + t > 2046) return ldexp(x, t);
    return dfrom(u + ((uint64_t)(int64_t)t << 52));
}

// floor(B 2^20) clamped to the int64 range: R <= B iff R_fx <= this, for
// every fixed-point rate R_fx (B >= 0).
KVQ_HD inline long long budget_fx(double B) {
    const double v = floor(B * 1048576.0);
    if (!(v < 9.2e18)) return 0x7fffffffffffffffll;
    return (long long)v;
}

KVQ_HD inline void search_init(SearchState &s) {
    s.hi0 = 0.0;
    s.lo = s.hi = 0.0;
    s.xa = -1.0;
    s.xb = INFINITY;
    s.R_xb = 0;
    s.lambda = 0.0;
    for (int i = 0; i < kSearchProbes; ++i) s.probe[i] = 0.0;
    s.phase = kSearchBracket;
    s.step = 0;
    s.nprobe = kSearchProbes;
    s.xa_probe = s.xb_probe = -1;
    s.infeasible = 0;
    s.rounds = 0;
    s.pilot_stride = 0;
    s.pilot_blocks = 0;
    s.have_grid = 0;
    s.f32_lambda = 0;
}

// Start with a pilot round over every stride-th of nb blocks (stride <= 0: none).
KVQ_HD inline void search_set_pilot(SearchState &s, int64_t nb, int stride) {
    if (stride > 1 && nb >= 4 * (int64_t)stride) {
        s.pilot_stride = stride;
        s.pilot_blocks = (int32_t)((nb + stride - 1) / stride);
        s.phase = kSearchPilot;
    }
}

// hi0 * 2^(-1.5 k): a power-of-two scaling, times sqrt(1/2) (one correctly
// rounded constant) when k is odd
KVQ_HD inline double search_grid(double hi0, int k) {
    const double odd = 0.70710678118654752440;
    return (k & 1) ? pow2_scale(hi0 * odd, -(3 * k - 1) / 2) : pow2_scale(hi0, -(3 * k) / 2);
}

// Fine grid of round 0 around an estimate, k = 0..27: 14 probes on each side
// of est, the j-th out (j = 0..13) at est * 2^(+-c (g^(j+1) - 1) / (g - 1)),
// c = 0.0215, g = 1.25: cells of 1.5 % next to the estimate, growing by a
// quarter per probe out to a factor 3.7 either way, so that the grid spans
// the pilot's whole bracket (a factor 2^1.5) wherever the estimate falls in
// it, and the window after round 0 is narrow when the estimate is good.  In
// single precision (the grid only places probes).
KVQ_HD inline double search_fine(double est, int k) {
    const int j = k < 14 ? 13 - k : k - 14;
    const float off = 0.0215f * (exp2f((float)(j + 1) * 0.32192809f) - 1.0f) * 4.0f;   // log2(1.25)
    return est * (double)exp2f(k < 14 ? -off : off);
}

// lambda evaluated by probe p this round
KVQ_HD inline double search_probe(const SearchState &s, int p) {
    if (s.phase == kSearchBracket || s.phase == kSearchPilot) {
        if (p == 0) return 0.0;
        if (p <= kSearchFirstDoublings) return pow2_scale(s.hi0, p - 1);
        if (s.phase == kSearchBracket && s.have_grid) return s.probe[p];
        return search_grid(s.hi0, p - kSearchFirstDoublings);
    }
    if (s.phase == kSearchDouble) {
        const int t = kSearchFirstDoublings + p;
        return pow2_scale(s.hi0, t <= kSearchMaxDoublings ? t : kSearchMaxDoublings);
    }
    return s.probe[p < s.nprobe ? p : 0];
}

// What the window (xa, xb) fixes about the predicate at a midpoint: order
// keys of both ends, and, when R depends on lambda only through its binary32
// rounding (the GPU evaluates the DP at float(lambda)), the binary32 values
// of both ends: a midpoint that rounds to float(xb) is feasible, one that
// rounds to float(xa) is not.  For positive midpoints the same tests are
// integer comparisons of raw bits: mid >= xb (rxb), mid <= xa (rxa), and,
// inside the window, float(mid) == float(xb) iff mid >= the smallest double
// rounding to float(xb) (lb), float(mid) == float(xa) iff mid <= the largest
// double rounding to float(xa) (ha).
struct SearchWindow {
    uint64_t kxa, kxb;
    float fxa, fxb;
    int f32;
    uint64_t rxa, rxb, lb, ha;
};
KVQ_HD inline SearchWindow search_window_of(const SearchState &s) {
    SearchWindow w;
    w.kxa = okey(s.xa);
    w.kxb = okey(s.xb);
    w.fxa = (float)s.xa;
    w.fxb = (float)s.xb;
    w.f32 = s.f32_lambda;
    w.rxb = w.kxb ^ (1ull << 63);                               // xb >= 0 (or +inf)
    w.rxa = (w.kxa >> 63) ? (w.kxa ^ (1ull << 63)) : 0ull;      // xa < 0: none
    w.lb = ~0ull;                                               // never reached
    w.ha = 0ull;
    if (w.f32) {
        if (s.xb >= 0.0) w.lb = w.fxb > 0.f ? f32_low_bits(w.fxb) : 0ull;
        if (s.xa >= 0.0)                                        // -0 compares equal to +0
            w.ha = w.fxa < INFINITY ? f32_high_bits(w.fxa == 0.f ? 0.f : w.fxa) : dbits(INFINITY);
    }
    return w;
}
// P(mid) if it follows from the window, else -1
KVQ_HD inline int search_known_w(const SearchWindow &w, double mid) {
    const uint64_t km = okey(mid);
    if (km >= w.kxb) return 1;
    if (km <= w.kxa) return 0;
    if (w.f32) {
        const float fm = (float)mid;
        if (fm == w.fxb) return 1;
        if (fm == w.fxa) return 0;
    }
    return -1;
}
KVQ_HD inline int search_known(const SearchState &s, double mid) {
    return search_known_w(search_window_of(s), mid);
}

// Take bisection steps from depth `step` on [lo, hi] while the midpoint is
// known from the window; returns the depth of the first unknown midpoint
// (kSearchSteps if none), with lo, hi the interval there.  Fast path (every
// practical case): lo = 0 with hi far from the subnormal range, or lo normal
// -- then every midpoint is a positive normal number, computed on raw bits
// (lo = 0: an exponent decrement; same exponent: the rounded integer mean;
// else one binary64 add of the halves), and the window tests are the raw-bit
// comparisons above.  Elsewhere the same steps with half_sum and order keys.
KVQ_HD inline bool walk_fast(uint64_t ul, uint64_t uh) {
    const uint32_t el = (uint32_t)(ul >> 52), eh = (uint32_t)(uh >> 52);
    return eh <= 2046 && (ul >> 63) == 0 && ((ul == 0 && eh >= 48) || el >= 3);
}
// The midpoint's raw bits on the fast path.
KVQ_HD inline KVQ_COLD uint64_t mid_bits_halves(uint64_t ul, uint64_t uh) {
    return dbits(dfrom(ul - (1ull << 52)) + dfrom(uh - (1ull << 52)));
}
KVQ_HD inline uint64_t mid_bits_fast(uint64_t ul, uint64_t uh) {
    if (ul == 0) return uh - (1ull << 52);
    if ((ul ^ uh) >> 52 == 0) return mean_bits_same_exponent(ul, uh);
    return mid_bits_halves(ul, uh);
}
KVQ_HD inline bool window_known(uint64_t um, const SearchWindow &w, bool &k) {
    const bool f1 = um >= w.rxb, f0 = um <= w.rxa, g1 = um >= w.lb, g0 = um <= w.ha;
    k = f1 || (!f0 && g1);
    return f1 || f0 || g1 || g0;
}
KVQ_HD inline int walk_known(double &lo, double &hi, int step, const SearchWindow &w) {
    uint64_t ul = dbits(lo), uh = dbits(hi);
    if (walk_fast(ul, uh)) {
        // three phases, each a loop without inner branches: lo = 0 (the
        // midpoint halves hi), lo and hi in different binades (one add of
        // the halves), the same binade (integer mean; it stays so)
        bool k = false;
        for (; step < kSearchSteps && ul == 0; ++step) {
            const uint64_t um = uh - (1ull << 52);
            if (!window_known(um, w, k)) goto done;
            ul = k ? ul : um;
            uh = k ? um : uh;
        }
        for (; step < kSearchSteps && ((ul ^ uh) >> 52) != 0; ++step) {
            const uint64_t um = mid_bits_halves(ul, uh);
            if (!window_known(um, w, k)) goto done;
            ul = k ? ul : um;
            uh = k ? um : uh;
        }
#pragma unroll 4
        for (; step < kSearchSteps; ++step) {
            const uint64_t um = mean_bits_same_exponent(ul, uh);
            if (!window_known(um, w, k)) goto done;
            ul = k ? ul : um;
            uh = k ? um : uh;
        }
    done:
        lo = dfrom(ul);
        hi = dfrom(uh);
        return step;
    }
    while (step < kSearchSteps) {
        const double mid = half_sum(lo, hi);
        const int k = search_known_w(w, mid);
        if (k < 0) break;
        if (k) hi = mid; else lo = mid;
        ++step;
    }
    return step;
}

// The update is split so that a warp can run it with one lane per probe:
//   search_window   fold the round's evaluations into (xa, xb)
//   search_advance  bracket decisions and the walk (cheap, sequential)
//   search_path     probe generation: lane L follows the decision bits of L
//                   through the unknown midpoints; the node reached after u
//                   unknown decisions with prefix bits p gets id 2^u - 1 + p,
//                   so the 32 paths together write the 31 unknown nodes of
//                   the next 5 unknown levels (breadth-first set)
// search_update runs the three in order on one thread (host tests); the
// device runs the same functions across a warp.

// (xb, its probe) = smallest feasible evaluation; (xa, its probe) = largest
// infeasible evaluation below xb.  Infeasible evaluations above xb contradict
// monotonicity (a rounding tie) and are ignored.
KVQ_HD inline void search_window(SearchState &s, double vb, int ib, long long Rb, double va,
                                 int ia) {
    s.xa_probe = s.xb_probe = -1;
    if (ib >= 0 && okey(vb) < okey(s.xb)) { s.xb = vb; s.xb_probe = ib; s.R_xb = Rb; }
    if (ia >= 0 && okey(va) > okey(s.xa) && okey(va) < okey(s.xb)) { s.xa = va; s.xa_probe = ia; }
}

// The round's bracket decisions (phase changes; lambda = 0; infeasible).
// Returns 1 if the bisection walk goes on.
KVQ_HD inline int search_decide(SearchState &s, const long long *R, long long Bfx) {
    s.rounds += 1;
    if (s.phase == kSearchBracket || s.phase == kSearchDouble) {
        if (s.phase == kSearchBracket && R[0] <= Bfx) {          // lambda = 0
            s.lo = s.hi = s.lambda = 0.0;
            s.xb = 0.0;
            s.xb_probe = 0;
            s.R_xb = R[0];
            s.phase = kSearchDone;
            return 0;
        }
        int t = -1;
        const int pmax = s.phase == kSearchBracket ? kSearchFirstDoublings
                                                   : kSearchMaxDoublings - kSearchFirstDoublings;
        for (int p = (s.phase == kSearchBracket ? 1 : 0); p <= pmax && p < s.nprobe; ++p) {
            const int tt = s.phase == kSearchBracket ? p - 1 : kSearchFirstDoublings + p;
            if (R[p] <= Bfx) { t = tt; break; }
        }
        if (t < 0) {
            if (s.phase == kSearchBracket) {
                s.phase = kSearchDouble;
                s.nprobe = kSearchMaxDoublings - kSearchFirstDoublings + 1;   // 2^3 .. 2^30
                return 0;
            }
            // infeasible at hi0 * 2^30: keep the choice there
            s.lo = 0.0;
            s.hi = s.lambda = pow2_scale(s.hi0, kSearchMaxDoublings);
            s.xb_probe = s.nprobe - 1;
            s.R_xb = R[s.nprobe - 1];
            s.infeasible = 1;
            s.phase = kSearchDone;
            return 0;
        }
        s.lo = 0.0;
        s.hi = pow2_scale(s.hi0, t);
        s.step = 0;
        s.phase = kSearchWalk;
    }
    return 1;
}

// The walk: the bisection steps the window decides.  Returns 1 if probes
// must be generated (phase stays Walk), 0 when the 40 steps are done.  The
// window is the one search_window_of gives for s (the walk does not change
// it).
KVQ_HD inline int search_walk_w(SearchState &s, const SearchWindow &win) {
    s.step = walk_known(s.lo, s.hi, s.step, win);
    if (s.step >= kSearchSteps) {
        s.lambda = s.hi;
        s.phase = kSearchDone;
        return 0;
    }
    s.nprobe = kSearchProbes - 1;
    return 1;
}
KVQ_HD inline int search_walk(SearchState &s) { return search_walk_w(s, search_window_of(s)); }

// Bracket decisions and the walk.  Returns 1 if probes must be generated.
KVQ_HD inline int search_advance(SearchState &s, const long long *R, long long Bfx) {
    return search_decide(s, R, Bfx) ? search_walk(s) : 0;
}

// The first unknown midpoint (all paths start there).
KVQ_HD inline double search_first_unknown(const SearchState &s) { return half_sum(s.lo, s.hi); }

// Path of lane L: writes the unknown midpoints it meets into probe[id].
// Generic form (half_sum and order keys), for any bracket.
KVQ_HD inline void search_path_generic(const SearchState &s, int L, double *probe) {
    const SearchWindow win = search_window_of(s);
    double a = s.lo, b = s.hi;
    int dep = s.step;
    for (int u = 0, pre = 0; u < 5; ++u) {
        dep = walk_known(a, b, dep, win);           // known steps up to the next unknown
        if (dep >= kSearchSteps) break;
        const double mid = half_sum(a, b);
        probe[(1 << u) - 1 + pre] = mid;
        const int k = ((L >> (4 - u)) & 1) ? 0 : 1;  // bit 1: take the infeasible branch
        pre = 2 * pre + (k ? 0 : 1);
        if (k) b = mid; else a = mid;
        ++dep;
    }
}

// Path of lane L (see search_path_generic), on the walk's fast path; `win`
// is search_window_of(s).
KVQ_HD inline void search_path_w(const SearchState &s, const SearchWindow &win, int L,
                                 double *probe) {
    uint64_t ul = dbits(s.lo), uh = dbits(s.hi);
    if (walk_fast(ul, uh)) {
        // the same steps on raw bits (see walk_known), the loop bodies
        // without branches so that the lanes of a warp stay converged: while
        // lo = 0 or lo and hi lie in different binades, then (the usual
        // case, and it stays so) in one binade
        int u = 0, pre = 0, dep = s.step;
        auto take = [&](uint64_t um) {
            bool k;
            const bool rec = !window_known(um, win, k);
            const int bit = (L >> (4 - u)) & 1;             // 1: take the infeasible branch
            const int id = (1 << u) - 1 + pre;
            if (rec) probe[id] = dfrom(um);
            k = rec ? bit == 0 : k;
            pre = rec ? 2 * pre + bit : pre;
            u += rec ? 1 : 0;
            ul = k ? ul : um;
            uh = k ? um : uh;
        };
        for (; dep < kSearchSteps && u < 5 && (ul == 0 || ((ul ^ uh) >> 52) != 0); ++dep)
            take(mid_bits_fast(ul, uh));
#pragma unroll 4
        for (; dep < kSearchSteps && u < 5; ++dep) take(mean_bits_same_exponent(ul, uh));
        return;
    }
    search_path_generic(s, L, probe);
}
KVQ_HD inline void search_path(const SearchState &s, int L, double *probe) {
    search_path_w(s, search_window_of(s), L, probe);
}

// Pilot round: estimate where R crosses B from the sample's rates (scaled to
// all blocks); round 0 then puts its fine grid there.  Nothing is concluded
// from the sample: the window only moves on evaluations of every block.
// The estimate from the pilot's smallest feasible probe (ib, vb, Rb) and
// largest infeasible probe below it (ia, va, Ra), rates scaled to all blocks
// (bits); ib / ia = -1 when there is none.  Single precision: the estimate
// only places probes.
KVQ_HD inline double search_pilot_finish(SearchState &s, int ib, double vb, double Rb, int ia,
                                         double va, double Ra, double B) {
    s.rounds += 1;
    s.xa_probe = s.xb_probe = -1;
    s.phase = kSearchBracket;
    s.have_grid = 0;
    if (ib <= 0 || !(vb > 0.0)) return 0.0;       // lambda = 0 likely, or no feasible probe
    double est;
    if (ia <= 0 || !(va > 0.0)) est = 0.5 * vb;
    else {
        const float fa = (float)Ra, fb = (float)Rb, fB = (float)B;
        float t = (fa - fB) / (fa - fb);              // log-linear interpolation
        t = t > 0.f ? (t < 1.f ? t : 1.f) : 0.f;
        est = va * (double)exp2f(t * log2f((float)(vb / va)));
    }
    s.have_grid = 1;
    return est;
}

KVQ_HD inline double search_pilot_estimate(SearchState &s, const long long *R, double B,
                                           int64_t nb) {
    const double scale =
        (double)nb / (double)(s.pilot_blocks > 0 ? s.pilot_blocks : 1) / 1048576.0;
    int ib = -1;
    double vb = INFINITY, Rb = 0.0;
    for (int p = 0; p < kSearchProbes; ++p) {
        const double v = search_probe(s, p), r = (double)R[p] * scale;
        if (r <= B && v < vb) { vb = v; ib = p; Rb = r; }
    }
    int ia = -1;
    double va = -1.0, Ra = 0.0;
    for (int p = 0; p < kSearchProbes; ++p) {
        const double v = search_probe(s, p), r = (double)R[p] * scale;
        if (!(r <= B) && v < vb && v > va) { va = v; ia = p; Ra = r; }
    }
    return search_pilot_finish(s, ib, vb, Rb, ia, va, Ra, B);
}

// Probe p of round 0 around the estimate (p > kSearchFirstDoublings).
KVQ_HD inline double search_pilot_probe(double est, int p) {
    return search_fine(est, p - 1 - kSearchFirstDoublings);
}

// Copy every field but the probe array.
KVQ_HD inline void search_copy_scalars(SearchState &d, const SearchState &s) {
    d.hi0 = s.hi0; d.lo = s.lo; d.hi = s.hi; d.xa = s.xa; d.xb = s.xb; d.R_xb = s.R_xb;
    d.lambda = s.lambda; d.phase = s.phase; d.step = s.step; d.nprobe = s.nprobe;
    d.xa_probe = s.xa_probe; d.xb_probe = s.xb_probe; d.infeasible = s.infeasible;
    d.rounds = s.rounds; d.pilot_stride = s.pilot_stride; d.pilot_blocks = s.pilot_blocks;
    d.have_grid = s.have_grid;
    d.f32_lambda = s.f32_lambda;
}

// Single-thread version (host tests).  R: fixed-point rates; B: the budget in
// bits; nb: number of blocks (pilot scaling).
KVQ_HD inline void search_update(SearchState &s, const long long *R, double B, int64_t nb = 0) {
    if (s.phase == kSearchPilot) {
        const double est = search_pilot_estimate(s, R, B, nb);
        if (s.have_grid)
            for (int p = 1 + kSearchFirstDoublings; p < kSearchProbes; ++p)
                s.probe[p] = search_pilot_probe(est, p);
        return;
    }
    const long long Bfx = budget_fx(B);
    int ib = -1, ia = -1;
    double vb = INFINITY, va = -INFINITY;
    long long Rb = 0;
    for (int p = 0; p < s.nprobe; ++p) {
        const double v = search_probe(s, p);
        if (R[p] <= Bfx && okey(v) < okey(vb)) { vb = v; ib = p; Rb = R[p]; }
    }
    const double xb_next = (ib >= 0 && okey(vb) < okey(s.xb)) ? vb : s.xb;
    for (int p = 0; p < s.nprobe; ++p) {
        const double v = search_probe(s, p);
        if (!(R[p] <= Bfx) && okey(v) > okey(va) && okey(v) < okey(xb_next)) { va = v; ia = p; }
    }
    search_window(s, vb, ib, Rb, va, ia);
    if (search_advance(s, R, Bfx)) {
        double probe[kSearchProbes];
        const double first = search_first_unknown(s);
        for (int p = 0; p < kSearchProbes; ++p) probe[p] = first;
        for (int L = 0; L < kSearchProbes; ++L) search_path(s, L, probe);
        for (int p = 0; p < kSearchProbes; ++p) s.probe[p] = probe[p];
    }
}

}  // namespace kvq
