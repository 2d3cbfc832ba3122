"""The lambda-search control (csrc/kvq_search.h, compiled for the host here)
walks exactly the fixed 40-step bisection: on monotone step functions R it
returns the same lambda as the sequential bisection, bit for bit, whatever the
breakpoints; and it needs far fewer rounds of evaluations than 40.  Its
integer helpers round and compare exactly as binary64 arithmetic does."""
import ctypes as C
import math
import os
import random
import struct
import subprocess
import tempfile

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "rate_adaptive_kv_block_b300", "csrc")

SHIM = r'''
#include "kvq_search.h"
#include <math.h>
static long long fx(double r) { return llround(r * 1048576.0); }
// mismatches of half_sum against the floating-point expression over n pairs
extern "C" long kvqs_half_sum_check(const double *a, const double *b, long n, long *first) {
    long bad = 0;
    *first = -1;
    for (long i = 0; i < n; ++i) {
        const double want = 0.5 * (a[i] + b[i]);
        const double got = kvq::half_sum(a[i], b[i]);
        if (kvq::dbits(want) != kvq::dbits(got)) { if (*first < 0) *first = i; ++bad; }
    }
    return bad;
}
extern "C" long kvqs_okey_check(const double *a, const double *b, long n) {
    long bad = 0;
    for (long i = 0; i < n; ++i) {
        if ((kvq::okey(a[i]) < kvq::okey(b[i])) != (a[i] < b[i])) ++bad;
        if ((kvq::okey(a[i]) == kvq::okey(b[i])) != (kvq::dbits(a[i]) == kvq::dbits(b[i]))) ++bad;
    }
    return bad;
}
extern "C" double kvqs_pow2_scale(double x, int t) { return kvq::pow2_scale(x, t); }
// the walk and the probe paths against the definition: 0.5 (lo + hi) and
// comparisons of doubles (and of their binary32 roundings); returns the
// number of mismatching states
static int ref_known(const kvq::SearchState &s, double m) {
    if (m >= s.xb) return 1;
    if (m <= s.xa) return 0;
    if (s.f32_lambda) {
        if ((float)m == (float)s.xb) return 1;
        if ((float)m == (float)s.xa) return 0;
    }
    return -1;
}
extern "C" long kvqs_path_check(const double *st, long n) {
    long bad = 0;
    for (long i = 0; i < n; ++i) {
        kvq::SearchState s;
        kvq::search_init(s);
        s.lo = st[5 * i]; s.hi = st[5 * i + 1]; s.xa = st[5 * i + 2]; s.xb = st[5 * i + 3];
        s.step = 0;
        s.f32_lambda = st[5 * i + 4] != 0.0;
        // the walk
        double lo = s.lo, hi = s.hi;
        int dep = 0;
        while (dep < kvq::kSearchSteps) {
            const double m = 0.5 * (lo + hi);
            const int k = ref_known(s, m);
            if (k < 0) break;
            if (k) hi = m; else lo = m;
            ++dep;
        }
        kvq::SearchState w = s;
        const int go = kvq::search_walk(w);
        if (w.step != dep || w.lo != lo || w.hi != hi || go != (dep < kvq::kSearchSteps)) { ++bad; continue; }
        if (!go) continue;
        // every lane's path
        double want[32], got[32];
        for (int p = 0; p < 32; ++p) want[p] = got[p] = -7.0;
        for (int L = 0; L < 32; ++L) {
            double a = lo, b = hi;
            int u = 0, pre = 0;
            for (int d = dep; d < kvq::kSearchSteps && u < 5; ++d) {
                const double m = 0.5 * (a + b);
                int k = ref_known(s, m);
                if (k < 0) {
                    want[(1 << u) - 1 + pre] = m;
                    k = ((L >> (4 - u)) & 1) == 0;
                    pre = 2 * pre + (k ? 0 : 1);
                    ++u;
                }
                if (k) b = m; else a = m;
            }
            kvq::search_path(w, L, got);
        }
        for (int p = 0; p < 32; ++p) if (kvq::dbits(want[p]) != kvq::dbits(got[p])) { ++bad; break; }
    }
    return bad;
}
extern "C" void kvqs_f32_bounds(const float *f, long n, unsigned long long *lo,
                                unsigned long long *hi) {
    for (long i = 0; i < n; ++i) {
        lo[i] = f[i] > 0.f ? kvq::f32_low_bits(f[i]) : 0ull;
        hi[i] = f[i] < INFINITY ? kvq::f32_high_bits(f[i]) : 0ull;
    }
}
extern "C" long long kvqs_budget_fx(double B) { return kvq::budget_fx(B); }
static double Rfun(double lam, int nbp, const double *bl, const double *br, double R0) {
    double r = R0;
    for (int i = 0; i < nbp; ++i) if (lam >= bl[i]) r = br[i];
    return r;
}
// pilot_bias < 0: no pilot; else the pilot sees R * (1 + pilot_bias) on 1/16 of the blocks
extern "C" int kvqs_run(double hi0, double B, int nbp, const double *bl, const double *br,
                        double R0, double *out, double pilot_bias, int f32) {
    kvq::SearchState s;
    kvq::search_init(s);
    s.hi0 = hi0;
    s.f32_lambda = f32 == 1;          // f32 = 2: R at float(lambda), rule off
    const int64_t nb = 4096;
    if (pilot_bias >= 0.0 || pilot_bias <= -1.0) {}
    if (pilot_bias > -1.0) kvq::search_set_pilot(s, nb, 16);
    int r = 0;
    for (; r < 64 && s.phase != kvq::kSearchDone; ++r) {
        long long R[kvq::kSearchProbes];
        const bool pilot = s.phase == kvq::kSearchPilot;
        for (int p = 0; p < kvq::kSearchProbes; ++p) {
            double lam = kvq::search_probe(s, p);
            if (f32) lam = (double)(float)lam;          // R sees lambda only as binary32
            double v = p < s.nprobe || pilot ? Rfun(lam, nbp, bl, br, R0) : 0.0;
            if (pilot) v = v * (1.0 + pilot_bias) * (double)s.pilot_blocks / (double)nb;
            R[p] = fx(v);
        }
        kvq::search_update(s, R, B, nb);
    }
    out[0] = s.lambda; out[1] = s.xb; out[2] = (double)s.R_xb / 1048576.0; out[3] = r;
    out[4] = s.infeasible; out[5] = s.step;
    return s.phase == kvq::kSearchDone ? 0 : 1;
}
'''


@pytest.fixture(scope="module")
def lib():
    d = tempfile.mkdtemp(prefix="kvqs_")
    src = os.path.join(d, "shim.cpp")
    so = os.path.join(d, "libshim.so")
    with open(src, "w") as f:
        f.write(SHIM)
    subprocess.check_call(["g++", "-O2", "-std=c++17", "-ffp-contract=off", "-fPIC", "-shared",
                           "-I", CSRC, "-o", so, src])
    L = C.CDLL(so)
    L.kvqs_half_sum_check.restype = C.c_long
    L.kvqs_half_sum_check.argtypes = [C.c_void_p, C.c_void_p, C.c_long, C.POINTER(C.c_long)]
    L.kvqs_okey_check.restype = C.c_long
    L.kvqs_okey_check.argtypes = [C.c_void_p, C.c_void_p, C.c_long]
    L.kvqs_pow2_scale.restype = C.c_double
    L.kvqs_pow2_scale.argtypes = [C.c_double, C.c_int]
    L.kvqs_path_check.restype = C.c_long
    L.kvqs_path_check.argtypes = [C.c_void_p, C.c_long]
    L.kvqs_f32_bounds.restype = None
    L.kvqs_f32_bounds.argtypes = [C.c_void_p, C.c_long, C.c_void_p, C.c_void_p]
    L.kvqs_budget_fx.restype = C.c_longlong
    L.kvqs_budget_fx.argtypes = [C.c_double]
    L.kvqs_run.restype = C.c_int
    L.kvqs_run.argtypes = [C.c_double, C.c_double, C.c_int, C.c_void_p, C.c_void_p, C.c_double,
                           C.c_void_p, C.c_double, C.c_int]
    return L


def R_of(lam, bl, br, R0):
    r = R0
    for a, v in zip(bl, br):
        if lam >= a:
            r = v
    return r


def bisect40(hi0, B, bl, br, R0, f32=False):
    """The sequential reading: lambda = 0 if feasible, else doubling, then 40 steps
    (f32: R evaluated at the binary32 rounding of lambda, as on the GPU)."""
    if f32:
        R = lambda lam: R_of(float(np.float32(lam)), bl, br, R0)
    else:
        R = lambda lam: R_of(lam, bl, br, R0)
    if R(0.0) <= B:
        return 0.0, 0
    hi, n = hi0, 0
    while R(hi) > B and n < 30:
        hi *= 2.0
        n += 1
    if R(hi) > B:
        return hi, 1
    lo = 0.0
    for _ in range(40):
        mid = 0.5 * (lo + hi)
        if R(mid) <= B:
            hi = mid
        else:
            lo = mid
    return hi, 0


def run(lib, hi0, B, bl, br, R0, pilot=-2.0, f32=0):
    out = (C.c_double * 6)()
    a = (C.c_double * len(bl))(*bl)
    b = (C.c_double * len(br))(*br)
    rc = lib.kvqs_run(hi0, B, len(bl), a, b, R0, out, pilot, f32)
    assert rc == 0
    return list(out)


def random_case(rng):
    hi0 = 10 ** rng.uniform(-2, 6)
    n = rng.randint(1, 400)
    # breakpoints spread over many decades below and a little above hi0
    bl = sorted(hi0 * 10 ** rng.uniform(-14, 0.7) for _ in range(n))
    R0 = 1e6
    br, r = [], R0
    for _ in bl:
        r -= rng.uniform(0, 2 * R0 / n)
        # rates are fixed-point sums (multiples of 2^-20 bit)
        br.append(round(max(r, 0.0) * 2 ** 20) / 2 ** 20)
    return hi0, bl, br, R0


def test_same_lambda_as_sequential_bisection(lib):
    rng = random.Random(0)
    rounds = []
    for _ in range(3000):
        hi0, bl, br, R0 = random_case(rng)
        B = rng.uniform(0, R0)
        want, infeasible = bisect40(hi0, B, bl, br, R0)
        lam, xb, Rxb, nr, inf, step = run(lib, hi0, B, bl, br, R0)
        assert lam == want, (hi0, B)
        assert inf == infeasible
        if not infeasible:
            assert Rxb <= B
            assert R_of(xb, bl, br, R0) == Rxb
            # the chosen allocation (at xb) and the reported lambda are within
            # the bisection's final interval
            assert lam == 0.0 or want - hi0 * 2 ** -39 <= xb <= want
        rounds.append(nr)
    assert sum(rounds) / len(rounds) < 8


def test_binary32_lambda_rule_keeps_the_bisection(lib):
    # when R sees lambda only through float(lambda), midpoints that round to
    # float(xa) or float(xb) are known without an evaluation: same lambda as
    # the 40 sequential steps of that R, in no more rounds
    rng = random.Random(11)
    saved = 0
    for _ in range(1500):
        hi0, bl, br, R0 = random_case(rng)
        # breakpoints close together near the answer, where binary32 matters
        B = rng.uniform(0, R0)
        want, infeasible = bisect40(hi0, B, bl, br, R0, f32=True)
        lam, xb, Rxb, nr, inf, step = run(lib, hi0, B, bl, br, R0, f32=1)
        assert lam == want, (hi0, B)
        assert inf == infeasible
        plain = run(lib, hi0, B, bl, br, R0, f32=2)
        assert plain[0] == want
        if not infeasible:
            assert Rxb <= B
        assert nr <= plain[3]
        saved += plain[3] - nr
    assert saved > 0


@pytest.mark.parametrize("bias", [0.0, 0.05, -0.05, 0.4, -0.4])
def test_pilot_estimate_never_changes_lambda(lib, bias):
    # the pilot (a biased estimate of R on a sample of blocks) only places the
    # probes of round 0; the answer is the sequential bisection's either way
    rng = random.Random(5)
    for _ in range(800):
        hi0, bl, br, R0 = random_case(rng)
        B = rng.uniform(0, R0)
        want, infeasible = bisect40(hi0, B, bl, br, R0)
        out = run(lib, hi0, B, bl, br, R0, pilot=bias)
        assert out[0] == want
        assert out[4] == infeasible


def test_budget_at_zero_lambda_and_large_hi(lib):
    # R(0) <= B: lambda = 0 in one round
    out = run(lib, 5.0, 100.0, [1.0], [50.0], 90.0)
    assert out[0] == 0.0 and out[3] == 1
    # only feasible after several doublings: one extra round
    bl, br = [40.0 * 5.0], [10.0]
    want, _ = bisect40(5.0, 20.0, bl, br, 90.0)
    out = run(lib, 5.0, 20.0, bl, br, 90.0)
    assert out[0] == want and out[3] <= 12
    # never feasible: status infeasible, lambda = hi0 * 2^30
    out = run(lib, 5.0, 1.0, [1.0], [50.0], 90.0)
    assert out[4] == 1 and out[0] == 5.0 * 2 ** 30
    # hi0 = 0 (all blocks constant): R = 0 <= B
    out = run(lib, 0.0, 0.0, [], [], 0.0)
    assert out[0] == 0.0


def _d(u):
    return struct.unpack("<d", struct.pack("<Q", u))[0]


def _pairs(rng, n):
    """Non-negative binary64 pairs that exercise every rounding case of
    a + b: random exponent gaps 0..60, random and extreme significands,
    exact half-ulp ties with odd and even b, carries, zeros, and a > b."""
    e = rng.integers(900, 1150, n)
    gap = rng.integers(0, 61, n)
    fa = rng.integers(0, 1 << 52, n, dtype=np.uint64)
    fb = rng.integers(0, 1 << 52, n, dtype=np.uint64)
    kind = rng.integers(0, 6, n)
    ones = np.uint64((1 << 52) - 1)
    fa = np.where(kind == 1, ones, fa)                       # all-ones: carries
    fb = np.where(kind == 1, ones, fb)
    fa = np.where(kind == 2, np.uint64(0), fa)               # a a power of two
    ub = (e.astype(np.uint64) << np.uint64(52)) | fb
    ua = (np.maximum(e - gap, 1).astype(np.uint64) << np.uint64(52)) | fa
    # ties: a exactly half an ulp of b (gap 53, a a power of two), b odd or even
    tie = kind == 3
    ua = np.where(tie, ((e - 53).astype(np.uint64) << np.uint64(52)), ua)
    ub = np.where(tie & (rng.integers(0, 2, n) == 1), ub | np.uint64(1), ub)
    a = ua.view(np.float64).copy()
    b = ub.view(np.float64).copy()
    a = np.where(kind == 4, 0.0, a)                          # lo = 0
    swap = rng.integers(0, 2, n) == 1                        # either order
    a2 = np.where(swap, b, a)
    b2 = np.where(swap, a, b)
    a2 = np.where(kind == 5, b2, a2)                         # a == b
    return np.ascontiguousarray(a2), np.ascontiguousarray(b2)


def test_half_sum_rounds_as_binary64(lib):
    rng = np.random.default_rng(3)
    a, b = _pairs(rng, 400000)
    first = C.c_long()
    bad = lib.kvqs_half_sum_check(a.ctypes.data, b.ctypes.data, len(a), C.byref(first))
    assert bad == 0, (bad, a[first.value], b[first.value])
    # the midpoints of real bisections over random brackets
    xs, ys = [], []
    r = random.Random(1)
    for _ in range(2000):
        lo, hi = 0.0, r.uniform(1e-9, 1e9)
        for _ in range(40):
            mid = 0.5 * (lo + hi)
            xs.append(lo)
            ys.append(hi)
            if r.random() < 0.5:
                hi = mid
            else:
                lo = mid
    xa, ya = np.array(xs), np.array(ys)
    assert lib.kvqs_half_sum_check(xa.ctypes.data, ya.ctypes.data, len(xa), C.byref(first)) == 0


def test_okey_orders_as_binary64(lib):
    rng = np.random.default_rng(4)
    a = rng.standard_normal(200000) * 10.0 ** rng.integers(-30, 30, 200000)
    b = np.where(rng.random(200000) < 0.2, a, rng.standard_normal(200000) * 1e3)
    a[:4] = [np.inf, -np.inf, -1.0, 0.0]
    b[:4] = [1e308, -1e308, -1.0, 1e-300]
    assert lib.kvqs_okey_check(a.ctypes.data, b.ctypes.data, len(a)) == 0


def test_pow2_scale_and_budget_fixed_point(lib):
    for x in (0.0, 1.0, 3.7e-12, 1.234e10, _d(0x0010000000000000), _d(1)):
        for t in (-40, -3, 0, 5, 30):
            assert lib.kvqs_pow2_scale(x, t) == np.ldexp(x, t)
    assert lib.kvqs_budget_fx(2.5) == 2621440
    assert lib.kvqs_budget_fx(0.1) == int(np.floor(0.1 * 2 ** 20))
    assert lib.kvqs_budget_fx(1e300) == 2 ** 63 - 1
    for B in (0.0, 3.0, 83886080.0, 123456.789):
        fxB = lib.kvqs_budget_fx(B)
        # R <= B  iff  R_fx <= floor(B 2^20), for integer R_fx
        for R in (fxB - 1, fxB, fxB + 1):
            assert (R / 2 ** 20 <= B) == (R <= fxB)


def test_binary32_rounding_bounds(lib):
    """The raw-bit bounds of the walk's binary32 rule: the smallest double that
    rounds to f rounds to f and its predecessor does not; the largest one
    rounds to f and its successor does not (ties to even on both sides,
    subnormals, zero, the largest finite value and +inf included)."""
    rng = np.random.default_rng(6)
    bits = rng.integers(0, 0x7F800000, 200000, dtype=np.uint32)
    bits[:8] = [0, 1, 2, 3, 0x007FFFFF, 0x00800000, 0x7F7FFFFF, 0x3F800000]
    bits[8:4096] = (bits[8:4096] & 0x7F800000) | rng.integers(0, 2, 4088).astype(np.uint32)
    f = np.concatenate([bits.view(np.float32), np.array([np.inf], dtype=np.float32)])
    lo = np.zeros(len(f), dtype=np.uint64)
    hi = np.zeros(len(f), dtype=np.uint64)
    lib.kvqs_f32_bounds(f.ctypes.data, len(f), lo.ctypes.data, hi.ctypes.data)
    to32 = lambda u: u.view(np.float64).astype(np.float32)
    with np.errstate(over="ignore"):
        pos = f > 0
        assert np.array_equal(to32(lo[pos]), f[pos])
        assert np.all(to32(lo[pos] - np.uint64(1)) < f[pos])
        fin = np.isfinite(f)
        assert np.array_equal(to32(hi[fin]), f[fin])
        assert np.all(to32(hi[fin] + np.uint64(1)) > f[fin])


def test_walk_and_probe_paths_follow_the_definition(lib):
    """search_walk and search_path (integer midpoints, raw-bit window tests)
    against 0.5 (lo + hi) and double / binary32 comparisons, on brackets from
    real bisections: lo = 0 or a midpoint, windows from far wider than the
    bracket to a few binary32 ulps (where the binary32 rule decides), answers
    near powers of two (brackets across binades) and tiny or huge scales."""
    rng = random.Random(7)
    rows = []
    for i in range(6000):
        scale = 10 ** rng.uniform(-12, 12)
        lam = scale * rng.uniform(0.5, 2.0)
        if i % 5 == 0:
            lam = 2.0 ** rng.randint(-30, 30) * (1 + rng.choice([-1, 1]) * 10 ** rng.uniform(-9, -2))
        hi = 2.0 ** math.ceil(math.log2(lam) + rng.randint(0, 3))
        lo = 0.0
        for _ in range(rng.randint(0, 30)):      # some steps of the true bisection
            mid = 0.5 * (lo + hi)
            if mid >= lam:
                hi = mid
            else:
                lo = mid
        width = lam * 10 ** rng.uniform(-9.5, -0.5)
        if rng.random() < 0.2:
            ulp = float(np.spacing(np.float32(lam)))
            width = ulp * rng.uniform(0.5, 6.0)
        xa = lam - width * rng.uniform(0.05, 1.0)
        xb = lam + width * rng.uniform(0.05, 1.0)
        xa = max(xa, lo) if rng.random() < 0.5 else xa
        if rng.random() < 0.1:
            xa = -1.0                            # nothing infeasible known yet
        if not (xa < xb):
            continue
        rows.append((lo, hi, xa, xb, float(rng.random() < 0.6)))
    a = np.ascontiguousarray(np.array(rows, dtype=np.float64).ravel())
    assert lib.kvqs_path_check(a.ctypes.data, len(rows)) == 0
