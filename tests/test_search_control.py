"""The lambda-search control (csrc/kvq_search.h, compiled for the host here)
walks exactly the fixed 40-step bisection: on monotone step functions R it
returns the same lambda as the sequential bisection, bit for bit, whatever the
breakpoints; and it needs far fewer rounds of evaluations than 40."""
import ctypes as C
import os
import random
import subprocess
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "rate_adaptive_kv_block_b300", "csrc")

SHIM = r'''
#include "kvq_search.h"
static double Rfun(double lam, int nbp, const double *bl, const double *br, double R0) {
    double r = R0;
    for (int i = 0; i < nbp; ++i) if (lam >= bl[i]) r = br[i];
    return r;
}
// pilot_bias < 0: no pilot; else the pilot sees R * (1 + pilot_bias) on 1/16 of the blocks
extern "C" int kvqs_run(double hi0, double B, int nbp, const double *bl, const double *br,
                        double R0, double *out, double pilot_bias) {
    kvq::SearchState s;
    kvq::search_init(s);
    s.hi0 = hi0;
    const int64_t nb = 4096;
    if (pilot_bias >= 0.0 || pilot_bias <= -1.0) {}
    if (pilot_bias > -1.0) kvq::search_set_pilot(s, nb, 16);
    int r = 0;
    for (; r < 64 && s.phase != kvq::kSearchDone; ++r) {
        double R[kvq::kSearchProbes];
        const bool pilot = s.phase == kvq::kSearchPilot;
        for (int p = 0; p < kvq::kSearchProbes; ++p) {
            double v = p < s.nprobe || pilot ? Rfun(kvq::search_probe(s, p), nbp, bl, br, R0) : 0.0;
            if (pilot) v = v * (1.0 + pilot_bias) * (double)s.pilot_blocks / (double)nb;
            R[p] = v;
        }
        kvq::search_update(s, R, B, nb);
    }
    out[0] = s.lambda; out[1] = s.xb; out[2] = s.R_xb; out[3] = r;
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
    L.kvqs_run.restype = C.c_int
    L.kvqs_run.argtypes = [C.c_double, C.c_double, C.c_int, C.c_void_p, C.c_void_p, C.c_double,
                           C.c_void_p, C.c_double]
    return L


def R_of(lam, bl, br, R0):
    r = R0
    for a, v in zip(bl, br):
        if lam >= a:
            r = v
    return r


def bisect40(hi0, B, bl, br, R0):
    """The sequential reading: lambda = 0 if feasible, else doubling, then 40 steps."""
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


def run(lib, hi0, B, bl, br, R0, pilot=-2.0):
    out = (C.c_double * 6)()
    a = (C.c_double * len(bl))(*bl)
    b = (C.c_double * len(br))(*br)
    rc = lib.kvqs_run(hi0, B, len(bl), a, b, R0, out, pilot)
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
        br.append(max(r, 0.0))
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
