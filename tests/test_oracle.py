"""Pins of the CPU oracle against what the page and the mathematics fix.

None of these compare the oracle with itself: each checks it against a
published value, a closed form, an invariant of the optimisation, or the
element-by-element brute force of tests/bruteforce.py.
"""
import math
import os

import numpy as np
import pytest

import oracle
import bruteforce as bf
from rate_adaptive_kv_block_b300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def golden(name):
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            k, v = line.split()[:2]
            out[k] = float(v)
    return out


def tiny_x(blocks):
    """[S=nblocks, T=32, D=1] binary16 tensor, block b = stream b (G = 1)."""
    a = np.asarray(blocks, dtype=np.float16).reshape(len(blocks), 32, 1)
    return a.view(np.uint16)


def f16(v):
    return np.asarray(v, dtype=np.float16).astype(np.float64)


# --------------------------------------------------------------------- hash

# Known-answer vectors of the Philox4x32 block function published with the
# Random123 library (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as
# easy as 1, 2, 3", SC 2011): rounds, counter (4 words), key (2 words) ->
# output (4 words).
PHILOX_KAT = [
    (7, [0, 0, 0, 0], [0, 0], [0x5F6FB709, 0x0D893F64, 0x4F121F81, 0x4F730A48]),
    (10, [0, 0, 0, 0], [0, 0], [0x6627E8D5, 0xE169C58D, 0xBC57AC4C, 0x9B00DBD8]),
    (10, [0xFFFFFFFF] * 4, [0xFFFFFFFF] * 2, [0x408F276D, 0x41C83B0E, 0xA20BC7C6, 0x6D5451FD]),
    (10, [0x243F6A88, 0x85A308D3, 0x13198A2E, 0x03707344], [0xA4093822, 0x299F31D0],
     [0xD16CFE09, 0x94FDCCEB, 0x5001E420, 0x24126EA1]),
]


@pytest.mark.parametrize("rounds,ctr,key,want", PHILOX_KAT)
def test_philox_published_vectors(rounds, ctr, key, want):
    assert oracle.philox4x32(ctr, key, rounds) == want


def test_hash_is_philox7_word_of_the_counter_block():
    # hash(seed, i) = word i mod 4 of Philox4x32-7 at counter (i >> 2 as two
    # 32-bit words, 0, 0) and key (seed as two 32-bit words)
    assert [oracle.hash32(0, i) for i in range(4)] == PHILOX_KAT[0][3]
    for seed, c in [(1, 0), (0x123456789ABCDEF0, 5), (7, (1 << 38) + 3), (2 ** 64 - 1, 2 ** 40 // 4)]:
        want = oracle.philox4x32([c & 0xFFFFFFFF, c >> 32, 0, 0],
                                 [seed & 0xFFFFFFFF, seed >> 32], 7)
        assert [oracle.hash32(seed, 4 * c + j) for j in range(4)] == want
    assert list(oracle.hash_many(9, 4 * 77, 8)) == [oracle.hash32(9, 4 * 77 + j) for j in range(8)]


def _find_index(seed, pred, start=0, n=1 << 18):
    h = oracle.hash_many(seed, start, n)
    hits = np.nonzero(pred(h >> 8))[0]
    assert len(hits), "no index found"
    return start + int(hits[0]), int(h[hits[0]] >> 8)


def test_rounding_rule_is_strict_at_a_tie():
    # Levels 0 and 1: w = 1, so fl(u 2^-24 * w) = u 2^-24 exactly.  For an
    # index whose u has at most 11 significant bits, x = u 2^-24 is a binary16
    # value and the rule's two sides are equal: the entry must stay at the
    # lower level (choose q_{i+1} only when fl(t w) < fl(x - q_i)); one
    # binary16 step above x it must move up, one step below it must not.
    seed = 4242
    idx, u = _find_index(seed, lambda u: ((u & 0x1FFF) == 0) & (u >= (1 << 13)))
    x_tie = u * 2.0 ** -24
    assert float(np.float16(x_tie)) == x_tie
    up = float(np.nextafter(np.float16(x_tie), np.float16(1)))
    dn = float(np.nextafter(np.float16(x_tie), np.float16(0)))
    q = np.zeros((1, 16), dtype=np.float32)
    q[0, 1:] = 1.0
    k = np.array([2], dtype=np.uint8)
    for xv, want in [(x_tie, 0), (up, 1), (dn, 0)]:
        # block of 32 x 1 entries (G = 1): put the value at the entry whose
        # global index is idx (index_base = idx - e for entry e = 0)
        x = np.zeros((1, 32, 1), dtype=np.float16)
        x[0, 0, 0] = xv
        x[0, 1:, 0] = 0.5
        codes = oracle.quantize(x.view(np.uint16), 1, q, k, seed, idx)
        assert codes[0, 0] & 15 == want, (xv, want)


def test_rounding_rule_uses_the_interval_below_a_level():
    # x equal to a level: interval i is the largest with q_i <= x (capped at
    # k-2), and under the rule the code is exactly that level whatever u is
    q = np.array([[-1.0, 0.25, 0.5, 3.0] + [3.0] * 12], dtype=np.float32)
    k = np.array([4], dtype=np.uint8)
    x = np.tile(np.array([-1.0, 0.25, 0.5, 3.0], dtype=np.float16), 8).reshape(1, 32, 1)
    for seed in range(20):
        codes = oracle.quantize(x.view(np.uint16), 1, q, k, seed, 4 * seed)
        c = np.stack([codes[0] & 15, codes[0] >> 4], axis=-1).reshape(-1)
        assert np.array_equal(c, np.tile([0, 1, 2, 3], 8))


def test_hash_uniform_chi2():
    n = 1 << 20
    u = oracle.hash_many(12345, 1 << 33, n) >> 8          # 24-bit uniforms
    bins = np.bincount((u >> 16).astype(np.int64), minlength=256)
    exp = n / 256
    chi2 = float(((bins - exp) ** 2 / exp).sum())
    # 255 dof: mean 255, sd ~22.6; 5 sd either side
    assert 255 - 5 * 22.6 < chi2 < 255 + 5 * 22.6
    # low bits too, and consecutive pairs are not correlated
    bins = np.bincount((u & 255).astype(np.int64), minlength=256)
    chi2 = float(((bins - exp) ** 2 / exp).sum())
    assert 255 - 5 * 22.6 < chi2 < 255 + 5 * 22.6
    a = u[0::2].astype(np.float64)
    b = u[1::2].astype(np.float64)
    assert abs(np.corrcoef(a, b)[0, 1]) < 5 / math.sqrt(n / 2)


# ------------------------------------------------------------------ binary16

def test_f16_decode_matches_numpy():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    for h in range(0, 1 << 16, 7):
        v = oracle.f16_to_double(h)
        r = ref[h]
        if np.isnan(r):
            assert math.isnan(v)
        else:
            assert v == r
            if np.isfinite(r):
                hh, ok = oracle.double_to_f16(v)
                assert ok
                assert np.uint16(hh).view(np.float16) == np.float16(r)


# ---------------------------------------------------------------- candidates

@pytest.mark.parametrize("G", [1, 8, 32, 128])
def test_candidates_are_sorted_ranks(G):
    rng = np.random.default_rng(G)
    S, T, D = 2, 64, max(G, 8) * 2
    vals = rng.standard_normal((S, T, D)).astype(np.float16)
    vals[0, :, :4] = 0.5                         # ties inside blocks
    vals[1, 3:9, :] = -0.0                       # -0 among +0 values
    vals[1, 9:12, :] = 0.0
    x = vals.view(np.uint16)
    st = oracle.stats(x, G)
    d = 32 * G
    nb = oracle.num_blocks(S, T, D, G)
    for b in range(nb):
        v = [float(np.float16(vals.reshape(-1)[oracle.flat_index(T, D, G, b, e)]))
             for e in range(d)]
        s = sorted(v)
        want = []
        for j in range(17):
            a = s[(j * (d - 1) + 8) // 16]
            if not want or a != want[-1]:
                want.append(a)
        mp = st["mprime"][b]
        assert mp == len(want)
        assert list(st["cand"][b, :mp]) == want
        assert all(st["cand"][b, mp:] == want[-1])


# ------------------------------------------------ interval tables and atoms

def test_chain_cost_matches_elementwise():
    rng = np.random.default_rng(1)
    blocks = [rng.standard_normal(32), rng.standard_t(3, 32),
              np.round(rng.standard_normal(32) * 3)]      # ties
    x = tiny_x(blocks)
    for b in range(len(blocks)):
        v = f16(blocks[b])
        c = bf.candidates(v)
        for _ in range(40):
            inner = [j for j in range(1, len(c) - 1) if rng.random() < 0.4]
            ch = [0] + inner + [len(c) - 1]
            D1, R1 = oracle.chain_cost(x, 1, b, bf.mask_of(ch))
            D2, R2, _ = bf.chain_cost_elementwise(v, c[ch])
            assert D1 == pytest.approx(D2, rel=1e-12, abs=1e-12)
            assert R1 == pytest.approx(R2, rel=1e-12, abs=1e-12)


def test_atoms_reassemble_interval_tables():
    # Identity: for a = c_P < b = c_Q, sum over atoms p in [P, Q) of
    # n A B + A t1 + B s1 + e (A = c_p - a, B = b - c_{p+1}) equals
    # sum (b - x)(x - a) over the interval, and the masses split as
    # sum(s1 + n A)/W and sum(t1 + n B)/W.
    w = synth.workload("llama3_8b_layer", T=64)
    x = synth.make_numpy(w, seed=3)
    st = oracle.stats(x, w.G, 0, 6)
    for b in range(6):
        mp, cand, Dpq, Mup, Mdn = oracle.block_tables(x, w.G, b)
        assert mp == st["mprime"][b]
        c = st["cand"][b]
        at = st["atoms"][b]
        assert at[:mp - 1, 0].sum() == 32 * w.G
        for P in range(mp):
            for Q in range(P + 1, mp):
                a, bb = c[P], c[Q]
                Dv = Up = Dn = 0.0
                for p in range(P, Q):
                    n, s1, t1, e = at[p]
                    A, B = c[p] - a, bb - c[p + 1]
                    Dv += n * A * B + A * t1 + B * s1 + e
                    Up += s1 + n * A
                    Dn += t1 + n * B
                W = bb - a
                assert Dv == pytest.approx(Dpq[P, Q], rel=1e-9)
                assert Up / W == pytest.approx(Mup[P, Q], rel=1e-9, abs=1e-9)
                assert Dn / W == pytest.approx(Mdn[P, Q], rel=1e-9, abs=1e-9)


def test_distortion_slope_minus_two():
    # Page "Verification": distortion ~ (k-1)^-2, observed slope -2.000.
    # Closed form: for x uniform on [0, L] and k equally spaced levels of
    # spacing W = L/(k-1), D/d -> W^2/6.
    g = golden("page1_verification.txt")
    d = 4096
    v = np.linspace(0.0, 8.0, d).astype(np.float16)
    x = v.reshape(1, 32, 128).view(np.uint16)
    c = bf.candidates(f16(v))
    assert len(c) == 17
    ks, Ds = [], []
    for km1 in (1, 2, 4, 8, 16):
        ch = list(range(0, 17, 16 // km1))
        Dr, _ = oracle.chain_cost(x, 128, 0, bf.mask_of(ch))
        W = (c[-1] - c[0]) / km1
        assert Dr / d == pytest.approx(W * W / 6, rel=0.02)
        ks.append(km1)
        Ds.append(Dr)
    slope = np.polyfit(np.log(ks), np.log(Ds), 1)[0]
    assert slope == pytest.approx(g["distortion_slope_vs_levels_minus_1"], abs=0.01)


# ---------------------------------------------------------- the choice (DP)

@pytest.mark.parametrize("s", [2, 3, 5, 16])
def test_dp_matches_bruteforce_tiny(s):
    rng = np.random.default_rng(100 + s)
    blocks = [rng.standard_normal(32),
              np.round(rng.standard_normal(32) * 2) / 2,     # few distinct
              rng.standard_t(2, 32),
              np.concatenate([np.zeros(30), [1.0, -1.0]])]
    if s == 16:
        blocks = blocks[:2]          # 2^15 chains each: keep it quick
    x = tiny_x(blocks)
    for lam in (0.0, 0.01, 0.1, 1.0, 10.0):
        got = oracle.allocate_at(x, 1, s, lam)
        for b, raw in enumerate(blocks):
            v = f16(raw)
            obj, ch, D, R, obj2 = bf.best_chain(v, s, lam)
            go = got["D_r"][b] + lam * got["H_r"][b] * 32
            assert go == pytest.approx(obj, rel=1e-10, abs=1e-12)
            if obj2 - obj > 1e-9 * max(abs(obj), 1e-12):
                assert got["mask"][b] == bf.mask_of(ch)
                assert got["D_r"][b] == pytest.approx(D, rel=1e-10, abs=1e-12)
            gap = got["gap"][b]
            if np.isfinite(obj2) and obj > 0:
                assert gap == pytest.approx((obj2 - obj) / obj, rel=1e-6, abs=1e-9)


def test_dp_real_block_beats_sampled_chains():
    w = synth.workload("llama3_8b_layer", T=32)
    x = synth.make_numpy(w, seed=5)
    ids = [0, 9]                                   # one K block, one V block
    rng = np.random.default_rng(0)
    for lam in (0.02, 0.2):
        got = oracle.allocate_at(x, w.G, 16, lam, ids=ids)
        for i, b in enumerate(ids):
            d = 32 * w.G
            v = np.array([f16(x.view(np.float16).reshape(-1)[oracle.flat_index(w.T, w.D, w.G, b, e)])
                          for e in range(d)])
            c = bf.candidates(v)
            mask = int(got["mask"][i])
            ch = [j for j in range(len(c)) if mask >> j & 1]
            assert 2 <= len(ch) <= 16 and ch[0] == 0 and ch[-1] == len(c) - 1
            D, R, _ = bf.chain_cost_elementwise(v, c[ch])
            best = D + lam * R
            assert got["D_r"][i] == pytest.approx(D, rel=1e-9)
            assert got["H_r"][i] * d == pytest.approx(R, rel=1e-9)
            for _ in range(300):
                inner = sorted(rng.choice(np.arange(1, len(c) - 1),
                                          size=rng.integers(0, 15), replace=False))
                D2, R2, _ = bf.chain_cost_elementwise(v, c[[0] + list(inner) + [len(c) - 1]])
                assert best <= D2 + lam * R2 + 1e-9 * best


def test_lambda_crossings_are_analytic():
    # Page "Verification": lambda transitions match the analytically
    # predicted crossings.  Walking lambda upwards, each switch from the
    # optimal chain A to its successor B sits at (D_A - D_B) / (R_B - R_A).
    rng = np.random.default_rng(7)
    blocks = [rng.standard_normal(32) * 0.3, rng.standard_normal(32) * 2.0]
    x = tiny_x(blocks)
    g = golden("page1_verification.txt")

    def at(lam, b):
        r = oracle.allocate_at(x, 1, 8, lam, ids=[b])
        return int(r["mask"][0]), r["D_r"][0], r["H_r"][0] * 32

    for b in range(len(blocks)):
        seen = 0
        lam, top = 1e-4, 1e2
        cur = at(lam, b)
        grid = list(np.geomspace(lam, top, 60)[1:])
        while grid:
            nxt = grid[0]
            other = at(nxt, b)
            if other[0] == cur[0]:
                lam, cur = nxt, other
                grid.pop(0)
                continue
            lo, hi = lam, nxt                     # first switch out of cur
            for _ in range(80):
                mid = 0.5 * (lo + hi)
                if at(mid, b)[0] == cur[0]:
                    lo = mid
                else:
                    hi = mid
            succ = at(hi, b)
            lam_star = (cur[1] - succ[1]) / (succ[2] - cur[2])
            assert abs(lam_star - hi) <= 1e-9 * hi
            assert abs(hi - lam_star) / lam_star < g["lambda_transition_tolerance"]
            seen += 1
            lam, cur = hi, succ
        assert seen >= 2


def test_rate_nonincreasing_in_lambda():
    w = synth.workload("llama3_8b_layer", T=64)
    x = synth.make_numpy(w, seed=11)
    ids = list(range(0, 32, 3))
    Rs = [oracle.rate_at(x, w.G, 16, lam, ids=ids) for lam in np.geomspace(1e-4, 1e3, 30)]
    assert all(a >= b for a, b in zip(Rs, Rs[1:]))
    assert Rs[0] > Rs[-1]


def test_high_variance_block_gets_more_levels():
    # Page "Verification": adaptive allocation gave fewer levels to the
    # low-variance block and more to the high-variance block.
    rng = np.random.default_rng(2)
    lo = (0.1 * rng.standard_normal((1, 32, 128))).astype(np.float16)
    hi = (1.0 * rng.standard_normal((1, 32, 128))).astype(np.float16)
    x = np.concatenate([lo, hi]).view(np.uint16)
    r = oracle.allocate_bisect(x, 128, 16, 2.0 * x.size)
    assert r["status"] == 0
    assert r["k"][1] > r["k"][0]
    assert r["H_r"][1] > r["H_r"][0]


def test_dual_separability_bruteforce():
    # Page "Mathematical statement": with lambda the blocks decouple, so the
    # joint minimum of sum_r (D_r + lambda d_r H_r) is the sum of the block
    # minima.  Joint brute force over every pair of chains of two blocks.
    rng = np.random.default_rng(4)
    blocks = [np.round(rng.standard_normal(32) * 2), np.round(rng.standard_normal(32))]
    x = tiny_x(blocks)
    lam = 0.05
    per = []
    for raw in blocks:
        v = f16(raw)
        c = bf.candidates(v)
        per.append([sum(bf.chain_cost_elementwise(v, c[list(ch)])[:2] * np.array([1, lam]))
                    for ch in bf.all_chains(len(c), 4)])
    joint = min(a + b for a in per[0] for b in per[1])
    got = oracle.allocate_at(x, 1, 4, lam)
    total = got["totals"][1] + lam * got["totals"][0]
    assert total == pytest.approx(joint, rel=1e-12)


# ----------------------------------------------------------- global lambda

def test_bisection_properties():
    w = synth.workload("llama3_8b_layer", T=96)
    x = synth.make_numpy(w, seed=21)
    B = 2.5 * x.size
    r = oracle.allocate_bisect(x, w.G, 16, B)
    lam = r["lambda"]
    lo, hi = r["bracket"]
    assert r["status"] == 0
    assert lam == hi and lo < hi
    assert r["totals"][0] <= B                                # budget met
    assert oracle.rate_at(x, w.G, 16, lo) > B                 # lo infeasible
    st = oracle.stats(x, w.G)
    h0 = max((c[m - 1] - c[0]) ** 2 for c, m in zip(st["cand"], st["mprime"]))
    n = 0
    while h0 * 2 ** n < hi:
        n += 1
    assert (hi - lo) == pytest.approx(h0 * 2 ** n / 2 ** 40, rel=1e-9)
    assert r["totals"][0] == pytest.approx(np.sum(r["H_r"] * 32 * w.G), rel=1e-12)
    assert r["totals"][1] == pytest.approx(np.sum(r["D_r"]), rel=1e-12)


def test_bisection_lambda_zero_and_infeasible():
    w = synth.workload("k_head_small", T=64, S=2)
    x = synth.make_numpy(w, seed=2)
    r = oracle.allocate_bisect(x, w.G, 8, 100.0 * x.size)
    assert r["status"] == 0 and r["lambda"] == 0.0
    assert np.all(r["k"] == 8)
    r = oracle.allocate_bisect(x, w.G, 8, 0.0)
    assert r["status"] == 4                                   # infeasible


def test_subgradient_one_step():
    # Page "Key formulas": lambda <- max{0, lambda + eta (sum d_r H_r - B)}.
    w = synth.workload("k_head_small", T=64, S=2)
    x = synth.make_numpy(w, seed=8)
    for lam, eta, B in [(0.1, 1e-6, 2.5 * x.size), (0.1, 1e-3, 1e9), (0.0, 1e-6, 0.0)]:
        r = oracle.allocate_at(x, w.G, 16, lam, eta, B)
        R = r["totals"][0]
        assert r["lambda_next"] == max(0.0, lam + eta * (R - B))
    r = oracle.allocate_at(x, w.G, 16, 0.05, 1.0, 1e12)
    assert r["lambda_next"] == 0.0                            # clamp at zero


# ------------------------------------------- stochastic interpolation (a7)

def _exact_pup(xv, q0, q1):
    """Exact P(choose q1) over the 2^24-point u grid, in the fp32 rule."""
    xv, q0, q1 = np.float32(xv), np.float32(q0), np.float32(q1)
    w = np.float32(q1 - q0)
    r = np.float32(xv - q0)
    lo, hi = 0, 1 << 24                   # count u with fl(fl(u 2^-24) w) < r
    while lo < hi:
        mid = (lo + hi) // 2
        if np.float32(np.float32(mid * 2.0 ** -24) * w) < r:
            lo = mid + 1
        else:
            hi = mid
    return lo / float(1 << 24)


def test_conditional_mean_exact_expectation():
    # Page "Key formulas" / "Verification": E[hat x | x] = x.  With a 24-bit
    # uniform the exact expectation is within w 2^-24 of x (the page's toy
    # reports 8.9e-16 with continuous uniforms).
    rng = np.random.default_rng(9)
    for _ in range(200):
        q0, q1 = np.sort(rng.standard_normal(2).astype(np.float16).astype(np.float64))
        if q0 == q1:
            continue
        xv = float(np.float16(rng.uniform(q0, q1)))
        p = _exact_pup(xv, q0, q1)
        mean = q0 + p * (q1 - q0)
        assert abs(mean - xv) <= (q1 - q0) * 2.0 ** -24 * 1.0001
        mse = (1 - p) * (xv - q0) ** 2 + p * (q1 - xv) ** 2
        assert mse == pytest.approx((q1 - xv) * (xv - q0), rel=1e-6, abs=(q1 - q0) ** 2 * 2.0 ** -23)


def test_unbiased_monte_carlo_over_seeds():
    # Mean and MSE of hat x over 10^5 seeds against the closed forms.
    rng = np.random.default_rng(10)
    vals = rng.standard_normal((1, 32, 8)).astype(np.float16)
    x = vals.view(np.uint16)
    q = np.array([-1.5, -0.25, 0.5, 2.0], dtype=np.float16).astype(np.float32)
    cb = np.zeros((1, 16), dtype=np.float32)
    cb[0, :4] = q
    cb[0, 4:] = q[-1]
    k = np.array([4], dtype=np.uint8)
    v = vals.reshape(-1).astype(np.float64)
    inside = (v >= q[0]) & (v <= q[-1])
    N = 100000
    s1 = np.zeros(256)
    s2 = np.zeros(256)
    for seed in range(N):
        c = oracle.quantize(x, 8, cb, k, seed)
        codes = np.stack([c & 15, c >> 4], axis=-1).reshape(-1)
        xh = q[codes].astype(np.float64)
        s1 += xh
        s2 += (xh - v) ** 2
    i = np.clip(np.searchsorted(q, v, side="right") - 1, 0, 2)
    var = (q[i + 1] - v) * (v - q[i])
    mean = s1 / N
    z = (mean - v) / np.sqrt(np.maximum(var, 1e-30) / N)
    z = z[inside & (var > 0)]
    assert np.mean(np.abs(z) > 3) < 0.02 and np.max(np.abs(z)) < 5
    mse = s2 / N
    ok = inside & (var > 0)
    assert np.all(np.abs(mse[ok] - var[ok]) < 5 * np.sqrt(var[ok] * (q[i + 1] - q[i])[ok] ** 2 / N) + 1e-12)


def test_entropy_from_expected_frequencies():
    # H_r uses expected frequencies (page "Implementation notes"): they sum to
    # d, and the empirical code frequencies over many seeds converge to them.
    rng = np.random.default_rng(12)
    raw = rng.standard_normal(32)
    x = tiny_x([raw])
    r = oracle.allocate_at(x, 1, 4, 0.05)
    v = f16(raw)
    c = bf.candidates(v)
    mask = int(r["mask"][0])
    ch = [j for j in range(len(c)) if mask >> j & 1]
    D, R, M = bf.chain_cost_elementwise(v, c[ch])
    assert M.sum() == pytest.approx(32, rel=1e-12)
    assert r["H_r"][0] * 32 == pytest.approx(R, rel=1e-12)
    cnt = np.zeros(len(ch))
    N = 20000
    for seed in range(N):
        cd = oracle.quantize(x, 1, r["codebook"], r["k"], seed)
        codes = np.stack([cd & 15, cd >> 4], axis=-1).reshape(-1)
        cnt += np.bincount(codes, minlength=len(ch))[:len(ch)]
    freq = cnt / (N * 32)
    assert np.allclose(freq, M / 32, atol=4 * np.sqrt(0.25 / (N * 32)))
    # two-point data: all mass on the two levels -> binary entropy
    two = tiny_x([np.concatenate([np.zeros(24), np.ones(8)])])
    r2 = oracle.allocate_at(two, 1, 4, 0.0)
    p = 8 / 32
    assert r2["H_r"][0] == pytest.approx(-(p * math.log2(p) + (1 - p) * math.log2(1 - p)), rel=1e-12)
    assert r2["D_r"][0] == 0.0


def test_pack_layout_and_decode():
    rng = np.random.default_rng(13)
    vals = rng.standard_normal((1, 32, 8)).astype(np.float16)
    x = vals.view(np.uint16)
    r = oracle.allocate_at(x, 8, 6, 0.01)
    codes = oracle.quantize(x, 8, r["codebook"], r["k"], seed=3, index_base=1 << 20)
    assert codes.shape == (1, 128)
    v = vals.reshape(-1).astype(np.float32)
    q = r["codebook"][0]
    k = int(r["k"][0])
    for e in range(256):
        c = (codes[0, e // 2] >> (4 * (e & 1))) & 15
        assert c < k
        # the chosen level is one of the two ends of x's interval
        i = min(max(np.searchsorted(q[:k], v[e], side="right") - 1, 0), k - 2)
        assert c in (i, i + 1)
    y = oracle.dequantize(codes, r["codebook"], (1, 32, 8), 8)
    yv = y.view(np.float16).reshape(-1)
    for e in range(256):
        c = (codes[0, e // 2] >> (4 * (e & 1))) & 15
        assert yv[e] == np.float16(q[c])


# --------------------------------------------------------------- edge cases

def test_constant_and_two_valued_blocks():
    x = tiny_x([np.full(32, 0.75), np.concatenate([np.full(16, -1.0), np.full(16, 2.0)])])
    st = oracle.stats(x, 1)
    assert list(st["mprime"]) == [1, 2]
    r = oracle.allocate_bisect(x, 1, 16, 1.0 * x.size)
    assert r["k"][0] == 1 and r["D_r"][0] == 0 and r["H_r"][0] == 0
    assert np.all(r["codebook"][0] == np.float32(0.75))
    assert r["k"][1] == 2 and r["D_r"][1] == 0 and r["H_r"][1] == pytest.approx(1.0)
    codes = oracle.quantize(x, 1, r["codebook"], r["k"], seed=1)
    assert np.all(codes[0] == 0)
    y = oracle.dequantize(codes, r["codebook"], (2, 32, 1), 1)
    assert np.array_equal(y, x)          # both blocks lie on their levels


def test_nonfinite_flag():
    vals = np.random.default_rng(0).standard_normal((2, 32, 8)).astype(np.float16)
    vals[1, 5, 3] = np.inf
    x = vals.view(np.uint16)
    st = oracle.stats(x, 8)
    assert list(st["nonfinite"]) == [0, 1]
    assert oracle.allocate_bisect(x, 8, 8, 3.0 * x.size)["status"] == 3
