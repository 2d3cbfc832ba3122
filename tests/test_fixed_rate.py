"""The fixed-rate comparator ("Rate-adaptive KV-cache quantizer",
"Implementation notes": compare against fixed-rate entropy coding at equal
total cache bytes): every block runs the 40-step bisection on its own lambda_r
with the budget b d_r, so each block, not only the total, meets the rate.

Oracle pins (CPU): on tiny blocks, the bisection restated in Python over the
element-by-element brute-force optimum (tests/bruteforce.py) gives the same
lambda_r and chain; every block meets its budget and, unless lambda_r = 0, is
over it at the interval's infeasible end; a constant block takes lambda_r = 0;
the comparator spends no more than the rate-adaptive allocation at the same
total budget and, on the synthetic layer, distorts more.
GPU parity (marked gpu): kvq_allocate_fixed_rate against the oracle: every
block within its budget; lambda_r within 2e-3 relative (one block's crossing
of two chains is conditioned by how close their rates are); wherever lambda_r
differs by more than 1e-4 or the chain differs, the GPU's chain is one of the
chains tied at the oracle's crossing (objective at the oracle's lambda_r
within 2e-5 of the optimum); D_r and H_r within 1e-4 where the chains agree;
total distortion within 1e-4.
"""
import numpy as np
import pytest
import torch

import oracle
import bruteforce as bf
from rate_adaptive_kv_block_b300 import kvq, synth


def _bisect_py(v, s, budget):
    """The bisection of the page's one global lambda applied to one block,
    on the brute-force optimum: R(0) <= budget -> 0; hi = (c_max - c_min)^2,
    doubled at most 30 times; 40 steps of mid = 0.5 (lo + hi); hi."""
    def rate(lam):
        return bf.best_chain(v, s, lam)[3]
    if rate(0.0) <= budget:
        return 0.0
    c = bf.candidates(v)
    lo, hi = 0.0, (c[-1] - c[0]) ** 2
    n = 0
    while rate(hi) > budget and n < 30:
        hi *= 2.0
        n += 1
    for _ in range(40):
        mid = 0.5 * (lo + hi)
        if rate(mid) <= budget:
            hi = mid
        else:
            lo = mid
    return hi


def _tiny(seed, nblocks, d):
    rng = np.random.default_rng(seed)
    out = []
    for b in range(nblocks):
        if b % 3 == 0:
            v = rng.standard_normal(d) * np.exp(rng.standard_normal())
        elif b % 3 == 1:
            v = rng.standard_t(3, d)
        else:
            v = np.round(rng.standard_normal(d) * 2) / 2           # ties
        out.append(v.astype(np.float16))
    return out


@pytest.mark.parametrize("s,bpe", [(3, 1.2), (4, 1.5), (5, 1.8)])
def test_fixed_rate_matches_bruteforce_bisection(s, bpe):
    blocks = _tiny(7 + s, 6, 32)
    x = np.stack(blocks).reshape(len(blocks), 32, 1).view(np.uint16)   # G = 1: d = 32
    r = oracle.allocate_fixed_rate(x, 1, s, bpe)
    assert r["status"] == 0
    for b, v in enumerate(blocks):
        vd = v.astype(np.float64)
        lam = _bisect_py(vd, s, bpe * 32)
        assert r["lambdas"][b] == lam
        obj, ch, D, R, obj2 = bf.best_chain(vd, s, lam)
        assert r["mask"][b] == bf.mask_of(ch) or obj2 - obj <= 1e-12 * abs(obj)
        assert R <= bpe * 32 + 1e-9
        assert r["H_r"][b] * 32 == pytest.approx(R, rel=1e-12, abs=1e-12)
        assert r["D_r"][b] == pytest.approx(D, rel=1e-12, abs=1e-12)


def test_fixed_rate_budget_per_block_and_constant_block():
    w = synth.workload("llama3_8b_layer", T=128)
    x = synth.make_numpy(w, seed=3)
    x[0, :32, :] = np.float16(0.5).view(np.uint16)                  # block 0: constant
    bpe = 2.5
    r = oracle.allocate_fixed_rate(x, w.G, w.s, bpe)
    d = 32 * w.G
    assert r["status"] == 0
    assert np.all(r["H_r"] * d <= bpe * d + 1e-6)                   # every block meets it
    assert r["lambdas"][0] == 0.0 and r["k"][0] == 1
    # unless lambda_r = 0, the block is over its budget at the bisection's
    # infeasible end, lambda_r minus the final interval width
    for b in range(1, 12):
        lam = r["lambdas"][b]
        if lam == 0.0:
            continue
        ids = [b]
        st = oracle.stats(x, w.G, b0=b, nb=1)
        h0 = (st["cand"][0][st["mprime"][0] - 1] - st["cand"][0][0]) ** 2
        n = 0
        while h0 * 2 ** n < lam:
            n += 1
        lo = lam - h0 * 2 ** n / 2 ** 40
        assert oracle.rate_at(x, w.G, w.s, lo, ids=ids) > bpe * d
        assert oracle.rate_at(x, w.G, w.s, lam, ids=ids) <= bpe * d


def test_fixed_rate_against_rate_adaptive():
    # same total budget: the fixed-rate allocation spends at most as much
    # (each block is capped) and the one global lambda distorts less
    w = synth.workload("llama3_8b_layer", T=256)
    x = synth.make_numpy(w, seed=0)
    bpe = 2.5
    f = oracle.allocate_fixed_rate(x, w.G, w.s, bpe)
    g = oracle.allocate_bisect(x, w.G, w.s, bpe * x.size)
    assert f["totals"][0] <= bpe * x.size
    assert g["totals"][0] <= bpe * x.size
    assert g["totals"][1] < f["totals"][1]
    # one block alone: the same as the global bisection over that block
    for b in (0, 5, 17):
        one = oracle.allocate_bisect(x, w.G, w.s, bpe * 32 * w.G, ids=[b])
        assert one["lambda"] == f["lambdas"][b]


# ------------------------------------------------------------------ GPU

@pytest.mark.gpu
@pytest.mark.parametrize("name,T,S,bi", [("llama3_8b_layer", 512, None, 0),
                                         ("hadamard_groups", 256, None, 1),
                                         ("k_head_small", None, None, 0)])
def test_fixed_rate_gpu_matches_oracle(name, T, S, bi):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import gpu_common as gc
    w = synth.workload(name, T=T, S=S)
    x = synth.make_numpy(w, seed=4)
    L = kvq.Layout(w.S, w.T, w.D, w.G)
    bpe = w.budgets[bi]
    xd = gc.to_dev(x)
    buf = kvq.Buffers(L, w.s)
    kvq.kvq_stats(xd, L, buf.stats, buf.status_stats)
    lams = torch.zeros(L.nblocks, dtype=torch.float64, device="cuda")
    kvq.kvq_allocate_fixed_rate(buf.stats, L, w.s, bpe, buf.codebook, buf.k, buf.D_r, buf.H_r,
                                lams, buf.totals, buf.status)
    torch.cuda.synchronize()
    assert int(buf.status.item()) == 0
    o = oracle.allocate_fixed_rate(x, w.G, w.s, bpe)
    lg = lams.cpu().numpy()
    lo = o["lambdas"]
    both0 = (lg == 0) & (lo == 0)
    rel = np.where(both0, 0.0, np.abs(lg - lo) / np.maximum(np.abs(lo), 1e-300))
    # lambda_r is one block's crossing of two chains, lambda* = dD / dR: the
    # DP's binary32 objective error (about 16 * 2^-24 of the objective O ~ 2
    # lambda R) moves it by about 2e-6 R / dR relative, large when the two
    # chains' rates are close; the global lambda averages this over every
    # block, one block's does not
    assert np.all(rel <= 2e-3), rel.max()
    d = 32 * w.G
    H = buf.H_r.cpu().numpy().astype(np.float64)
    assert np.all(H * d <= bpe * d * (1 + 1e-6))
    cb, kk = buf.codebook.cpu().numpy(), buf.k.cpu().numpy()
    Dg = buf.D_r.cpu().numpy().astype(np.float64)
    same = np.all(cb == o["codebook"], axis=1) & (kk == o["k"])
    # where lambda_r or the chain differs, the GPU's chain is one of the two
    # chains tied at the oracle's crossing: its objective at the oracle's
    # lambda_r is the optimum's within the fp32 tolerance of the tie rule
    for b in np.nonzero(~same | (rel > gc.LAM_REL))[0]:
        mp, cand, _, _, _ = oracle.block_tables(x, w.G, int(b))
        m = gc.chain_mask_from_codebook(cand, mp, cb[b], int(kk[b]))
        Dc, Rc = oracle.chain_cost(x, w.G, int(b), m)
        obj_g = Dc + lo[b] * Rc
        obj_o = o["D_r"][b] + lo[b] * o["H_r"][b] * d
        assert obj_g <= obj_o * (1 + 2 * gc.GAP) + 1e-9, (b, rel[b], obj_g, obj_o)
    okD = np.abs(Dg - o["D_r"]) <= np.maximum(gc.DH_REL * np.abs(o["D_r"]), 1e-6)
    okH = np.abs(H - o["H_r"]) <= np.maximum(gc.DH_REL * np.abs(o["H_r"]), 1e-6)
    assert (okD | ~same).all() and (okH | ~same).all()
    assert np.sum(Dg) == pytest.approx(np.sum(o["D_r"]), rel=1e-4)
    tot = buf.totals.cpu().numpy()
    assert tot[0] == pytest.approx(np.sum(H * d), rel=1e-6)
    assert tot[1] == pytest.approx(np.sum(Dg), rel=1e-6)
