"""Distortion weighted by attention sensitivity ("Rate-adaptive KV-cache
quantizer", "Implementation notes": optionally weight D_r by the sensitivity
measured on a calibration batch).  D_r = sum_e w_e (q_hi - x_e)(x_e - q_lo)
with caller-supplied w_e >= 0; H_r stays the entropy of the unweighted
expected codepoint frequencies.

Oracle pins (none compares the oracle with itself): the element-by-element
brute force over every admissible level subset with weights; the weighted atom
moments from their definition; unit weights give the unweighted results
exactly; a power-of-two weight c scales D_r by c and lambda by c exactly; a
constant weight per block is the unweighted choice at lambda / w; the weighted
D_r is the expectation of sum w (hat x - x)^2 over the interpolation's
randomness (Monte Carlo over seeds); zero weights leave only the rate, so the
chain of least rate wins (brute force); invalid weights are flagged.
GPU: weighted stats rows against the oracle, the allocation, codes, repeated
calls bit-identical, edge weights and the status words.
"""
import numpy as np
import pytest

import oracle
import bruteforce as bf
from rate_adaptive_kv_block_b300 import synth


def tiny_x(blocks):
    a = np.asarray(blocks, dtype=np.float16).reshape(len(blocks), 32, 1)
    return a.view(np.uint16)


def f16(v):
    return np.asarray(v, dtype=np.float16).astype(np.float64)


def tiny_blocks(rng):
    return [rng.standard_normal(32),
            np.round(rng.standard_normal(32) * 2) / 2,
            rng.standard_t(2, 32),
            np.concatenate([np.zeros(28), [1.0, -1.0, 3.0, 0.5]])]


def tiny_weights(rng, n):
    w = np.exp(1.5 * rng.standard_normal((n, 32))).astype(np.float32)
    w[:, rng.permutation(32)[:5]] = 0.0           # some entries do not matter
    return w


# ------------------------------------------------------------------ oracle

@pytest.mark.parametrize("s", [2, 3, 5])
def test_weighted_dp_matches_bruteforce_tiny(s):
    rng = np.random.default_rng(200 + s)
    blocks = tiny_blocks(rng)
    W = tiny_weights(rng, len(blocks))
    x = tiny_x(blocks)
    w = W.reshape(len(blocks), 32, 1)
    for lam in (0.0, 0.01, 0.1, 1.0, 10.0):
        got = oracle.allocate_at(x, 1, s, lam, w=w)
        for b, raw in enumerate(blocks):
            obj, ch, D, R, obj2 = bf.best_chain(f16(raw), s, lam, W[b].astype(np.float64))
            go = got["D_r"][b] + lam * got["H_r"][b] * 32
            assert go == pytest.approx(obj, rel=1e-10, abs=1e-12)
            if obj2 - obj > 1e-9 * max(abs(obj), 1e-12):
                assert got["mask"][b] == bf.mask_of(ch)
                assert got["D_r"][b] == pytest.approx(D, rel=1e-10, abs=1e-12)
                assert got["H_r"][b] * 32 == pytest.approx(R, rel=1e-10, abs=1e-12)


def test_weighted_atoms_from_definition():
    rng = np.random.default_rng(21)
    blocks = tiny_blocks(rng)
    W = tiny_weights(rng, len(blocks))
    st = oracle.stats(tiny_x(blocks), 1, w=W.reshape(-1, 32, 1))
    for b, raw in enumerate(blocks):
        v = f16(raw)
        c = bf.candidates(v)
        mp = len(c)
        assert st["mprime"][b] == mp
        want = np.zeros((16, 4))
        for e in range(32):
            # atom p: c_p <= x < c_{p+1}; the maximum joins the last atom
            p = max(j for j in range(mp - 1) if c[j] <= v[e])
            y, t = v[e] - c[p], c[p + 1] - v[e]
            want[p] += W[b, e] * np.array([1.0, y, t, y * t])
        assert np.allclose(st["atoms"][b], want, rtol=1e-12, atol=1e-12)


def test_unit_weights_are_the_unweighted_method():
    w = synth.workload("llama3_8b_layer", T=64, S=4)
    x = synth.make_numpy(w, seed=22)
    ones = np.ones(x.shape, dtype=np.float32)
    a, b = oracle.stats(x, w.G), oracle.stats(x, w.G, w=ones)
    assert np.array_equal(a["atoms"], b["atoms"]) and np.array_equal(a["cand"], b["cand"])
    B = 2.5 * x.size
    r0 = oracle.allocate_bisect(x, w.G, 16, B)
    r1 = oracle.allocate_bisect(x, w.G, 16, B, w=ones)
    assert r0["lambda"] == r1["lambda"]
    for key in ("codebook", "k", "D_r", "H_r", "mask", "totals"):
        assert np.array_equal(r0[key], r1[key]), key


def test_power_of_two_weight_scales_lambda_exactly():
    # D -> c D with c = 2^3 leaves every comparison of D + lambda R at
    # lambda c unchanged; the bisection's bracket starts at c max W^2 and only
    # halves, so lambda_w = c lambda exactly.
    w = synth.workload("hadamard_groups", T=64, S=2)
    x = synth.make_numpy(w, seed=23)
    B = 2.0 * x.size
    r0 = oracle.allocate_bisect(x, w.G, 16, B)
    r1 = oracle.allocate_bisect(x, w.G, 16, B, w=np.full(x.shape, 8.0, dtype=np.float32))
    assert r1["lambda"] == 8.0 * r0["lambda"] and r0["lambda"] > 0
    assert np.array_equal(r0["mask"], r1["mask"])
    assert np.array_equal(r1["D_r"], 8.0 * r0["D_r"])
    assert np.array_equal(r0["H_r"], r1["H_r"])


def test_block_constant_weight_is_a_lambda_rescale():
    # argmin w D + lam R = argmin D + (lam / w) R
    w = synth.workload("llama3_8b_layer", T=64, S=2)
    x = synth.make_numpy(w, seed=24)
    nb = oracle.num_blocks(*x.shape, w.G)
    rng = np.random.default_rng(24)
    om = np.exp(rng.standard_normal(nb)).astype(np.float32)
    W = np.repeat(om.reshape(x.shape[0], -1), 32, axis=1)[:, :, None] * np.ones((1, 1, x.shape[2]), np.float32)
    lam = 0.05
    got = oracle.allocate_at(x, w.G, 16, lam, w=W)
    checked = 0
    for b in range(nb):
        ref = oracle.allocate_at(x, w.G, 16, lam / float(om[b]), ids=[b])
        if ref["gap"][0] > 1e-9:
            assert got["mask"][b] == ref["mask"][0]
            assert got["D_r"][b] == pytest.approx(float(om[b]) * ref["D_r"][0], rel=1e-12)
            checked += 1
    assert checked >= nb - 2


def test_weighted_distortion_is_the_expected_weighted_error():
    rng = np.random.default_rng(25)
    raw = rng.standard_normal(32)
    Wb = tiny_weights(rng, 1)[0]
    x = tiny_x([raw])
    r = oracle.allocate_at(x, 1, 4, 0.02, w=Wb.reshape(1, 32, 1))
    v = f16(raw)
    N = 20000
    tot = np.empty(N)
    for seed in range(N):
        cd = oracle.quantize(x, 1, r["codebook"], r["k"], seed)
        codes = np.stack([cd & 15, cd >> 4], axis=-1).reshape(-1)
        xh = r["codebook"][0][codes].astype(np.float64)
        tot[seed] = np.sum(Wb * (xh - v) ** 2)
    se = tot.std() / np.sqrt(N)
    assert abs(tot.mean() - r["D_r"][0]) < 4 * se + 1e-12


def test_zero_weights_leave_the_rate_alone():
    # D_r = 0 for every chain: at lambda > 0 the chain of least rate wins
    # (brute force over every admissible chain), at lambda = 0 every chain
    # ties and the fewest levels win; the other blocks are unaffected.
    rng = np.random.default_rng(26)
    blocks = tiny_blocks(rng)
    x = tiny_x(blocks)
    W = np.ones((len(blocks), 32, 1), dtype=np.float32)
    W[1] = 0.0
    v = f16(blocks[1])
    c = bf.candidates(v)
    rmin = min(bf.chain_cost_elementwise(v, c[list(ch)])[1] for ch in bf.all_chains(len(c), 8))
    for lam in (0.0, 0.3):
        got = oracle.allocate_at(x, 1, 8, lam, w=W)
        ref = oracle.allocate_at(x, 1, 8, lam)
        assert got["D_r"][1] == 0.0
        if lam == 0.0:
            assert got["k"][1] == 2
        else:
            assert got["H_r"][1] * 32 == pytest.approx(rmin, rel=1e-12)
        keep = [0, 2, 3]
        assert np.array_equal(got["mask"][keep], ref["mask"][keep])


def test_invalid_weights_are_flagged():
    rng = np.random.default_rng(27)
    blocks = tiny_blocks(rng)
    x = tiny_x(blocks)
    for bad in (-1.0, np.nan, np.inf):
        W = np.ones((len(blocks), 32, 1), dtype=np.float32)
        W[2, 5, 0] = bad
        st = oracle.stats(x, 1, w=W)
        assert list(st["nonfinite"]) == [0, 0, 2, 0]
        assert oracle.allocate_at(x, 1, 8, 0.1, w=W)["status"] == 8
    # an invalid weight outranks a non-finite value
    xb = x.copy()
    xb[0, 0, 0] = 0x7c00
    assert oracle.allocate_at(xb, 1, 8, 0.1, w=W)["status"] == 8
    assert oracle.allocate_at(xb, 1, 8, 0.1)["status"] == 3


def test_weighted_choice_is_optimal_for_the_weighted_objective():
    # At the weighted bisection's lambda, no block does better (in the weighted
    # objective) with the codebook the unweighted method picks at that lambda.
    w = synth.workload("llama3_8b_layer", T=32, S=4)
    x = synth.make_numpy(w, seed=28)
    W = synth.weights_numpy(w, seed=28)
    rw = oracle.allocate_bisect(x, w.G, 16, 2.5 * x.size, w=W)
    lam = rw["lambda"]
    ru = oracle.allocate_at(x, w.G, 16, lam)
    d = 32 * w.G
    for b in range(len(rw["k"])):
        Du, Ru = oracle.chain_cost(x, w.G, b, int(ru["mask"][b]), w=W)
        assert rw["D_r"][b] + lam * rw["H_r"][b] * d <= Du + lam * Ru * (1 + 1e-12) + 1e-12


# --------------------------------------------------------------------- GPU

def _gpu():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


WCASES = [("k_head_small", None, None), ("llama3_8b_layer", 512, None),
          ("hadamard_groups", 256, None)]


@pytest.mark.gpu
@pytest.mark.parametrize("name,T,S", WCASES)
def test_weighted_stats_and_allocation_match_oracle(name, T, S):
    _gpu()
    import gpu_common as gc
    wl = synth.workload(name, T=T, S=S)
    x = synth.make_numpy(wl, seed=31)
    W = synth.weights_numpy(wl, seed=31)
    B = wl.budgets[0] * x.size
    g = gc.run(x, wl.G, wl.s, B, seed=5, w=W)
    assert g["status_stats"] == 0 and g["status"] == 0
    assert np.all(g["flags"] == 4)                              # weighted rows
    gc.check_stats(g, oracle.stats(x, wl.G, w=W), weighted=True)
    ora = oracle.allocate_bisect(x, wl.G, wl.s, B, w=W)
    assert g["lambda"] == pytest.approx(ora["lambda"], rel=gc.LAM_REL)
    gc.check_choice(g, x, wl.G, wl.s, g["lambda"], w=W)
    gc.check_codes(g, x, wl.G, 5, 0)


@pytest.mark.gpu
def test_weighted_small_groups_and_repeatable():
    _gpu()
    import torch
    import gpu_common as gc
    from rate_adaptive_kv_block_b300 import kvq
    wl = synth.workload("k_head_small", T=128, S=4)
    x = synth.make_numpy(wl, seed=32)
    W = synth.weights_numpy(wl, seed=32)
    for G in (8, 32):
        g = gc.run(x, G, 16, 3.0 * x.size, w=W)
        gc.check_stats(g, oracle.stats(x, G, w=W), weighted=True)
        gc.check_choice(g, x, G, 16, g["lambda"], w=W)
    # repeated calls give identical stats bytes
    L = kvq.Layout(*x.shape, 128)
    xd, wd = gc.to_dev(x), torch.from_numpy(W).cuda()
    outs = []
    for _ in range(2):
        st = torch.zeros(kvq.kvq_stats_bytes(L), dtype=torch.uint8, device="cuda")
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        kvq.kvq_stats_weighted(xd, wd, L, st, status)
        outs.append(st.cpu().numpy())
    assert np.array_equal(outs[0], outs[1])


@pytest.mark.gpu
def test_weighted_edge_weights_and_status():
    _gpu()
    import gpu_common as gc
    from rate_adaptive_kv_block_b300 import kvq
    r = np.random.default_rng(33)
    x = (r.standard_normal((6, 32, 128)) * np.exp(r.standard_normal((6, 1, 128)))).astype(np.float16)
    x = x.view(np.uint16)
    W = np.ones(x.shape, dtype=np.float32)
    W[0] = 0.0                                      # a block that does not matter
    W[1] = 1e20                                     # huge
    W[2] = 1e-30                                    # tiny
    W[3] = np.where(r.random((32, 128)) < 0.9, 0.0, 5.0)   # sparse
    W[4, :, :64] = 3.0                              # half the features
    B = 2.5 * x.size
    g = gc.run(x, 128, 16, B, w=W)
    assert g["status_stats"] == 0 and g["status"] == 0
    gc.check_stats(g, oracle.stats(x, 128, w=W), weighted=True)
    ora = oracle.allocate_bisect(x, 128, 16, B, w=W)
    assert g["lambda"] == pytest.approx(ora["lambda"], rel=gc.LAM_REL)
    gc.check_choice(g, x, 128, 16, g["lambda"], w=W)
    assert g["D_r"][0] == 0.0                       # no weight, no distortion
    # all weights zero: lambda 0, the fewest levels everywhere
    g0 = gc.run(x, 128, 16, B, w=np.zeros(x.shape, dtype=np.float32))
    assert g0["status"] == 0 and g0["lambda"] == 0.0 and np.all(g0["k"] == 2)
    # invalid weights: both status words report it
    for bad in (-2.0, np.nan, np.inf):
        Wb = W.copy()
        Wb[5, 7, 9] = bad
        gb = gc.run(x, 128, 16, B, w=Wb)
        assert gb["status_stats"] == kvq.KVQ_ERR_BAD_WEIGHT
        assert gb["status"] == kvq.KVQ_ERR_BAD_WEIGHT
        assert gb["flags"][5] & 2 and not (gb["flags"][:5] & 2).any()


@pytest.mark.gpu
def test_weighted_bench_layer_full_size():
    """The bench's weighted leg exactly: the full layer (4096 blocks), its
    input and its sensitivities, every block against the oracle."""
    _gpu()
    import gpu_common as gc
    wl = synth.workload("llama3_8b_layer")
    x = synth.make_numpy(wl, seed=0)
    W = synth.weights_torch(wl, seed=7).cpu().numpy()
    B = wl.budgets[0] * x.size
    g = gc.run(x, wl.G, wl.s, B, seed=0, w=W)
    assert g["status_stats"] == 0 and g["status"] == 0
    assert g["totals"][0] <= B
    gc.check_stats(g, oracle.stats(x, wl.G, w=W), weighted=True)
    ora = oracle.allocate_bisect(x, wl.G, wl.s, B, w=W)
    assert g["lambda"] == pytest.approx(ora["lambda"], rel=gc.LAM_REL)
    gc.check_choice(g, x, wl.G, wl.s, g["lambda"], w=W)
    gc.check_codes(g, x, wl.G, 0, 0)


@pytest.mark.gpu
@pytest.mark.parametrize("mode", [0, 1])
def test_weighted_fused_and_subgradient(mode):
    """With weighted stats, kvq_allocate_quantize gives exactly kvq_allocate +
    kvq_quantize (bisection and one subgradient step), and the subgradient
    step is the oracle's weighted one-step map."""
    _gpu()
    import torch
    from rate_adaptive_kv_block_b300 import kvq
    wl = synth.workload("llama3_8b_layer", T=1024)
    x = synth.make_numpy(wl, seed=43)
    W = synth.weights_numpy(wl, seed=43)
    xd = torch.from_numpy(x.view(np.int16)).view(torch.float16).cuda()
    wd = torch.from_numpy(W).cuda()
    L = kvq.Layout(*x.shape, wl.G)
    B = 2.5 * x.size
    lam0, eta = (0.0, 0.0) if mode == kvq.KVQ_BISECT40 else (0.12, 1e-7)
    ref, got = kvq.Buffers(L, 16), kvq.Buffers(L, 16)
    for b in (ref, got):
        b.lam.fill_(lam0)
    kvq.quantize(xd, L, B, 16, seed=3, mode=mode, eta=eta, buf=ref, weights=wd)
    kvq.quantize(xd, L, B, 16, seed=3, mode=mode, eta=eta, buf=got, weights=wd, fused=True)
    torch.cuda.synchronize()
    assert int(ref.status.item()) == 0 and int(got.status.item()) == 0
    for key in ("codebook", "k", "D_r", "H_r", "totals", "lam", "codes"):
        a, b = getattr(ref, key), getattr(got, key)
        assert torch.equal(a.view(torch.uint8), b.view(torch.uint8)), key
    if mode == kvq.KVQ_SUBGRADIENT:
        o = oracle.allocate_at(x, wl.G, 16, lam0, eta, B, w=W)
        assert float(ref.lam.item()) == pytest.approx(o["lambda_next"], rel=1e-4, abs=eta * 1e-4 * B)


def test_synthetic_sensitivities_have_the_attention_structure():
    # keys: one weight per (stream, feature), the same for every token;
    # values: one weight per (stream, token), the same for every feature;
    # every stream's mean is 1, every weight positive and finite
    wl = synth.workload("llama3_8b_layer", T=128, S=6)
    W = synth.weights_numpy(wl, seed=3)
    assert W.shape == (6, 128, 128) and W.dtype == np.float32
    assert np.all(np.isfinite(W)) and np.all(W > 0)
    nk = 3
    assert np.all(W[:nk] == W[:nk, :1, :])                  # per feature
    assert np.all(W[nk:] == W[nk:, :, :1])                  # per token
    assert np.allclose(W.reshape(6, -1).mean(axis=1), 1.0, rtol=1e-5)
    assert np.all(W[nk:, :4, 0] > W[nk:, 4:, 0].mean(axis=1, keepdims=True))   # sink tokens
