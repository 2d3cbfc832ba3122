"""Parity of the CUDA path with the oracle at the workloads' full sizes, every
block checked.

  * full_model_cache: 32 layers x {K, V} x 8 heads x 32768 tokens x 128
    (524 288 blocks of 4096), s = 16, B = 2.0 bits/entry, one global lambda;
  * hadamard_groups: 8 heads x 131072 tokens x 128 after the 128-point
    Hadamard rotation, 32-feature groups (131 072 blocks of 1024), s = 16,
    the budget sweep 1.5 / 2 / 3 / 4 bits/entry on one kvq_stats result;
  * decode_admission: 64 sequences x 32 layers x {K, V} x 8 heads appending
    one 32-token block each (32 768 blocks of 4096) per step, lambda from the
    40-step bisection at step 0, then 8 subgradient steps
    lambda <- max(0, lambda + eta (sum_r d_r H_r - B)), eta = 1e-6, B = 2.5.

Rules ("Rate-adaptive KV-cache quantizer": one global lambda coupling the
blocks, "Mathematical statement"; the lambda update, "Key formulas"): lambda
within 1e-4 relative of the oracle's 40-step bisection (or, for a subgradient
step, of the oracle's one-step map from the GPU's lambda_t); at the GPU's
lambda, codebook and k equal to the oracle's on every block whose best-vs-
second objective gap exceeds 1e-5 relative, D_r and H_r within 1e-4; codes bit
for bit on several thousand blocks (contiguous runs at seeded offsets).

The inputs are drawn on the device (torch Philox, seeded) and copied to the
host for the oracle.  Each case costs minutes of the oracle's CPU time, so
these tests carry the extra marker `full` (deselect with -m "gpu and not
full" for quick runs).
"""
import numpy as np
import pytest
import torch

import oracle
import gpu_common as gc
from rate_adaptive_kv_block_b300 import kvq, synth

pytestmark = [pytest.mark.gpu, pytest.mark.full]

CODE_RUNS = 4            # contiguous runs of blocks whose codes are compared
CODE_RUN_BLOCKS = 1024


def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _host(buf):
    return {
        "codebook": buf.codebook.cpu().numpy(),
        "k": buf.k.cpu().numpy(),
        "D_r": buf.D_r.cpu().numpy().astype(np.float64),
        "H_r": buf.H_r.cpu().numpy().astype(np.float64),
        "totals": buf.totals.cpu().numpy(),
        "lambda": float(buf.lam.item()),
        "status": int(buf.status.item()),
    }


def _check_codes(x_np, G, g_codes, g, seed, index_base, rng):
    """Codes of CODE_RUNS runs of CODE_RUN_BLOCKS consecutive blocks: the
    oracle quantizes with the GPU's codebooks."""
    nb = g["k"].shape[0]
    run = min(CODE_RUN_BLOCKS, nb)
    starts = sorted(set([0] + [int(v) for v in rng.integers(0, nb - run + 1, size=CODE_RUNS - 1)]))
    for b0 in starts:
        want = oracle.quantize(x_np, G, g["codebook"][b0:b0 + run], g["k"][b0:b0 + run], seed,
                               index_base, b0, run)
        got = g_codes[b0:b0 + run].cpu().numpy()
        assert np.array_equal(want, got), "codes differ in %d blocks of the run at %d" % (
            np.any(want != got, axis=1).sum(), b0)


def _check_lambda(lam_g, lam_o):
    assert abs(lam_g - lam_o) <= gc.LAM_REL * abs(lam_o), (lam_g, lam_o)


def _check_totals(g, d):
    assert g["totals"][0] == pytest.approx(np.sum(g["H_r"] * d), rel=1e-6)
    assert g["totals"][1] == pytest.approx(np.sum(g["D_r"]), rel=1e-6)


def test_full_model_cache_every_block():
    _need_gpu()
    w = synth.workload("full_model_cache")
    L = kvq.Layout(w.S, w.T, w.D, w.G)
    B = w.budgets[0] * w.entries
    xd = synth.make_torch(w, seed=0)
    buf = kvq.Buffers(L, w.s)
    kvq.quantize(xd, L, B, w.s, seed=11, index_base=0, buf=buf)
    torch.cuda.synchronize()
    g = _host(buf)
    assert g["status"] == 0 and int(buf.status_stats.item()) == 0
    assert g["totals"][0] <= B
    x_np = gc.to_np(xd)
    del xd
    oracle.set_threads(0)
    ob = oracle.allocate_bisect(x_np, w.G, w.s, B)
    assert ob["status"] == 0
    _check_lambda(g["lambda"], ob["lambda"])
    del ob
    _, nontie = gc.check_choice(g, x_np, w.G, w.s, g["lambda"])
    assert nontie.mean() > 0.9
    _check_totals(g, 32 * w.G)
    _check_codes(x_np, w.G, buf.codes, g, 11, 0, np.random.default_rng(3))


def test_hadamard_groups_budget_sweep_on_one_stats():
    _need_gpu()
    w = synth.workload("hadamard_groups")
    L = kvq.Layout(w.S, w.T, w.D, w.G)
    xd = synth.make_torch(w, seed=0)
    buf = kvq.Buffers(L, w.s)
    kvq.kvq_stats(xd, L, buf.stats, buf.status_stats)          # once for every budget
    x_np = gc.to_np(xd)
    oracle.set_threads(0)
    lams = []
    for bi, bpe in enumerate(w.budgets):
        B = bpe * w.entries
        kvq.kvq_allocate(buf.stats, L, w.s, B, kvq.KVQ_BISECT40, 0.0, buf.lam, buf.workspace,
                         buf.codebook, buf.k, buf.D_r, buf.H_r, buf.totals, buf.status)
        kvq.kvq_quantize(xd, L, buf.codebook, buf.k, 20 + bi, 0, buf.codes, buf.status_quant)
        torch.cuda.synchronize()
        g = _host(buf)
        assert g["status"] == 0 and int(buf.status_quant.item()) == 0
        assert g["totals"][0] <= B
        ob = oracle.allocate_bisect(x_np, w.G, w.s, B)
        _check_lambda(g["lambda"], ob["lambda"])
        _, nontie = gc.check_choice(g, x_np, w.G, w.s, g["lambda"])
        assert nontie.mean() > 0.9
        _check_totals(g, 32 * w.G)
        _check_codes(x_np, w.G, buf.codes, g, 20 + bi, 0, np.random.default_rng(bi))
        lams.append(g["lambda"])
    # more bits, smaller lambda
    assert all(a > b for a, b in zip(lams, lams[1:])), lams


def test_decode_admission_subgradient_steps():
    _need_gpu()
    w = synth.workload("decode_admission")
    L = kvq.Layout(w.S, w.T, w.D, w.G)
    B = w.budgets[0] * w.entries
    oracle.set_threads(0)
    buf = kvq.Buffers(L, w.s)
    lam = None
    for t in range(9):
        xd = synth.make_torch(w, seed=1000 + t)
        if t == 0:
            kvq.quantize(xd, L, B, w.s, seed=t, index_base=0, buf=buf)
        else:
            buf.lam.fill_(lam)
            kvq.quantize(xd, L, B, w.s, seed=t, index_base=0, mode=kvq.KVQ_SUBGRADIENT,
                         eta=w.eta, buf=buf)
        torch.cuda.synchronize()
        g = _host(buf)
        assert g["status"] == 0
        x_np = gc.to_np(xd)
        if t == 0:
            ob = oracle.allocate_bisect(x_np, w.G, w.s, B)
            _check_lambda(g["lambda"], ob["lambda"])
            lam_choice = g["lambda"]
        else:
            assert g["totals"][2] == lam                  # chosen at lambda_t
            lam_choice = lam
        at, nontie = gc.check_choice(g, x_np, w.G, w.s, lam_choice)
        assert nontie.mean() > 0.9
        _check_totals(g, 32 * w.G)
        if t > 0:
            R = g["totals"][0]
            assert R == pytest.approx(at["totals"][0], rel=1e-3)
            o = oracle.allocate_at(x_np, w.G, w.s, lam, w.eta, B)
            assert g["lambda"] == pytest.approx(o["lambda_next"], rel=gc.LAM_REL,
                                                abs=w.eta * 1e-4 * B)
        _check_codes(x_np, w.G, buf.codes, g, t, 0, np.random.default_rng(100 + t))
        lam = g["lambda"]
