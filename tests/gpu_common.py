"""Helpers for the GPU parity tests: run the CUDA path through the C ABI and
compare it with the oracle under the parity rules:
  * candidates bit-exact, atom moments within 2e-5 relative;
  * lambda within 1e-4 relative;
  * at the GPU's lambda, every block whose best-vs-second objective gap (the
    oracle's) exceeds 1e-5 relative has the oracle's codebook and k, and D_r,
    H_r within 1e-4 relative (1e-6 absolute floor); the other blocks' choice
    is within 1e-5 of the optimum objective;
  * codes bit-exact (the oracle quantizes with the GPU's codebooks), decode
    exact.
"""
import numpy as np
import torch

import oracle
from rate_adaptive_kv_block_b300 import kvq

GAP = 1e-5
LAM_REL = 1e-4
DH_REL = 1e-4
MOM_REL = 2e-5


def to_dev(x_np):
    return torch.from_numpy(np.ascontiguousarray(x_np).view(np.int16)).view(torch.float16).cuda()


def to_np(x_t):
    return x_t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def run(x, G, s, budget, seed=0, index_base=0, mode=kvq.KVQ_BISECT40, eta=0.0, lam0=0.0, w=None):
    """Whole path on the GPU (kvq_stats_weighted when per-entry weights w are
    given); returns numpy copies of every output."""
    S, T, D = x.shape
    L = kvq.Layout(S, T, D, G)
    xd = x if isinstance(x, torch.Tensor) else to_dev(x)
    wd = None if w is None else torch.from_numpy(np.ascontiguousarray(w, dtype=np.float32)).to(xd.device)
    buf = kvq.Buffers(L, s, xd.device)
    buf.lam.fill_(lam0)
    kvq.quantize(xd, L, budget, s, seed=seed, index_base=index_base, mode=mode, eta=eta, buf=buf,
                 weights=wd)
    y = torch.empty_like(xd)
    kvq.kvq_dequantize(buf.codes, buf.codebook, L, y)
    torch.cuda.synchronize()
    rows = kvq.stats_rows(buf.stats).cpu().numpy()
    return {
        "L": L,
        "rows": rows,
        "cand": rows[:, :17].astype(np.float64),
        "mprime": rows[:, 17].view(np.int32).copy(),
        "flags": rows[:, 18].view(np.int32).copy(),
        "atoms": np.stack([rows[:, 20:36], rows[:, 36:52], rows[:, 52:68], rows[:, 68:84]],
                          axis=-1).astype(np.float64),
        "codebook": buf.codebook.cpu().numpy(),
        "k": buf.k.cpu().numpy(),
        "D_r": buf.D_r.cpu().numpy().astype(np.float64),
        "H_r": buf.H_r.cpu().numpy().astype(np.float64),
        "totals": buf.totals.cpu().numpy(),
        "lambda": float(buf.lam.cpu().numpy()[0]),
        "status_stats": int(buf.status_stats.cpu().numpy()[0]),
        "status": int(buf.status.cpu().numpy()[0]),
        "codes": buf.codes.cpu().numpy(),
        "y": to_np(y),
    }


def check_stats(g, ora, ids=None, weighted=False):
    """GPU stats rows (ids: which GPU blocks the oracle rows are) vs oracle;
    weighted: the moments are weighted sums, the first one too."""
    ids = np.arange(len(ora["mprime"])) if ids is None else np.asarray(ids)
    mp = ora["mprime"]
    assert np.array_equal(g["mprime"][ids], mp)
    c_g = g["cand"][ids]
    assert np.array_equal(c_g, ora["cand"]), "candidates differ"
    assert np.array_equal(g["flags"][ids] & 3, ora["nonfinite"])
    a_g, a_o = g["atoms"][ids], ora["atoms"]
    if not weighted:
        assert np.array_equal(a_g[..., 0], a_o[..., 0]), "atom counts differ"
    for q in ((0, 1, 2, 3) if weighted else (1, 2, 3)):
        err = np.abs(a_g[..., q] - a_o[..., q])
        tol = MOM_REL * np.abs(a_o[..., q]) + 1e-7 * np.abs(a_o[..., q]).max(axis=1, keepdims=True)
        bad = err > tol + 1e-30
        assert not bad.any(), "moment %d: %d blocks off, worst rel %.3g" % (
            q, bad.any(axis=1).sum(), (err / (np.abs(a_o[..., q]) + 1e-30))[bad].max())


def chain_mask_from_codebook(cand, mp, q, k):
    """Candidate-index mask of a codebook (levels are exact candidate values)."""
    m = 0
    for t in range(k):
        hit = np.nonzero(cand[:mp] == np.float64(q[t]))[0]
        assert len(hit) == 1, "codebook level is not a candidate"
        m |= 1 << int(hit[0])
    return m


def check_choice(g, x_np, G, s, lam, ids=None, slab_ids=None, w=None):
    """Codebooks / k / D_r / H_r of the GPU against the oracle's choice at the
    same lambda.  ids: oracle block ids (in x_np); slab_ids: the GPU block ids
    they correspond to; w: distortion weights.  Returns the oracle result and
    the non-tie mask."""
    at = oracle.allocate_at(x_np, G, s, lam, ids=ids, w=w)
    gi = np.arange(len(at["k"])) if slab_ids is None else np.asarray(slab_ids)
    nontie = at["gap"] > GAP
    cb_g, k_g = g["codebook"][gi], g["k"][gi]
    same = np.all(cb_g == at["codebook"], axis=1) & (k_g == at["k"])
    assert same[nontie].all(), "%d of %d non-tie blocks chose another codebook" % (
        (~same[nontie]).sum(), nontie.sum())
    d = 32 * G
    Dg, Hg = g["D_r"][gi], g["H_r"][gi]
    rel_D = np.abs(Dg - at["D_r"]) / np.maximum(np.abs(at["D_r"]), 1e-30)
    err_H = np.abs(Hg - at["H_r"])
    okD = (rel_D <= DH_REL) | (np.abs(Dg - at["D_r"]) <= 1e-6)
    okH = err_H <= np.maximum(DH_REL * np.abs(at["H_r"]), 1e-6)
    assert okD[nontie].all(), "D_r off on %d blocks (worst %.3g)" % ((~okD[nontie]).sum(), rel_D[nontie].max())
    assert okH[nontie].all(), "H_r off on %d blocks" % (~okH[nontie]).sum()
    # tie blocks: the GPU's choice is (near-)optimal too
    for i in np.nonzero(~nontie & ~same)[0]:
        b = int(i) if ids is None else int(ids[i])
        mp, cand, _, _, _ = oracle.block_tables(x_np, G, b, w=w)
        m = chain_mask_from_codebook(cand, mp, cb_g[i], int(k_g[i]))
        Dc, Rc = oracle.chain_cost(x_np, G, b, m, w=w)
        obj_g = Dc + lam * Rc
        obj_o = at["D_r"][i] + lam * at["H_r"][i] * d
        assert obj_g <= obj_o * (1 + 2 * GAP) + 1e-9
        assert int(k_g[i]) <= s
    return at, nontie


def check_codes(g, x_np, G, seed, index_base, slab_ids=None, b0=0):
    """The oracle quantizes with the GPU's codebooks: codes must be equal."""
    gi = np.arange(g["codes"].shape[0]) if slab_ids is None else np.asarray(slab_ids)
    codes_o = oracle.quantize(x_np, G, g["codebook"][gi], g["k"][gi], seed, index_base, b0, len(gi))
    assert np.array_equal(codes_o, g["codes"][gi]), "%d blocks' codes differ" % (
        np.any(codes_o != g["codes"][gi], axis=1).sum())
