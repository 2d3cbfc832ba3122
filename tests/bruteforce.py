"""Brute-force reference for tiny cases (numpy, fp64), independent of oracle/.

It restates the definitions of the "Rate-adaptive KV-cache quantizer" page
("Mathematical statement", "Key formulas") element by element: every x is
sent to its interval [q_i, q_{i+1}], contributes (q_{i+1}-x)(x-q_i) to the
distortion and its interpolation probabilities to the expected codepoint
counts; the entropy is taken from those expected frequencies; the optimum is
the minimum over every admissible level subset.
"""
import itertools

import numpy as np


def candidates(v):
    """17 order statistics at ranks floor((j(d-1)+8)/16), duplicates merged."""
    v = np.sort(np.asarray(v, dtype=np.float64))
    d = len(v)
    vals = [v[(j * (d - 1) + 8) // 16] for j in range(17)]
    out = []
    for a in vals:
        if not out or a != out[-1]:
            out.append(a)
    return np.array(out)


def chain_cost_elementwise(v, q, wt=None):
    """(D, d*H, expected counts) of levels q for values v, per element; with
    per-element weights wt the distortion is sum wt (q_hi - x)(x - q_lo) and
    the counts stay unweighted."""
    v = np.asarray(v, dtype=np.float64)
    q = np.asarray(q, dtype=np.float64)
    wt = np.ones_like(v) if wt is None else np.asarray(wt, dtype=np.float64)
    d = len(v)
    k = len(q)
    if k == 1:
        return 0.0, 0.0, np.array([float(d)])
    i = np.searchsorted(q, v, side="right") - 1
    i = np.clip(i, 0, k - 2)
    lo, hi = q[i], q[i + 1]
    w = hi - lo
    pup = (v - lo) / w
    D = float(np.sum(wt * (hi - v) * (v - lo)))
    M = np.zeros(k)
    np.add.at(M, i, 1.0 - pup)
    np.add.at(M, i + 1, pup)
    pi = M / d
    nz = pi > 0
    R = float(-np.sum(M[nz] * np.log2(pi[nz])))
    return D, R, M


def all_chains(mp, s):
    """Index lists 0 = l_0 < ... < l_{k-1} = mp-1 with 2 <= k <= s."""
    if mp == 1:
        return [(0,)]
    inner = range(1, mp - 1)
    out = []
    for r in range(0, min(s, mp) - 1):
        for sub in itertools.combinations(inner, r):
            out.append((0,) + sub + (mp - 1,))
    return out


def better(a, b):
    """(obj, chain) order: objective, then fewer levels, then lexicographic."""
    if a[0] != b[0]:
        return a[0] < b[0]
    if len(a[1]) != len(b[1]):
        return len(a[1]) < len(b[1])
    return a[1] < b[1]


def best_chain(v, s, lam, wt=None):
    """Minimum of D + lam*d*H over all admissible chains, per element.
    Returns (obj, chain, D, R, second_obj)."""
    c = candidates(v)
    best = None
    second = None
    for ch in all_chains(len(c), s):
        D, R, _ = chain_cost_elementwise(v, c[list(ch)], wt)
        cand = (D + lam * R, ch, D, R)
        if best is None or better(cand, best):
            second = best
            best = cand
        elif second is None or better(cand, second):
            second = cand
    return best[0], best[1], best[2], best[3], (second[0] if second else np.inf)


def mask_of(chain):
    m = 0
    for j in chain:
        m |= 1 << j
    return m
