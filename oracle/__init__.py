"""CPU oracle for the rate-adaptive KV-cache block quantizer.

TEST INFRASTRUCTURE ONLY: imported by tests/, by __graft_entry__.smoke() and by
the cpu_baseline / reference leg of bench.py.  The product package never
imports it, and it never imports the product package.  It wraps the plain fp64
C implementation in kvq_oracle.c (see that file for the page passages each step
follows and for the readings of the open points).

Arrays: x is a uint16 numpy array of binary16 bit patterns, shape [S, T, D].
"""
import ctypes as C
import os

import numpy as np

from . import build as _build

_lib = None


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = C.CDLL(path)
        i64, i32, u64, dbl = C.c_int64, C.c_int32, C.c_uint64, C.c_double
        vp = C.c_void_p
        L.kvqo_hash32.restype = C.c_uint32
        L.kvqo_hash32.argtypes = [u64, u64]
        L.kvqo_philox4x32.restype = None
        L.kvqo_philox4x32.argtypes = [vp, vp, C.c_int, vp]
        L.kvqo_hash_many.restype = None
        L.kvqo_hash_many.argtypes = [u64, u64, i64, vp]
        L.kvqo_set_threads.restype = C.c_int
        L.kvqo_set_threads.argtypes = [C.c_int]
        L.kvqo_f16_to_double.restype = dbl
        L.kvqo_f16_to_double.argtypes = [C.c_uint16]
        L.kvqo_double_to_f16.restype = C.c_uint16
        L.kvqo_double_to_f16.argtypes = [dbl, C.POINTER(C.c_int)]
        L.kvqo_num_blocks.restype = i64
        L.kvqo_num_blocks.argtypes = [i64, i64, C.c_int, C.c_int]
        L.kvqo_flat_index.restype = i64
        L.kvqo_flat_index.argtypes = [i64, C.c_int, C.c_int, i64, C.c_int]
        L.kvqo_stats.restype = None
        L.kvqo_stats.argtypes = [vp, vp, i64, i64, C.c_int, C.c_int, i64, i64,
                                 vp, vp, vp, vp]
        L.kvqo_allocate_bisect.restype = C.c_int
        L.kvqo_allocate_bisect.argtypes = [vp, vp, i64, i64, C.c_int, C.c_int, vp,
                                           i64, C.c_int, dbl, vp, vp, vp, vp,
                                           vp, vp, vp, vp, vp]
        L.kvqo_allocate_at.restype = C.c_int
        L.kvqo_allocate_at.argtypes = [vp, vp, i64, i64, C.c_int, C.c_int, vp, i64,
                                       C.c_int, dbl, dbl, dbl, vp, vp, vp, vp,
                                       vp, vp, vp, vp]
        L.kvqo_allocate_fixed_rate.restype = C.c_int
        L.kvqo_allocate_fixed_rate.argtypes = [vp, vp, i64, i64, C.c_int, C.c_int, vp, i64,
                                               C.c_int, dbl, vp, vp, vp, vp, vp, vp, vp, vp]
        L.kvqo_rate_at.restype = dbl
        L.kvqo_rate_at.argtypes = [vp, vp, i64, i64, C.c_int, C.c_int, vp, i64,
                                   C.c_int, dbl]
        L.kvqo_block_tables.restype = C.c_int
        L.kvqo_block_tables.argtypes = [vp, vp, i64, C.c_int, C.c_int, i64, vp, vp,
                                        vp, vp]
        L.kvqo_chain_cost.restype = None
        L.kvqo_chain_cost.argtypes = [vp, vp, i64, C.c_int, C.c_int, i64,
                                      C.c_uint32, vp, vp]
        L.kvqo_quantize.restype = None
        L.kvqo_quantize.argtypes = [vp, i64, i64, C.c_int, C.c_int, vp, vp, u64,
                                    u64, i64, i64, vp]
        L.kvqo_dequantize.restype = C.c_int
        L.kvqo_dequantize.argtypes = [vp, vp, i64, i64, C.c_int, C.c_int, i64,
                                      i64, vp]
        _lib = L
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(C.c_void_p)


def _x(x):
    x = np.ascontiguousarray(x)
    if x.dtype == np.float16:
        x = x.view(np.uint16)
    assert x.dtype == np.uint16 and x.ndim == 3, "x must be [S,T,D] binary16"
    return x


def _w(w, x):
    """Per-entry weights (float32, the shape of x) or None (unweighted)."""
    if w is None:
        return None
    w = np.ascontiguousarray(np.asarray(w, dtype=np.float32))
    assert w.shape == x.shape, "weights must have the shape of x"
    return w


def _ids(ids):
    if ids is None:
        return None
    return np.ascontiguousarray(np.asarray(ids, dtype=np.int64))


def set_threads(n: int) -> int:
    return lib().kvqo_set_threads(int(n))


def hash32(seed: int, i: int) -> int:
    return lib().kvqo_hash32(seed, i)


def philox4x32(ctr, key, rounds: int):
    """The Philox4x32 block function: 4 counter words, 2 key words -> 4 words."""
    c = np.ascontiguousarray(np.asarray(ctr, dtype=np.uint32))
    k = np.ascontiguousarray(np.asarray(key, dtype=np.uint32))
    out = np.zeros(4, dtype=np.uint32)
    lib().kvqo_philox4x32(_p(c), _p(k), int(rounds), _p(out))
    return [int(v) for v in out]


def hash_many(seed: int, i0: int, n: int) -> np.ndarray:
    out = np.empty(n, dtype=np.uint32)
    lib().kvqo_hash_many(seed, i0, n, _p(out))
    return out


def f16_to_double(h: int) -> float:
    return lib().kvqo_f16_to_double(h)


def double_to_f16(v: float):
    ok = C.c_int(0)
    h = lib().kvqo_double_to_f16(v, C.byref(ok))
    return h, bool(ok.value)


def num_blocks(S, T, D, G) -> int:
    return lib().kvqo_num_blocks(S, T, D, G)


def flat_index(T, D, G, b, e) -> int:
    return lib().kvqo_flat_index(T, D, G, b, e)


def stats(x, G, b0=0, nb=None, w=None):
    """Candidates, m', atom moments (n, s1, t1, e) and the flags (bit 0: a
    non-finite value, bit 1: an invalid weight).  With per-entry weights w the
    moments are weighted (n = sum w, s1 = sum w (x - c_p), ...)."""
    x = _x(x)
    w = _w(w, x)
    S, T, D = x.shape
    if nb is None:
        nb = num_blocks(S, T, D, G) - b0
    cand = np.zeros((nb, 17))
    mp = np.zeros(nb, dtype=np.int32)
    atoms = np.zeros((nb, 16, 4))
    bad = np.zeros(nb, dtype=np.int32)
    lib().kvqo_stats(_p(x), _p(w), S, T, D, G, b0, nb, _p(cand), _p(mp),
                     _p(atoms), _p(bad))
    return {"cand": cand, "mprime": mp, "atoms": atoms, "nonfinite": bad}


def _alloc_out(nb):
    return {
        "codebook": np.zeros((nb, 16), dtype=np.float32),
        "k": np.zeros(nb, dtype=np.uint8),
        "D_r": np.zeros(nb),
        "H_r": np.zeros(nb),
        "gap": np.zeros(nb),
        "mask": np.zeros(nb, dtype=np.uint32),
        "totals": np.zeros(3),
    }


def allocate_bisect(x, G, s, budget_bits, ids=None, w=None):
    """Global lambda by the 40-step bisection, and the per-block choice there.
    Returns a dict with lambda, bracket (lo, hi), status and per-block arrays
    (ids order).  w: per-entry distortion weights (None: unweighted)."""
    x = _x(x)
    w = _w(w, x)
    S, T, D = x.shape
    ids = _ids(ids)
    nb = num_blocks(S, T, D, G) if ids is None else len(ids)
    out = _alloc_out(nb)
    lam = np.zeros(1)
    bracket = np.zeros(2)
    st = lib().kvqo_allocate_bisect(
        _p(x), _p(w), S, T, D, G, _p(ids), nb, s, float(budget_bits), _p(lam),
        _p(bracket), _p(out["codebook"]), _p(out["k"]), _p(out["D_r"]),
        _p(out["H_r"]), _p(out["gap"]), _p(out["mask"]), _p(out["totals"]))
    out.update(status=st, **{"lambda": float(lam[0])},
               bracket=(float(bracket[0]), float(bracket[1])))
    return out


def allocate_at(x, G, s, lam, eta=0.0, budget_bits=0.0, ids=None, w=None):
    """Per-block choice at a fixed lambda; lambda_next is the subgradient
    update max(0, lambda + eta (R - budget_bits))."""
    x = _x(x)
    w = _w(w, x)
    S, T, D = x.shape
    ids = _ids(ids)
    nb = num_blocks(S, T, D, G) if ids is None else len(ids)
    out = _alloc_out(nb)
    nxt = np.zeros(1)
    st = lib().kvqo_allocate_at(
        _p(x), _p(w), S, T, D, G, _p(ids), nb, s, float(lam), float(eta),
        float(budget_bits), _p(nxt), _p(out["codebook"]), _p(out["k"]),
        _p(out["D_r"]), _p(out["H_r"]), _p(out["gap"]), _p(out["mask"]),
        _p(out["totals"]))
    out.update(status=st, lambda_next=float(nxt[0]), **{"lambda": float(lam)})
    return out


def allocate_fixed_rate(x, G, s, bits_per_entry, ids=None, w=None):
    """The fixed-rate comparator: every block gets its own lambda_r from the
    40-step bisection applied to that block alone with budget
    bits_per_entry * d_r, so each block (not only the total) meets the rate.
    Returns the per-block arrays (ids order), "lambdas" and the status."""
    x = _x(x)
    w = _w(w, x)
    S, T, D = x.shape
    ids = _ids(ids)
    nb = num_blocks(S, T, D, G) if ids is None else len(ids)
    out = _alloc_out(nb)
    lams = np.zeros(nb)
    st = lib().kvqo_allocate_fixed_rate(
        _p(x), _p(w), S, T, D, G, _p(ids), nb, s, float(bits_per_entry), _p(lams),
        _p(out["codebook"]), _p(out["k"]), _p(out["D_r"]), _p(out["H_r"]), _p(out["gap"]),
        _p(out["mask"]), _p(out["totals"]))
    out.update(status=st, lambdas=lams)
    return out


def rate_at(x, G, s, lam, ids=None, w=None) -> float:
    x = _x(x)
    w = _w(w, x)
    S, T, D = x.shape
    ids = _ids(ids)
    nb = num_blocks(S, T, D, G) if ids is None else len(ids)
    return lib().kvqo_rate_at(_p(x), _p(w), S, T, D, G, _p(ids), nb, s, float(lam))


def block_tables(x, G, b, w=None):
    """(m', cand[17], Dpq, Mup, Mdn) of block b, each table 17x17 (Dpq
    weighted when w is given)."""
    x = _x(x)
    w = _w(w, x)
    S, T, D = x.shape
    cand = np.zeros(17)
    Dpq, Mup, Mdn = (np.zeros((17, 17)) for _ in range(3))
    mp = lib().kvqo_block_tables(_p(x), _p(w), T, D, G, b, _p(cand), _p(Dpq),
                                 _p(Mup), _p(Mdn))
    return mp, cand, Dpq, Mup, Mdn


def chain_cost(x, G, b, mask, w=None):
    """(D_r, d_r H_r) of the chain `mask` (bit j = candidate j) of block b."""
    x = _x(x)
    w = _w(w, x)
    S, T, D = x.shape
    Dr = np.zeros(1)
    Rr = np.zeros(1)
    lib().kvqo_chain_cost(_p(x), _p(w), T, D, G, b, int(mask), _p(Dr), _p(Rr))
    return float(Dr[0]), float(Rr[0])


def quantize(x, G, codebook, k, seed, index_base=0, b0=0, nb=None):
    """Packed 4-bit codes [nb, d/2] of blocks [b0, b0+nb); codebook/k are
    indexed from b0."""
    x = _x(x)
    S, T, D = x.shape
    if nb is None:
        nb = num_blocks(S, T, D, G) - b0
    codebook = np.ascontiguousarray(codebook, dtype=np.float32)
    k = np.ascontiguousarray(k, dtype=np.uint8)
    codes = np.zeros((nb, 16 * G), dtype=np.uint8)
    lib().kvqo_quantize(_p(x), S, T, D, G, _p(codebook), _p(k), int(seed),
                        int(index_base), b0, nb, _p(codes))
    return codes


def dequantize(codes, codebook, shape, G, b0=0, nb=None, y=None):
    """binary16 reconstruction written into y ([S,T,D] uint16) for blocks
    [b0, b0+nb)."""
    S, T, D = shape
    if nb is None:
        nb = num_blocks(S, T, D, G) - b0
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    codebook = np.ascontiguousarray(codebook, dtype=np.float32)
    if y is None:
        y = np.zeros((S, T, D), dtype=np.uint16)
    bad = lib().kvqo_dequantize(_p(codes), _p(codebook), S, T, D, G, b0, nb,
                                _p(y))
    if bad:
        raise ValueError("codebook level not representable in binary16")
    return y


def uniform_codebook(x, G):
    """Codebooks of the uniform comparator ("Rate-adaptive KV-cache quantizer",
    "Implementation notes": uniform INT4 and uniform stochastic quantization at
    equal bytes): per block from its minimum m and maximum M (a zero of either
    sign taken as +0), delta =
    fl32(fl32(M - m) / 15), level_j = binary16(fl32(m + fl32(j delta))) for
    j < 15, level_15 = M, repeats removed, slots k..15 repeat the top.
    Returns (codebook float32 [nb, 16], k uint8 [nb])."""
    xv = _f16(_x(x)).astype(np.float32)
    S, T, D = xv.shape
    blocks = xv.reshape(S, T // 32, 32, D // G, G).transpose(0, 1, 3, 2, 4).reshape(-1, 32 * G)
    nb = blocks.shape[0]
    cb = np.zeros((nb, 16), dtype=np.float32)
    k = np.zeros(nb, dtype=np.uint8)
    for b in range(nb):
        zero = np.float32(0)
        m = np.float32(np.float32(blocks[b].min()) + zero)      # -0 -> +0
        M = np.float32(np.float32(blocks[b].max()) + zero)
        delta = np.float32(np.float32(M - m) / np.float32(15))
        lv = [np.float32(np.float16(np.float32(m + np.float32(np.float32(j) * delta)))) for j in range(15)]
        lv.append(M)
        distinct = [lv[0]] + [v for a, v in zip(lv, lv[1:]) if v != a]
        k[b] = len(distinct)
        cb[b, :len(distinct)] = distinct
        cb[b, len(distinct):] = distinct[-1]
    return cb, k


def quantize_nearest(x, G, codebook, k):
    """Codes [nb, 16 G] of rounding every entry to the nearest level: i = the
    largest index with q_i <= x (at most k-2), code = i + [w < 2 r] with
    w = fl32(q_{i+1} - q_i), r = fl32(x - q_i); k = 1: code 0.  Packed as the
    quantizer's (low nibble = even entry)."""
    xv = _f16(_x(x)).astype(np.float32)
    S, T, D = xv.shape
    blocks = xv.reshape(S, T // 32, 32, D // G, G).transpose(0, 1, 3, 2, 4).reshape(-1, 32 * G)
    nb = blocks.shape[0]
    codes = np.zeros((nb, 32 * G), dtype=np.uint8)
    cb = np.asarray(codebook, dtype=np.float32)
    for b in range(nb):
        kb = int(k[b])
        if kb <= 1:
            continue
        q = cb[b, :kb]
        v = blocks[b]
        i = np.clip(np.searchsorted(q, v, side="right") - 1, 0, kb - 2)
        w = (q[i + 1] - q[i]).astype(np.float32)
        r = (v - q[i]).astype(np.float32)
        codes[b] = (i + (w < np.float32(2) * r)).astype(np.uint8)
    return (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)


RANS_L = 1 << 23


def _unpack(codes_row):
    c = np.asarray(codes_row, dtype=np.uint8)
    out = np.empty(2 * len(c), dtype=np.int64)
    out[0::2], out[1::2] = c & 15, c >> 4
    return out


def entropy_encode(codes, d):
    """Entropy coding of every block's symbols ("Rate-adaptive KV-cache
    quantizer", "Implementation notes": arithmetic coding of the symbol
    stream): rANS (Duda 2013) with 32-bit state in [L, 256 L), L = 2^23, byte
    renormalisation, the block's exact symbol counts as the model (total d);
    32 streams, stream l = entries l, l+32, ..; each stream stored as the
    encoder's final state (4 bytes little-endian) then its renormalisation
    bytes in reverse order of emission.  Slot = 16 u16 counts, 32 u16 stream
    lengths, the streams.  Returns a list of bytes objects (one per block)."""
    lg = int(d).bit_length() - 1
    n = d // 32
    slots = []
    for row in np.asarray(codes, dtype=np.uint8):
        sym = _unpack(row)
        cnt = np.bincount(sym, minlength=16)
        cum = np.concatenate([[0], np.cumsum(cnt)])
        streams = []
        for lane in range(32):
            x, emitted = RANS_L, []
            for j in range(n - 1, -1, -1):
                c = int(sym[lane + 32 * j])
                f, bc = int(cnt[c]), int(cum[c])
                xmax = ((RANS_L >> lg) << 8) * f
                while x >= xmax:
                    emitted.append(x & 255)
                    x >>= 8
                x = ((x // f) << lg) + (x % f) + bc
            streams.append(bytes([x & 255, (x >> 8) & 255, (x >> 16) & 255, (x >> 24) & 255]
                                 + emitted[::-1]))
        head = b"".join(int(v).to_bytes(2, "little") for v in cnt)
        head += b"".join(len(st).to_bytes(2, "little") for st in streams)
        slots.append(head + b"".join(streams))
    return slots


def entropy_decode(slot, d):
    """The packed codes [d/2] of one slot written by entropy_encode."""
    lg = int(d).bit_length() - 1
    n = d // 32
    cnt = [int.from_bytes(slot[2 * t:2 * t + 2], "little") for t in range(16)]
    cum = np.concatenate([[0], np.cumsum(cnt)])
    lens = [int.from_bytes(slot[32 + 2 * l:34 + 2 * l], "little") for l in range(32)]
    sym = np.zeros(d, dtype=np.int64)
    p = 96
    for lane in range(32):
        st = slot[p:p + lens[lane]]
        p += lens[lane]
        x = int.from_bytes(st[:4], "little")
        q = 4
        for j in range(n):
            s = x & (d - 1)
            c = int(np.searchsorted(cum, s, side="right") - 1)
            x = cnt[c] * (x >> lg) + s - int(cum[c])
            while x < RANS_L:
                x = (x << 8) | st[q]
                q += 1
            sym[lane + 32 * j] = c
    return (sym[0::2] | (sym[1::2] << 4)).astype(np.uint8)


def entropy_encode_runs(codes, d, nseg):
    """Entropy coding across adjacent blocks ("Rate-adaptive KV-cache
    quantizer", "Implementation notes": arithmetic coding across adjacent
    blocks): the blocks in runs of nseg consecutive blocks (the
    last run may be shorter), each run coded as 32 interleaved rANS streams
    whose state continues from block to block; stream l holds entries l, l+32,
    .. of the run's first block, then of its second, and so on; every symbol
    is coded with its own block's exact counts (total d), the rANS of
    entropy_encode otherwise (32-bit state in [L, 256 L), L = 2^23, byte
    renormalisation, encoded last symbol first).  Run slot = the m blocks'
    16 u16 counts each, 32 u16 stream lengths, the streams (each: final state
    4 bytes little-endian, then its bytes in the order the decoder reads
    them).  Returns a list of bytes objects (one per run)."""
    lg = int(d).bit_length() - 1
    n = d // 32
    rows = np.asarray(codes, dtype=np.uint8)
    out = []
    for s0 in range(0, rows.shape[0], nseg):
        blocks = rows[s0:s0 + nseg]
        syms = [_unpack(r) for r in blocks]
        cnts = [np.bincount(sy, minlength=16) for sy in syms]
        cums = [np.concatenate([[0], np.cumsum(c)]) for c in cnts]
        streams = []
        for lane in range(32):
            x, emitted = RANS_L, []
            for bi in range(len(blocks) - 1, -1, -1):
                sym, cnt, cum = syms[bi], cnts[bi], cums[bi]
                for j in range(n - 1, -1, -1):
                    c = int(sym[lane + 32 * j])
                    f, bc = int(cnt[c]), int(cum[c])
                    xmax = ((RANS_L >> lg) << 8) * f
                    while x >= xmax:
                        emitted.append(x & 255)
                        x >>= 8
                    x = ((x // f) << lg) + (x % f) + bc
            streams.append(bytes([x & 255, (x >> 8) & 255, (x >> 16) & 255, (x >> 24) & 255]
                                 + emitted[::-1]))
        head = b"".join(int(v).to_bytes(2, "little") for cnt in cnts for v in cnt)
        head += b"".join(len(st).to_bytes(2, "little") for st in streams)
        out.append(head + b"".join(streams))
    return out


def entropy_decode_runs(slot, d, m):
    """The packed codes [m, d/2] of one run slot of m blocks written by
    entropy_encode_runs."""
    lg = int(d).bit_length() - 1
    n = d // 32
    cnts = [[int.from_bytes(slot[32 * b + 2 * t:32 * b + 2 * t + 2], "little") for t in range(16)]
            for b in range(m)]
    cums = [np.concatenate([[0], np.cumsum(c)]) for c in cnts]
    h = 32 * m
    lens = [int.from_bytes(slot[h + 2 * l:h + 2 * l + 2], "little") for l in range(32)]
    sym = np.zeros((m, d), dtype=np.int64)
    p = h + 64
    for lane in range(32):
        st = slot[p:p + lens[lane]]
        p += lens[lane]
        x = int.from_bytes(st[:4], "little")
        q = 4
        for b in range(m):
            for j in range(n):
                s = x & (d - 1)
                c = int(np.searchsorted(cums[b], s, side="right") - 1)
                x = cnts[b][c] * (x >> lg) + s - int(cums[b][c])
                while x < RANS_L:
                    x = (x << 8) | st[q]
                    q += 1
                sym[b, lane + 32 * j] = c
    return (sym[:, 0::2] | (sym[:, 1::2] << 4)).astype(np.uint8)


def decode_attention(q, k_codes, k_codebook, v_codes, v_codebook, S, T, D, G, n_rep, T_valid,
                     scale):
    """One decoding step of attention over the stored cache, in fp64 ("Rate-
    adaptive KV-cache quantizer", "Implementation notes": decode before
    attention).  The K and V tensors [S, T, D] are decoded with dequantize;
    for query head hq = h * n_rep + r (q: [S * n_rep, D]):
        s_t = scale * sum_f q[hq, f] K[h, t, f]           (t < T_valid)
        out[hq] = sum_t exp(s_t - max s) V[h, t] / sum_t exp(s_t - max s)
    Returns float64 [S * n_rep, D]; zeros when T_valid = 0."""
    K = _f16(dequantize(k_codes, k_codebook, (S, T, D), G))[:, :T_valid]
    V = _f16(dequantize(v_codes, v_codebook, (S, T, D), G))[:, :T_valid]
    q = np.asarray(q, dtype=np.float64).reshape(S, n_rep, D)
    out = np.zeros((S, n_rep, D))
    if T_valid == 0:
        return out.reshape(S * n_rep, D)
    for h in range(S):
        s = scale * (q[h] @ K[h].T)                    # [n_rep, T_valid]
        w = np.exp(s - s.max(axis=1, keepdims=True))
        out[h] = (w @ V[h]) / w.sum(axis=1, keepdims=True)
    return out.reshape(S * n_rep, D)


def _f16(y):
    """uint16 binary16 bit patterns -> float64 values."""
    return np.asarray(y, dtype=np.uint16).view(np.float16).astype(np.float64)


if os.environ.get("KVQ_ORACLE_THREADS"):
    set_threads(int(os.environ["KVQ_ORACLE_THREADS"]))
