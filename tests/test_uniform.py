"""The uniform comparators ("Rate-adaptive KV-cache quantizer", "Implementation
notes": uniform INT4 and uniform stochastic quantization at equal cache
bytes): kvq_uniform_codebook + kvq_quantize_nearest (INT4) and
kvq_uniform_codebook + kvq_quantize (uniform stochastic), against the oracle.

Oracle pins: the grid runs from the block's minimum to its maximum in 15 equal
steps (up to binary16 rounding); rounding to the nearest level is within half
a step and picks the closest level (brute force); on uniform data the mean
squared error is step^2/12 for the nearest level and step^2/6 for unbiased
interpolation (closed forms); a constant block has one level and codes 0.
GPU: codebooks, k and codes byte for byte.
"""
import numpy as np
import pytest

import oracle


def _x16(a):
    return np.asarray(a, dtype=np.float16).view(np.uint16)


def _blocks(x, G):
    S, T, D = x.shape
    v = x.view(np.float16).astype(np.float64)
    return v.reshape(S, T // 32, 32, D // G, G).transpose(0, 1, 3, 2, 4).reshape(-1, 32 * G)


def test_uniform_grid_spans_min_to_max_in_equal_steps():
    rng = np.random.default_rng(1)
    x = _x16(rng.standard_normal((2, 64, 128)) * np.exp(rng.standard_normal((2, 1, 128))))
    cb, k = oracle.uniform_codebook(x, 32)
    B = _blocks(x, 32)
    assert np.all(k == 16)
    for b in range(len(k)):
        m, M = B[b].min(), B[b].max()
        assert cb[b, 0] == m and cb[b, 15] == M
        step = (M - m) / 15
        want = m + step * np.arange(16)
        # binary16 rounding of each level: half an ulp of binary16 at its size
        tol = np.maximum(np.abs(want), 2.0 ** -14) * 2.0 ** -11 + 1e-6 * abs(step)
        assert np.all(np.abs(cb[b] - want) <= tol)
        assert np.all(np.diff(cb[b]) > 0)


def test_nearest_is_the_closest_level():
    rng = np.random.default_rng(2)
    x = _x16(rng.standard_normal((1, 32, 64)))
    cb, k = oracle.uniform_codebook(x, 64)
    codes = oracle.quantize_nearest(x, 64, cb, k)
    c = np.empty((codes.shape[0], codes.shape[1] * 2), dtype=np.int64)
    c[:, 0::2], c[:, 1::2] = codes & 15, codes >> 4
    B = _blocks(x, 64)
    for b in range(len(k)):
        q = cb[b, :k[b]].astype(np.float64)
        d = np.abs(B[b][:, None] - q[None, :])
        best = d.min(axis=1)
        chosen = d[np.arange(len(B[b])), c[b]]
        assert np.all(chosen == best)                       # closest (ties: either is closest)
        assert np.all(chosen <= np.diff(q).max() / 2 + 1e-12)


def test_uniform_data_mse_closed_forms():
    # entries uniform on [0, 1] (binary16): step = 1/15; rounding to the
    # nearest level errs by step^2/12 on average, unbiased interpolation by
    # E[(q_{i+1} - x)(x - q_i)] = step^2/6
    rng = np.random.default_rng(3)
    n_tok = 32 * 64
    x = _x16(np.concatenate([[0.0, 1.0], rng.random(n_tok * 128 - 2)]).reshape(1, n_tok, 128))
    # one block per 32 tokens; put the exact ends into every block
    x = x.reshape(1, n_tok, 128).copy()
    xv = x.view(np.float16)
    xv[0, 0::32, 0] = 0.0
    xv[0, 1::32, 0] = 1.0
    cb, k = oracle.uniform_codebook(x, 128)
    step = 1.0 / 15
    codes = oracle.quantize_nearest(x, 128, cb, k)
    y = oracle.dequantize(codes, cb, x.shape, 128).view(np.float16).astype(np.float64)
    mse_near = np.mean((y - xv.astype(np.float64)) ** 2)
    assert abs(mse_near / (step ** 2 / 12) - 1) < 0.03
    codes_s = oracle.quantize(x, 128, cb, k, seed=5)
    ys = oracle.dequantize(codes_s, cb, x.shape, 128).view(np.float16).astype(np.float64)
    mse_sto = np.mean((ys - xv.astype(np.float64)) ** 2)
    assert abs(mse_sto / (step ** 2 / 6) - 1) < 0.03


def test_constant_block_has_one_level():
    x = _x16(np.full((1, 32, 32), -0.5))
    cb, k = oracle.uniform_codebook(x, 32)
    assert np.all(k == 1) and np.all(cb == -0.5)
    assert np.all(oracle.quantize_nearest(x, 32, cb, k) == 0)


@pytest.mark.gpu
@pytest.mark.parametrize("name,T,S,G", [("llama3_8b_layer", 512, 16, 128),
                                        ("hadamard_groups", 256, 8, 32),
                                        ("k_head_small", 256, 8, 8)])
def test_uniform_comparators_match_oracle(name, T, S, G):
    import torch
    from rate_adaptive_kv_block_b300 import kvq, synth
    w = synth.workload(name, T=T, S=S)
    x = synth.make_numpy(w, seed=4)
    xd = torch.from_numpy(x.view(np.int16)).view(torch.float16).cuda()
    L = kvq.Layout(w.S, w.T, w.D, G)
    nb = L.nblocks
    cb = torch.empty((nb, 16), dtype=torch.float32, device="cuda")
    k = torch.empty(nb, dtype=torch.uint8, device="cuda")
    st = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    codes = torch.empty((nb, 16 * G), dtype=torch.uint8, device="cuda")
    codes_s = torch.empty_like(codes)
    kvq.kvq_uniform_codebook(xd, L, cb, k, st)
    kvq.kvq_quantize_nearest(xd, L, cb, k, codes)
    kvq.kvq_quantize(xd, L, cb, k, 9, 0, codes_s)
    torch.cuda.synchronize()
    assert int(st.item()) == kvq.KVQ_OK
    want_cb, want_k = oracle.uniform_codebook(x, G)
    assert np.array_equal(k.cpu().numpy(), want_k)
    assert np.array_equal(cb.cpu().numpy().view(np.uint32), want_cb.view(np.uint32))
    assert np.array_equal(codes.cpu().numpy(), oracle.quantize_nearest(x, G, want_cb, want_k))
    assert np.array_equal(codes_s.cpu().numpy(), oracle.quantize(x, G, want_cb, want_k, 9))


@pytest.mark.gpu
def test_uniform_edge_blocks():
    """Constant, two-valued, signed-zero and huge blocks (the quantizer's own
    edge cases) through both comparators, byte for byte."""
    import torch
    from rate_adaptive_kv_block_b300 import kvq
    r = np.random.default_rng(5)
    blocks = [np.full((32, 128), 0.75),
              np.where(r.random((32, 128)) < 0.3, -1.0, 2.0),
              np.where(r.random((32, 128)) < 0.5, -0.0, 0.0),
              np.clip(r.standard_normal((32, 128)) * 3e4, -65504, 65504),
              r.standard_normal((32, 128)) * 1e-6]
    x = _x16(np.stack(blocks).reshape(len(blocks), 32, 128))
    xd = torch.from_numpy(x.view(np.int16)).view(torch.float16).cuda()
    L = kvq.Layout(len(blocks), 32, 128, 128)
    cb = torch.empty((len(blocks), 16), dtype=torch.float32, device="cuda")
    k = torch.empty(len(blocks), dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    codes = torch.empty((len(blocks), 2048), dtype=torch.uint8, device="cuda")
    kvq.kvq_uniform_codebook(xd, L, cb, k, st)
    kvq.kvq_quantize_nearest(xd, L, cb, k, codes)
    torch.cuda.synchronize()
    want_cb, want_k = oracle.uniform_codebook(x, 128)
    assert np.array_equal(k.cpu().numpy(), want_k)
    assert np.array_equal(cb.cpu().numpy().view(np.uint32), want_cb.view(np.uint32))
    assert np.array_equal(codes.cpu().numpy(), oracle.quantize_nearest(x, 128, want_cb, want_k))
