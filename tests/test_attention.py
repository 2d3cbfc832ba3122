"""Decode attention read from the stored cache (kvq_decode_attention) and its
fp64 oracle (oracle.decode_attention).

The oracle is pinned by what softmax attention must give in special cases:
equal scores average the values, a single token returns its value, a token
whose score dominates by hundreds returns its value, scale 0 averages, and the
order of the token blocks does not matter.  The GPU path is compared with the
oracle on codes and codebooks from the quantizer (both block shapes, ragged
token counts, every supported query-to-KV head ratio) and on the bench
workload at full size.
"""
import math

import numpy as np
import pytest

import oracle

D = 128


def _random_cache(rng, S, T, G, levels=None):
    """Random 4-bit codes and per-block codebooks of binary16 levels."""
    nb = S * (T // 32) * (D // G)
    codes = rng.integers(0, 256, size=(nb, 16 * G), dtype=np.uint8)
    if levels is None:
        lv = np.sort(rng.standard_normal((nb, 16)), axis=1)
    else:
        lv = np.broadcast_to(np.asarray(levels, dtype=np.float64), (nb, 16))
    cb = lv.astype(np.float16).astype(np.float32)
    return codes, np.ascontiguousarray(cb)


def _values(codes, cb, S, T, G):
    y = oracle.dequantize(codes, cb, (S, T, D), G)
    return y.view(np.float16).astype(np.float64)


def test_oracle_equal_scores_average_the_values():
    rng = np.random.default_rng(1)
    S, T, G, n_rep = 2, 96, 32, 2
    kc, kcb = _random_cache(rng, S, T, G, levels=[0.75] * 16)   # every key entry 0.75
    vc, vcb = _random_cache(rng, S, T, G)
    q = rng.standard_normal((S * n_rep, D))
    for T_valid in (96, 70, 33):
        out = oracle.decode_attention(q, kc, kcb, vc, vcb, S, T, D, G, n_rep, T_valid, 0.1)
        V = _values(vc, vcb, S, T, G)
        want = np.repeat(V[:, :T_valid].mean(axis=1), n_rep, axis=0)
        np.testing.assert_allclose(out, want, rtol=1e-12, atol=1e-12)


def test_oracle_scale_zero_averages_and_one_token_returns_its_value():
    rng = np.random.default_rng(2)
    S, T, G, n_rep = 3, 64, 128, 4
    kc, kcb = _random_cache(rng, S, T, G)
    vc, vcb = _random_cache(rng, S, T, G)
    q = rng.standard_normal((S * n_rep, D))
    V = _values(vc, vcb, S, T, G)
    out = oracle.decode_attention(q, kc, kcb, vc, vcb, S, T, D, G, n_rep, T, 0.0)
    np.testing.assert_allclose(out, np.repeat(V.mean(axis=1), n_rep, axis=0), rtol=1e-12, atol=1e-12)
    out1 = oracle.decode_attention(q, kc, kcb, vc, vcb, S, T, D, G, n_rep, 1, 0.3)
    assert np.array_equal(out1, np.repeat(V[:, 0], n_rep, axis=0))
    out0 = oracle.decode_attention(q, kc, kcb, vc, vcb, S, T, D, G, n_rep, 0, 0.3)
    assert np.array_equal(out0, np.zeros((S * n_rep, D)))


def test_oracle_dominant_token_returns_its_value():
    rng = np.random.default_rng(3)
    S, T, G, n_rep = 1, 64, 32, 1
    # keys: level 0 = 0 everywhere except token 37, whose codes select level 15 = 8
    kc = np.zeros((S * (T // 32) * (D // G), 16 * G), dtype=np.uint8)
    kcb = np.zeros((kc.shape[0], 16), dtype=np.float32)
    kcb[:, 15] = 8.0
    t_star = 37
    tb, t = divmod(t_star, 32)
    for g in range(D // G):
        kc[tb * (D // G) + g, t * G // 2:(t + 1) * G // 2] = 0xFF
    vc, vcb = _random_cache(rng, S, T, G)
    q = np.ones((1, D))
    out = oracle.decode_attention(q, kc, kcb, vc, vcb, S, T, D, G, n_rep, T, 1.0)
    V = _values(vc, vcb, S, T, G)
    assert np.array_equal(out[0], V[0, t_star])        # the others weigh exp(-1024) = 0


def test_oracle_token_block_order_does_not_matter():
    rng = np.random.default_rng(4)
    S, T, G, n_rep = 2, 128, 64, 2
    kc, kcb = _random_cache(rng, S, T, G)
    vc, vcb = _random_cache(rng, S, T, G)
    q = rng.standard_normal((S * n_rep, D))
    a = oracle.decode_attention(q, kc, kcb, vc, vcb, S, T, D, G, n_rep, T, 0.2)
    # reverse the token blocks of every stream (codes and codebooks together)
    nG, ntb = D // G, T // 32
    perm = np.arange(S * ntb * nG).reshape(S, ntb, nG)[:, ::-1, :].reshape(-1)
    b = oracle.decode_attention(q, kc[perm], kcb[perm], vc[perm], vcb[perm], S, T, D, G, n_rep, T, 0.2)
    np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-12)


# ------------------------------------------------------------------ GPU


def _gpu_case(name, T, S_kv, G, seed):
    """K and V codes from the quantizer: the workload's first S_kv streams are
    K, the next S_kv are V (one tensor, one lambda, as the bench quantizes it)."""
    import torch
    from rate_adaptive_kv_block_b300 import kvq, synth
    w = synth.workload(name, T=T, S=2 * S_kv)
    w.G = G
    x = synth.make_torch(w, seed=seed, device="cuda")
    L = kvq.Layout(w.S, w.T, w.D, G)
    buf = kvq.Buffers(L, 16)
    kvq.quantize(x, L, 2.5 * w.entries, 16, buf=buf)
    torch.cuda.synchronize()
    half = S_kv * (T // 32) * (D // G)              # blocks of the K streams
    return buf, half


@pytest.mark.gpu
@pytest.mark.parametrize("name,T,S_kv,G,n_rep,T_valid", [
    ("llama3_8b_layer", 1024, 8, 128, 4, 1024),
    ("llama3_8b_layer", 1024, 8, 128, 4, 1000),     # ragged last block
    ("llama3_8b_layer", 512, 4, 128, 2, 33),
    ("llama3_8b_layer", 512, 4, 128, 1, 1),
    ("hadamard_groups", 2048, 4, 32, 4, 2048),      # feature-group blocks
    ("hadamard_groups", 1024, 2, 32, 2, 777),
    ("llama3_8b_layer", 256, 2, 128, 4, 0),         # nothing attended
])
def test_decode_attention_matches_oracle(name, T, S_kv, G, n_rep, T_valid):
    import torch
    from rate_adaptive_kv_block_b300 import kvq
    buf, half = _gpu_case(name, T, S_kv, G, seed=7)
    L = kvq.Layout(S_kv, T, D, G)
    rng = np.random.default_rng(11)
    q = torch.from_numpy(rng.standard_normal((S_kv * n_rep, D)).astype(np.float32)).cuda()
    out = torch.full((S_kv * n_rep, D), float("nan"), dtype=torch.float32, device="cuda")
    ws = torch.empty(kvq.kvq_attention_workspace_bytes(L, n_rep), dtype=torch.uint8, device="cuda")
    scale = 1.0 / math.sqrt(D)
    kc, vc = buf.codes[:half], buf.codes[half:]
    kcb, vcb = buf.codebook[:half], buf.codebook[half:]
    kvq.kvq_decode_attention(q, n_rep, L, kc, kcb, vc, vcb, T_valid, scale, ws, out)
    torch.cuda.synchronize()
    got = out.cpu().numpy().astype(np.float64)
    want = oracle.decode_attention(q.cpu().numpy(), kc.cpu().numpy(), kcb.cpu().numpy(),
                                   vc.cpu().numpy(), vcb.cpu().numpy(), S_kv, T, D, G, n_rep,
                                   T_valid, scale)
    vmax = float(np.abs(vcb.cpu().numpy()).max())
    # fp32 scores, exponentials and sums over up to T tokens: well under 1e-5 of the
    # largest value (a wrong code, level or token shows up at the scale of the values)
    assert np.all(np.isfinite(got))
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-5 * vmax)


@pytest.mark.gpu
def test_decode_attention_bench_workload_full_size():
    """The layer the bench quantizes (8 KV heads x 8192 tokens, 32 query
    heads), against the oracle."""
    import torch
    from rate_adaptive_kv_block_b300 import kvq
    buf, half = _gpu_case("llama3_8b_layer", 8192, 8, 128, seed=0)
    L = kvq.Layout(8, 8192, D, 128)
    rng = np.random.default_rng(12)
    q = torch.from_numpy(rng.standard_normal((32, D)).astype(np.float32)).cuda()
    out = torch.empty((32, D), dtype=torch.float32, device="cuda")
    ws = torch.empty(kvq.kvq_attention_workspace_bytes(L, 4), dtype=torch.uint8, device="cuda")
    kc, vc = buf.codes[:half], buf.codes[half:]
    kcb, vcb = buf.codebook[:half], buf.codebook[half:]
    kvq.kvq_decode_attention(q, 4, L, kc, kcb, vc, vcb, 8192, 1.0 / math.sqrt(D), ws, out)
    torch.cuda.synchronize()
    want = oracle.decode_attention(q.cpu().numpy(), kc.cpu().numpy(), kcb.cpu().numpy(),
                                   vc.cpu().numpy(), vcb.cpu().numpy(), 8, 8192, D, 128, 4, 8192,
                                   1.0 / math.sqrt(D))
    vmax = float(np.abs(vcb.cpu().numpy()).max())
    np.testing.assert_allclose(out.cpu().numpy().astype(np.float64), want, rtol=0, atol=1e-5 * vmax)
