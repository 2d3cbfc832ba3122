"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Inputs are the seeded synthetic workloads of rate_adaptive_kv_block_b300.synth
at sizes the oracle finishes in seconds (several thousand blocks, both block
shapes, s < 16 and s = 16), the bench workload at its full size, and the
multi-GB workloads at full size on sampled 32-token slabs.
"""
import numpy as np
import pytest
import torch

import oracle
import gpu_common as gc
from rate_adaptive_kv_block_b300 import kvq, synth

pytestmark = pytest.mark.gpu


def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


# ------------------------------------------------------------------ stats

EDGE_BLOCKS = {
    "constant": lambda r: np.full((32, 128), 0.75),
    "two_values": lambda r: np.where(r.random((32, 128)) < 0.3, -1.0, 2.0),
    "ties": lambda r: np.round(r.standard_normal((32, 128)) * 4) / 4,
    "signed_zero": lambda r: np.where(r.random((32, 128)) < 0.5, -0.0, 0.0) + (r.random((32, 128)) < 0.1) * r.standard_normal((32, 128)),
    "subnormal": lambda r: r.standard_normal((32, 128)) * 1e-6,
    "huge": lambda r: np.clip(r.standard_normal((32, 128)) * 3e4, -65504, 65504),
    "negative": lambda r: -np.abs(r.standard_normal((32, 128))) - 1,
    "one_outlier": lambda r: np.where(np.arange(32 * 128).reshape(32, 128) == 77, 1000.0, r.standard_normal((32, 128)) * 0.01),
}


def _edge_tensor():
    r = np.random.default_rng(5)
    blocks = [f(r) for f in EDGE_BLOCKS.values()]
    x = np.stack(blocks).astype(np.float16)          # [nb, 32, 128]: one block each
    return x.view(np.uint16)


@pytest.mark.parametrize("name,T,S", [("k_head_small", None, None),
                                      ("llama3_8b_layer", 1024, None),
                                      ("hadamard_groups", 512, None)])
def test_stats_matches_oracle(name, T, S):
    _need_gpu()
    w = synth.workload(name, T=T, S=S)
    x = synth.make_numpy(w, seed=1)
    g = gc.run(x, w.G, w.s, w.budgets[0] * x.size)
    gc.check_stats(g, oracle.stats(x, w.G))
    assert g["status_stats"] == 0


def test_stats_edge_blocks():
    _need_gpu()
    x = _edge_tensor()
    g = gc.run(x, 128, 16, 2.0 * x.size)
    ora = oracle.stats(x, 128)
    gc.check_stats(g, ora)
    assert ora["mprime"][0] == 1 and ora["mprime"][1] == 2


def _boundary_tensor(nb=96, seed=7):
    """Blocks whose entries take a few keys each, at the edges of 8-key
    chunks and of 256-key bins (low bytes 0, 1, 7, 8, .., 255), in one to five
    bins, with skewed frequencies: several ranks share a bin or a key, and
    ranks land on chunk and bin edges."""
    r = np.random.default_rng(seed)
    lows = np.array([0, 1, 7, 8, 9, 15, 16, 31, 32, 127, 128, 200, 247, 248, 254, 255])
    out = np.empty((nb, 32, 128), dtype=np.uint16)
    for b in range(nb):
        bins = r.choice(np.arange(8, 248), size=int(r.integers(1, 6)), replace=False)
        keys = (bins[:, None] * 256 + lows[None, :]).ravel()
        k = r.choice(keys, size=32 * 128, p=r.dirichlet(np.full(keys.size, 0.3)))
        bits = np.where(k & 0x8000, k & 0x7fff, ~k & 0xffff).astype(np.uint16)   # key -> binary16
        out[b] = bits.reshape(32, 128)
    return out


def test_stats_ranks_on_chunk_and_bin_edges():
    _need_gpu()
    x = _boundary_tensor()
    g = gc.run(x, 128, 16, 2.0 * x.size)
    gc.check_stats(g, oracle.stats(x, 128))
    assert g["status_stats"] == 0


# --------------------------------------------------- quantize / dequantize

@pytest.mark.parametrize("name,T,G", [("llama3_8b_layer", 512, 128), ("hadamard_groups", 256, 32)])
def test_quantize_bit_exact_with_given_codebooks(name, T, G):
    _need_gpu()
    w = synth.workload(name, T=T)
    x = synth.make_numpy(w, seed=2)
    lam = 0.03
    at = oracle.allocate_at(x, G, 16, lam)
    L = kvq.Layout(*x.shape, G)
    xd = gc.to_dev(x)
    cb = torch.from_numpy(at["codebook"]).cuda()
    kk = torch.from_numpy(at["k"]).cuda()
    codes = torch.empty((L.nblocks, 16 * G), dtype=torch.uint8, device="cuda")
    for seed, base in [(0, 0), (12345, 4), (2**63 + 7, 2**39), (99, 2**40 - 2**22)]:
        kvq.kvq_quantize(xd, L, cb, kk, seed, base, codes)
        ref = oracle.quantize(x, G, at["codebook"], at["k"], seed, base)
        assert np.array_equal(codes.cpu().numpy(), ref)
    y = torch.empty_like(xd)
    kvq.kvq_dequantize(codes, cb, L, y)
    ref_y = oracle.dequantize(codes.cpu().numpy(), at["codebook"], x.shape, G)
    assert np.array_equal(gc.to_np(y), ref_y)


def _crowded_codebooks(nb, G, rng):
    """Codebooks (and data) where every other block has several levels in
    one quarter of a binade (two or more interval thresholds sharing the
    high byte of the binary16 key), the others ordinary levels."""
    x = rng.standard_normal((nb, 32, G)).astype(np.float16)
    cb = np.zeros((nb, 16), dtype=np.float32)
    k = np.zeros(nb, dtype=np.uint8)
    for b in range(nb):
        v = np.sort(x[b].astype(np.float32).ravel())
        if b % 2 == 0:
            # levels: min, four values in [1, 1.25), max
            lv = [v[0], 1.0, 1.0625, 1.125, 1.1875, v[-1]]
            x[b, 0, :6] = np.array(lv, dtype=np.float16)
            v = np.sort(x[b].astype(np.float32).ravel())
            lv = [v[0], 1.0, 1.0625, 1.125, 1.1875, v[-1]]
        else:
            lv = list(np.unique(v[np.linspace(0, len(v) - 1, 9).round().astype(int)]))
        lv = np.array(sorted(set(np.float16(lv).astype(np.float32))), dtype=np.float32)
        k[b] = len(lv)
        cb[b, :len(lv)] = lv
        cb[b, len(lv):] = lv[-1]
    return x.view(np.uint16), cb, k


@pytest.mark.parametrize("G", [128, 32])
def test_quantize_blocks_with_crowded_levels(G):
    """Blocks whose thresholds share a bin of the interval table take the
    binary-search path inside the same launch; codes bit-exact."""
    _need_gpu()
    rng = np.random.default_rng(17)
    D = 128
    nb_s = 64 if G == 128 else 16                  # 32-token slabs
    xb, cb, k = _crowded_codebooks(nb_s * (D // G), G, rng)
    # blocks [nb, 32, G] -> [S=1, T=32*nb_s, D]
    x = xb.view(np.float16).reshape(nb_s, D // G, 32, G).transpose(0, 2, 1, 3).reshape(1, 32 * nb_s, D)
    x = np.ascontiguousarray(x).view(np.uint16)
    L = kvq.Layout(1, 32 * nb_s, D, G)
    xd = gc.to_dev(x)
    codes = torch.empty((L.nblocks, 16 * G), dtype=torch.uint8, device="cuda")
    cbd, kd = torch.from_numpy(cb).cuda(), torch.from_numpy(k).cuda()
    for seed in (1, 2):
        kvq.kvq_quantize(xd, L, cbd, kd, seed, 8, codes)
        want = oracle.quantize(x, G, cb, k, seed, 8)
        assert np.array_equal(codes.cpu().numpy(), want)


def test_quantize_edge_blocks_with_oracle_codebooks():
    _need_gpu()
    x = _edge_tensor()                       # [8 blocks, 32, 128], one block per stream
    at = oracle.allocate_at(x, 128, 16, 0.05)
    L = kvq.Layout(x.shape[0], 32, 128, 128)
    xd = gc.to_dev(x)
    codes = torch.empty((L.nblocks, 16 * 128), dtype=torch.uint8, device="cuda")
    kvq.kvq_quantize(xd, L, torch.from_numpy(at["codebook"]).cuda(),
                     torch.from_numpy(at["k"]).cuda(), 5, 0, codes)
    assert np.array_equal(codes.cpu().numpy(), oracle.quantize(x, 128, at["codebook"], at["k"], 5, 0))


# ------------------------------------------------------------ allocation

ALLOC_CASES = [
    # name, T override, S override, s, budget index
    ("k_head_small", None, None, 8, 0),          # s < 16: general DP path
    ("llama3_8b_layer", None, None, 16, 0),      # the benchmark workload, full size
    ("full_model_cache", 2048, 32, 16, 0),
    ("decode_admission", None, 2048, 16, 0),
    ("hadamard_groups", 1024, None, 16, 0),
    ("hadamard_groups", 1024, None, 16, 1),
    ("hadamard_groups", 1024, None, 16, 2),
    ("hadamard_groups", 1024, None, 16, 3),
]


@pytest.mark.parametrize("name,T,S,s,bi", ALLOC_CASES)
def test_allocate_and_quantize_match_oracle(name, T, S, s, bi):
    _need_gpu()
    w = synth.workload(name, T=T, S=S)
    x = synth.make_numpy(w, seed=0)
    B = w.budgets[bi] * x.size
    g = gc.run(x, w.G, s, B, seed=7, index_base=1 << 20)
    assert g["status"] == 0 and g["status_stats"] == 0
    ob = oracle.allocate_bisect(x, w.G, s, B)
    lam_o, lam_g = ob["lambda"], g["lambda"]
    assert abs(lam_g - lam_o) <= gc.LAM_REL * abs(lam_o), (lam_g, lam_o)
    assert g["totals"][2] == lam_g
    assert g["totals"][0] <= B
    at, nontie = gc.check_choice(g, x, w.G, s, lam_g)
    assert nontie.mean() > 0.9
    # totals are the sums of the per-block values (checked block by block above;
    # tie blocks may legitimately hold another chain, so no total-vs-oracle check)
    d = 32 * w.G
    assert g["totals"][0] == pytest.approx(np.sum(g["H_r"] * d), rel=1e-6)
    assert g["totals"][1] == pytest.approx(np.sum(g["D_r"]), rel=1e-6)
    gc.check_codes(g, x, w.G, 7, 1 << 20)
    assert np.array_equal(g["y"], oracle.dequantize(g["codes"], g["codebook"], x.shape, w.G))


def test_budget_large_gives_lambda_zero_and_s_levels():
    _need_gpu()
    w = synth.workload("k_head_small", T=64)
    x = synth.make_numpy(w, seed=3)
    g = gc.run(x, w.G, 6, 16.0 * x.size)
    assert g["lambda"] == 0.0 and g["status"] == 0
    assert np.all(g["k"] == 6)
    gc.check_choice(g, x, w.G, 6, 0.0)


def test_infeasible_and_nonfinite_status():
    _need_gpu()
    w = synth.workload("k_head_small", T=64)
    x = synth.make_numpy(w, seed=4)
    g = gc.run(x, w.G, 8, 0.0)
    assert g["status"] == kvq.KVQ_ERR_INFEASIBLE
    ob = oracle.allocate_bisect(x, w.G, 8, 0.0)
    assert ob["status"] == 4 and g["lambda"] == pytest.approx(ob["lambda"], rel=1e-12)
    xb = x.copy()
    xb[1, 40, 3] = 0x7C00                  # +inf
    g = gc.run(xb, w.G, 8, 3.0 * x.size)
    assert g["status_stats"] == kvq.KVQ_ERR_NONFINITE
    assert g["status"] == kvq.KVQ_ERR_NONFINITE


def test_empty_layout():
    _need_gpu()
    L = kvq.Layout(0, 64, 128, 128)
    buf = kvq.Buffers(L, 16)
    x = torch.empty((0, 64, 128), dtype=torch.float16, device="cuda")
    buf.status.fill_(9)
    kvq.quantize(x, L, 100.0, 16, buf=buf)
    torch.cuda.synchronize()
    assert int(buf.status.item()) == 0 and float(buf.totals[0].item()) == 0.0


# ---------------------------------------------- decode-time subgradient lambda

def test_subgradient_steps_match_one_step_map():
    _need_gpu()
    w = synth.workload("decode_admission", S=1024)
    B = w.budgets[0] * w.entries
    x0 = synth.make_numpy(w, seed=100)
    g = gc.run(x0, w.G, 16, B)                          # step 0: bisection warm start
    lam = g["lambda"]
    for t in range(1, 4):
        x = synth.make_numpy(w, seed=100 + t)
        g = gc.run(x, w.G, 16, B, seed=t, mode=kvq.KVQ_SUBGRADIENT, eta=w.eta, lam0=lam)
        assert g["status"] == 0
        assert g["totals"][2] == lam                      # chosen at lambda_t
        at, nontie = gc.check_choice(g, x, w.G, 16, lam)
        R = g["totals"][0]
        assert R == pytest.approx(np.sum(g["H_r"] * 32 * w.G), rel=1e-6)
        assert R == pytest.approx(at["totals"][0], rel=1e-3)
        # lambda_{t+1} from the GPU's own R (the device may fuse the multiply-add)
        assert g["lambda"] == pytest.approx(max(0.0, lam + w.eta * (R - B)), rel=1e-12, abs=1e-300)
        o = oracle.allocate_at(x, w.G, 16, lam, w.eta, B)
        assert g["lambda"] == pytest.approx(o["lambda_next"], rel=1e-4, abs=w.eta * 1e-4 * B)
        gc.check_codes(g, x, w.G, t, 0)
        lam = g["lambda"]


# ------------------------------------------------ full sizes, sampled slabs

FULL = [("full_model_cache", 0), ("decode_admission", 0), ("hadamard_groups", 0),
        ("hadamard_groups", 3)]


@pytest.mark.parametrize("name,bi", FULL)
def test_full_size_sampled_slabs(name, bi):
    _need_gpu()
    w = synth.workload(name)
    xd = synth.make_torch(w, seed=0)
    B = w.budgets[bi] * w.entries
    g_buf = kvq.Buffers(kvq.Layout(w.S, w.T, w.D, w.G), w.s)
    L = g_buf.L
    kvq.quantize(xd, L, B, w.s, seed=11, index_base=0, buf=g_buf)
    torch.cuda.synchronize()
    assert int(g_buf.status.item()) == 0
    tot = g_buf.totals.cpu().numpy()
    assert tot[0] <= B
    lam = float(g_buf.lam.item())
    rng = np.random.default_rng(1)
    nTB, nG = w.T // 32, w.D // w.G
    slabs = rng.choice(w.S * nTB, size=6, replace=False)
    rows = kvq.stats_rows(g_buf.stats)
    for sl in slabs:
        h, tb = divmod(int(sl), nTB)
        xs = gc.to_np(xd[h, 32 * tb:32 * tb + 32, :].unsqueeze(0))
        gid = np.arange(nG) + int(sl) * nG
        gidt = torch.from_numpy(gid).cuda()
        r = rows[gidt].cpu().numpy()
        g = {
            "cand": r[:, :17].astype(np.float64), "mprime": r[:, 17].view(np.int32).copy(),
            "flags": r[:, 18].view(np.int32).copy(),
            "atoms": np.stack([r[:, 20:36], r[:, 36:52], r[:, 52:68], r[:, 68:84]], axis=-1).astype(np.float64),
            "codebook": g_buf.codebook[gidt].cpu().numpy(), "k": g_buf.k[gidt].cpu().numpy(),
            "D_r": g_buf.D_r[gidt].cpu().numpy().astype(np.float64),
            "H_r": g_buf.H_r[gidt].cpu().numpy().astype(np.float64),
            "codes": g_buf.codes[gidt].cpu().numpy(),
        }
        gc.check_stats(g, oracle.stats(xs, w.G))
        gc.check_choice(g, xs, w.G, w.s, lam)
        gc.check_codes(g, xs, w.G, 11, (h * w.T + 32 * tb) * w.D)


# ------------------------------------------------------ CUDA graph capture

def test_graph_capture_replays_the_eager_results():
    """The three calls captured as one CUDA graph (after a first eager call on
    the device) and replayed on new data give the eager results bit for bit."""
    _need_gpu()
    w = synth.workload("llama3_8b_layer", T=1024)
    L = kvq.Layout(w.S, w.T, w.D, w.G)
    B = w.budgets[0] * w.entries
    xd = synth.make_torch(w, seed=31)
    gbuf = kvq.Buffers(L, w.s)
    kvq.quantize(xd, L, B, w.s, seed=5, buf=gbuf)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        kvq.quantize(xd, L, B, w.s, seed=5, buf=gbuf)
    for sd in (32, 33):
        xn = synth.make_torch(w, seed=sd)
        xd.copy_(xn)
        graph.replay()
        ebuf = kvq.Buffers(L, w.s)
        kvq.quantize(xn, L, B, w.s, seed=5, buf=ebuf)
        torch.cuda.synchronize()
        for key in ("codebook", "k", "D_r", "H_r", "totals", "lam", "status", "codes"):
            a, b = getattr(gbuf, key), getattr(ebuf, key)
            assert torch.equal(a.view(torch.uint8), b.view(torch.uint8)), key


# ------------------------------------------- fused allocate + quantize

FUSED_CASES = [
    # name, T, S, s, budget index, mode
    ("llama3_8b_layer", None, None, 16, 0, kvq.KVQ_BISECT40),    # the benchmark workload
    ("k_head_small", None, None, 8, 0, kvq.KVQ_BISECT40),        # s < 16: general DP path
    ("hadamard_groups", 1024, None, 16, 1, kvq.KVQ_BISECT40),    # 32-feature groups
    ("full_model_cache", 2048, 32, 16, 0, kvq.KVQ_BISECT40),
    ("decode_admission", None, 1024, 16, 0, kvq.KVQ_SUBGRADIENT),
]


@pytest.mark.parametrize("name,T,S,s,bi,mode", FUSED_CASES)
def test_fused_allocate_quantize_equals_separate_calls(name, T, S, s, bi, mode):
    """kvq_allocate_quantize gives exactly kvq_allocate + kvq_quantize."""
    _need_gpu()
    w = synth.workload(name, T=T, S=S)
    xd = synth.make_torch(w, seed=41)
    L = kvq.Layout(w.S, w.T, w.D, w.G)
    B = w.budgets[bi] * w.entries
    lam0 = 0.05 if mode == kvq.KVQ_SUBGRADIENT else 0.0
    eta = 1e-6 if mode == kvq.KVQ_SUBGRADIENT else 0.0
    ref, got = kvq.Buffers(L, s), kvq.Buffers(L, s)
    for b in (ref, got):
        b.lam.fill_(lam0)
        b.codes.fill_(0xAB)
    kvq.quantize(xd, L, B, s, seed=9, index_base=4 * 77, mode=mode, eta=eta, buf=ref)
    kvq.quantize(xd, L, B, s, seed=9, index_base=4 * 77, mode=mode, eta=eta, buf=got, fused=True)
    torch.cuda.synchronize()
    assert int(got.status.item()) == 0
    for key in ("codebook", "k", "D_r", "H_r", "totals", "lam", "status", "codes"):
        a, b = getattr(ref, key), getattr(got, key)
        assert torch.equal(a.view(torch.uint8), b.view(torch.uint8)), key


def test_fused_edge_layouts():
    """Empty layout, lambda = 0 (large budget) and a layout of a few blocks."""
    _need_gpu()
    for S, T, D, G, bpe in [(0, 64, 128, 128, 2.0), (2, 64, 128, 128, 20.0), (1, 32, 64, 8, 1.0),
                           (3, 96, 256, 16, 2.5)]:
        L = kvq.Layout(S, T, D, G)
        x = torch.randn((S, T, D), device="cuda").to(torch.float16)
        ref, got = kvq.Buffers(L, 16), kvq.Buffers(L, 16)
        B = bpe * S * T * D
        kvq.quantize(x, L, B, 16, seed=3, buf=ref)
        kvq.quantize(x, L, B, 16, seed=3, buf=got, fused=True)
        torch.cuda.synchronize()
        for key in ("codebook", "k", "D_r", "H_r", "totals", "lam", "status", "codes"):
            a, b = getattr(ref, key), getattr(got, key)
            assert torch.equal(a.view(torch.uint8), b.view(torch.uint8)), (S, T, D, G, key)


# ---------------------------------------------------------- search rounds

ROUND_CASES = [
    # (workload, T, S, bits/entry): budgets whose pilot estimate is off by
    # 30-45 %, where a fine grid of fixed width around it missed lambda
    ("llama3_8b_layer", 2048, 16, 2.0),
    ("full_model_cache", 2048, 16, 2.0),
    ("decode_admission", 32, 2048, 1.5),
    ("hadamard_groups", 4096, 8, 2.0),
]


@pytest.mark.parametrize("name,T,S,bpe", ROUND_CASES)
def test_search_needs_one_round_over_every_block(name, T, S, bpe):
    """Round 0's grid spans the pilot's whole bracket, so after it only the
    blocks whose rate can still change are evaluated again; lambda is still
    the sequential bisection's (the oracle's within the parity tolerance)."""
    _need_gpu()
    w = synth.workload(name, T=T, S=S)
    x = synth.make_numpy(w, seed=0)
    xd = torch.from_numpy(x.view(np.int16)).view(torch.float16).cuda()
    L = kvq.Layout(w.S, w.T, w.D, w.G)
    nb = L.nblocks
    assert nb >= 1024                      # large enough for a pilot round
    buf = kvq.Buffers(L, 16)
    kvq.quantize(xd, L, bpe * w.entries, 16, buf=buf)
    torch.cuda.synchronize()
    rep = kvq.kvq_allocate_report(buf.workspace)
    active = rep["active"]
    assert active[0] < nb                  # the pilot: a sample
    assert active[1] == nb                 # round 0: every block
    assert all(a < nb // 2 for a in active[2:]), active
    want = oracle.allocate_bisect(x.view(np.float16), w.G, 16, bpe * w.entries)["lambda"]
    assert abs(float(buf.lam.item()) - want) <= 1e-4 * want


# ------------------------------------------- the write path from host memory

@pytest.mark.parametrize("name,T,S", [("k_head_small", 64, None), ("hadamard_groups", 256, None),
                                      ("llama3_8b_layer", 512, None)])
def test_encode_host_matches_oracle_and_device_calls(name, T, S):
    """kvq_encode_host (host input copied in pieces on several streams, host
    outputs) gives the oracle's lambda and codes, and the device-resident
    calls' results byte for byte."""
    _need_gpu()
    w = synth.workload(name, T=T, S=S)
    x = synth.make_numpy(w, seed=12)
    L = kvq.Layout(*x.shape, w.G)
    B = w.budgets[0] * x.size
    xh = torch.from_numpy(x.view(np.int16)).view(torch.float16).pin_memory()
    xd = torch.empty(x.shape, dtype=torch.float16, device="cuda")
    buf = kvq.Buffers(L, w.s)
    status = torch.full((3,), 9, dtype=torch.int32, device="cuda")
    out = dict(codes=torch.empty(buf.codes.shape, dtype=torch.uint8).pin_memory(),
               codebook=torch.empty(buf.codebook.shape, dtype=torch.float32).pin_memory(),
               k=torch.empty(buf.k.shape, dtype=torch.uint8).pin_memory(),
               totals=torch.empty(3, dtype=torch.float64).pin_memory())
    side = torch.cuda.Stream()
    kvq.kvq_encode_host(xh, L, w.s, B, 7, 1 << 20, xd, buf, status, out["codes"], out["codebook"],
                        out["k"], out["totals"], stream=side)
    side.synchronize()
    assert status.tolist() == [0, 0, 0]
    assert torch.equal(xd.view(torch.int16).cpu(), xh.view(torch.int16))      # the copy in
    ref = kvq.quantize(gc.to_dev(x), L, B, w.s, seed=7, index_base=1 << 20)
    torch.cuda.synchronize()
    for key in ("codes", "codebook", "k", "totals"):
        assert torch.equal(out[key].view(torch.uint8), getattr(ref, key).cpu().view(torch.uint8)), key
    lam = float(out["totals"][2])
    ob = oracle.allocate_bisect(x, w.G, w.s, B)
    assert abs(lam - ob["lambda"]) <= gc.LAM_REL * abs(ob["lambda"]), (lam, ob["lambda"])
    codes_o = oracle.quantize(x, w.G, out["codebook"].numpy(), out["k"].numpy(), 7, 1 << 20)
    assert np.array_equal(codes_o, out["codes"].numpy())


def test_encode_host_empty_layout_and_skipped_outputs():
    _need_gpu()
    L = kvq.Layout(0, 64, 128, 128)
    buf = kvq.Buffers(L, 16)
    status = torch.full((3,), 9, dtype=torch.int32, device="cuda")
    xh = torch.empty((0, 64, 128), dtype=torch.float16).pin_memory()
    xd = torch.empty((0, 64, 128), dtype=torch.float16, device="cuda")
    kvq.kvq_encode_host(xh, L, 16, 100.0, 0, 0, xd, buf, status)
    torch.cuda.synchronize()
    assert status.tolist() == [0, 0, 0] and float(buf.totals[0].item()) == 0.0


def test_encode_host_in_a_cuda_graph():
    """kvq_encode_host captured in a CUDA graph (its copy streams join the
    capture through events) and replayed on new host data gives the eager
    call's outputs byte for byte."""
    _need_gpu()
    w = synth.workload("llama3_8b_layer", T=512)
    L = kvq.Layout(w.S, w.T, w.D, w.G)
    B = w.budgets[0] * w.entries
    x0 = synth.make_numpy(w, seed=21)
    xh = torch.from_numpy(x0.view(np.int16)).view(torch.float16).pin_memory()
    xd = torch.empty(x0.shape, dtype=torch.float16, device="cuda")
    buf = kvq.Buffers(L, w.s)
    status = torch.zeros(3, dtype=torch.int32, device="cuda")
    outs = dict(codes=torch.empty(buf.codes.shape, dtype=torch.uint8).pin_memory(),
                codebook=torch.empty(buf.codebook.shape, dtype=torch.float32).pin_memory(),
                k=torch.empty(buf.k.shape, dtype=torch.uint8).pin_memory(),
                totals=torch.empty(3, dtype=torch.float64).pin_memory())

    def call(stream=None):
        kvq.kvq_encode_host(xh, L, w.s, B, 9, 0, xd, buf, status, outs["codes"], outs["codebook"],
                            outs["k"], outs["totals"], stream=stream)
    call()                                   # first call outside the capture (set-up)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        call()
    for sd in (22, 23):
        xn = synth.make_numpy(w, seed=sd)
        xh.copy_(torch.from_numpy(xn.view(np.int16)).view(torch.float16))
        graph.replay()
        torch.cuda.synchronize()
        got = {k: v.clone() for k, v in outs.items()}
        ref = kvq.quantize(gc.to_dev(xn), L, B, w.s, seed=9)
        torch.cuda.synchronize()
        assert status.tolist() == [0, 0, 0]
        for key in ("codes", "codebook", "k", "totals"):
            assert torch.equal(got[key].view(torch.uint8), getattr(ref, key).cpu().view(torch.uint8)), key
