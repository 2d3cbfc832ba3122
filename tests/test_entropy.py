"""Entropy coding of the symbol stream (kvq_entropy_encode / kvq_entropy_decode)
and its oracle (oracle.entropy_encode / entropy_decode): rANS with the block's
exact symbol counts.

Oracle pins: decoding gives back the symbols (skewed, uniform, one-symbol and
gap-ridden distributions); the stored bytes are within the rANS bounds of the
block's empirical entropy: d H / 8 <= payload <= d H / 8 + 6 bytes per
stream (state and renormalisation slack).  GPU: the slots (their stored
bytes) and sizes equal the oracle's byte for byte, decode inverts encode, and
a damaged slot is reported without reading outside it.
"""
import zlib

import numpy as np
import pytest

import oracle


def _pack(sym):
    sym = np.asarray(sym, dtype=np.uint8)
    return (sym[..., 0::2] | (sym[..., 1::2] << 4)).astype(np.uint8)


def _entropy_bits(sym):
    n = np.bincount(sym, minlength=16)
    p = n[n > 0] / len(sym)
    return float(-(n[n > 0] * np.log2(p)).sum())


CASES = {
    "skewed": lambda r, d: np.minimum(r.geometric(0.45, d) - 1, 15),
    "uniform16": lambda r, d: r.permutation(np.repeat(np.arange(16), d // 16)),
    "one_symbol": lambda r, d: np.full(d, 7),
    "gaps": lambda r, d: r.choice([0, 3, 15], size=d, p=[0.7, 0.2, 0.1]),
    "rare": lambda r, d: np.where(r.random(d) < 0.002, 13, 2),
}


@pytest.mark.parametrize("d", [4096, 1024, 256])
@pytest.mark.parametrize("case", sorted(CASES))
def test_oracle_round_trip_and_size_bounds(case, d):
    r = np.random.default_rng(zlib.crc32(("%s/%d" % (case, d)).encode()))
    sym = CASES[case](r, d).astype(np.int64)
    codes = _pack(sym)[None, :]
    slot = oracle.entropy_encode(codes, d)[0]
    assert np.array_equal(oracle.entropy_decode(slot, d), codes[0])
    payload = len(slot) - 96
    h = _entropy_bits(sym)
    assert h / 8 <= payload + 1e-9
    assert payload <= h / 8 + 32 * 6
    if case == "uniform16":
        assert abs(payload - d / 2) <= 32 * 6          # exactly 4 bits a symbol, plus the states


def _run_blocks(r, d, m):
    names = sorted(CASES)
    return np.stack([CASES[names[(i * 3) % len(names)]](r, d) for i in range(m)]).astype(np.int64)


@pytest.mark.parametrize("d,m,nseg", [(256, 7, 3), (1024, 5, 1), (256, 16, 16), (4096, 3, 2)])
def test_oracle_runs_round_trip_and_size_bounds(d, m, nseg):
    # runs of adjacent blocks with different distributions, a ragged last run
    r = np.random.default_rng(d * 131 + m * 7 + nseg)
    sym = _run_blocks(r, d, m)
    codes = _pack(sym)
    slots = oracle.entropy_encode_runs(codes, d, nseg)
    assert len(slots) == -(-m // nseg)
    for i, slot in enumerate(slots):
        blk = sym[i * nseg:(i + 1) * nseg]
        mb = blk.shape[0]
        assert np.array_equal(oracle.entropy_decode_runs(slot, d, mb),
                              codes[i * nseg:i * nseg + mb])
        # rANS bounds of the run: at least the blocks' empirical entropy, at
        # most that plus each stream's state and one byte of slack
        payload = len(slot) - 32 * mb - 64
        h = sum(_entropy_bits(b) for b in blk)
        assert h / 8 <= payload + 1e-9
        assert payload <= h / 8 + 32 * 6


def test_oracle_runs_share_the_state_and_cost_less():
    # one block per run: the streams are those of the per-block coder; longer
    # runs store the 32 states and lengths once per run
    r = np.random.default_rng(3)
    d, m = 1024, 12
    sym = _run_blocks(r, d, m)
    codes = _pack(sym)
    per_block = oracle.entropy_encode(codes, d)
    one = oracle.entropy_encode_runs(codes, d, 1)
    for a, b in zip(per_block, one):
        assert a[96:] == b[96:]                       # the same streams
    runs = oracle.entropy_encode_runs(codes, d, 6)
    assert sum(map(len, runs)) < sum(map(len, per_block)) - (m - 2) * 96


@pytest.mark.gpu
@pytest.mark.parametrize("name,T,S,G", [("llama3_8b_layer", 256, 16, 128),
                                        ("hadamard_groups", 256, 8, 32),
                                        ("k_head_small", 128, 4, 8)])
def test_entropy_coder_matches_oracle_and_round_trips(name, T, S, G):
    import torch
    from rate_adaptive_kv_block_b300 import kvq, synth
    w = synth.workload(name, T=T, S=S)
    x = synth.make_torch(w, seed=2, device="cuda")
    L = kvq.Layout(w.S, w.T, w.D, G)
    buf = kvq.Buffers(L, 16)
    kvq.quantize(x, L, 2.5 * w.entries, 16, buf=buf)
    nb, d = L.nblocks, 32 * G
    cap = kvq.kvq_entropy_slot_bytes(L)
    assert cap == d // 2 + 288
    out = torch.zeros((nb, cap), dtype=torch.uint8, device="cuda")
    nbytes = torch.zeros(nb, dtype=torch.int32, device="cuda")
    kvq.kvq_entropy_encode(buf.codes, L, out, nbytes)
    back = torch.empty_like(buf.codes)
    st = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    kvq.kvq_entropy_decode(out, L, back, st)
    torch.cuda.synchronize()
    assert int(st.item()) == kvq.KVQ_OK
    assert torch.equal(back, buf.codes)
    want = oracle.entropy_encode(buf.codes.cpu().numpy(), d)
    got, sizes = out.cpu().numpy(), nbytes.cpu().numpy()
    for b in range(nb):
        assert sizes[b] == len(want[b])
        assert bytes(got[b, :sizes[b]]) == want[b]


@pytest.mark.gpu
def test_entropy_coder_with_one_stream_far_above_four_bits_a_symbol():
    """Blocks whose stream 0 (entries 0, 32, 64, ..) holds only rare symbols,
    so that it needs far more than 4 bits a symbol, between ordinary blocks
    (distributions of the oracle pins): every slot equals the oracle's byte
    for byte and decodes back."""
    import torch
    from rate_adaptive_kv_block_b300 import kvq
    G, nb = 128, 37
    d = 32 * G
    e = np.arange(d)
    r = np.random.default_rng(12)
    names = sorted(CASES)
    sym = np.empty((nb, d), dtype=np.uint8)
    for b in range(nb):
        if b % 3 == 0:
            sym[b] = np.where(e % 32 == 0, 1 + (e // 32 + b) % 15, 0)
        else:
            sym[b] = CASES[names[b % len(names)]](r, d)
    codes_np = _pack(sym)
    want = oracle.entropy_encode(codes_np, d)
    len0 = want[0][32] | (want[0][33] << 8)
    assert len0 - 4 > d // 32 // 2 + 32           # well above 4 bits a symbol
    L = kvq.Layout(1, 32 * nb, G, G)
    assert L.nblocks == nb
    codes = torch.from_numpy(codes_np).cuda()
    cap = kvq.kvq_entropy_slot_bytes(L)
    out = torch.zeros((nb, cap), dtype=torch.uint8, device="cuda")
    nbytes = torch.zeros(nb, dtype=torch.int32, device="cuda")
    kvq.kvq_entropy_encode(codes, L, out, nbytes)
    back = torch.empty_like(codes)
    st = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    kvq.kvq_entropy_decode(out, L, back, st)
    torch.cuda.synchronize()
    assert int(st.item()) == kvq.KVQ_OK
    assert torch.equal(back, codes)
    got, sizes = out.cpu().numpy(), nbytes.cpu().numpy()
    for b in range(nb):
        assert sizes[b] == len(want[b])
        assert bytes(got[b, :sizes[b]]) == want[b]


@pytest.mark.gpu
def test_entropy_decode_reports_a_damaged_slot():
    import torch
    from rate_adaptive_kv_block_b300 import kvq, synth
    w = synth.workload("llama3_8b_layer", T=64, S=4)
    x = synth.make_torch(w, seed=3, device="cuda")
    L = kvq.Layout(w.S, w.T, w.D, w.G)
    buf = kvq.Buffers(L, 16)
    kvq.quantize(x, L, 2.5 * w.entries, 16, buf=buf)
    cap = kvq.kvq_entropy_slot_bytes(L)
    out = torch.zeros((L.nblocks, cap), dtype=torch.uint8, device="cuda")
    nbytes = torch.zeros(L.nblocks, dtype=torch.int32, device="cuda")
    kvq.kvq_entropy_encode(buf.codes, L, out, nbytes)
    torch.cuda.synchronize()
    back = torch.empty_like(buf.codes)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    for damage in ("counts", "lengths", "stream", "short"):
        bad = out.clone()
        if damage == "counts":
            bad[1, 0] ^= 1                      # counts no longer add up to d
        elif damage == "lengths":
            bad[2, 33] = 0xFF                   # a stream longer than the slot
        elif damage == "stream":
            bad[3, 32] = 3                      # stream 0 shorter than its state
            bad[3, 33] = 0
        else:
            # stream 0 one byte short: it runs out just before its last symbols
            n0 = int(bad[4, 32]) | (int(bad[4, 33]) << 8)
            assert n0 > 4
            bad[4, 32] = (n0 - 1) & 0xFF
            bad[4, 33] = (n0 - 1) >> 8
        kvq.kvq_entropy_decode(bad, L, back, st)
        torch.cuda.synchronize()
        assert int(st.item()) == kvq.KVQ_ERR_CORRUPT, damage


@pytest.mark.gpu
@pytest.mark.parametrize("name,T,S,G,nseg", [("llama3_8b_layer", 256, 16, 128, 16),
                                             ("llama3_8b_layer", 96, 16, 128, 5),
                                             ("hadamard_groups", 256, 8, 32, 32),
                                             ("k_head_small", 128, 4, 8, 3)])
def test_run_coder_matches_oracle_and_round_trips(name, T, S, G, nseg):
    """Coding across adjacent blocks: the runs' slots and sizes equal the
    oracle's byte for byte (ragged last runs included), decode inverts
    encode, and the stored bytes are below the per-block coder's."""
    import torch
    from rate_adaptive_kv_block_b300 import kvq, synth
    w = synth.workload(name, T=T, S=S)
    x = synth.make_torch(w, seed=4, device="cuda")
    L = kvq.Layout(w.S, w.T, w.D, G)
    buf = kvq.Buffers(L, 16)
    kvq.quantize(x, L, 2.5 * w.entries, 16, buf=buf)
    nb, d = L.nblocks, 32 * G
    nruns = -(-nb // nseg)
    cap = kvq.kvq_entropy_run_bytes(L, nseg)
    assert cap >= nseg * (d // 2 + 32) + 64 and cap % 16 == 0
    out = torch.zeros((nruns, cap), dtype=torch.uint8, device="cuda")
    nbytes = torch.zeros(nruns, dtype=torch.int32, device="cuda")
    kvq.kvq_entropy_encode_runs(buf.codes, L, nseg, out, nbytes)
    back = torch.empty_like(buf.codes)
    st = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    kvq.kvq_entropy_decode_runs(out, L, nseg, back, st)
    torch.cuda.synchronize()
    assert int(st.item()) == kvq.KVQ_OK
    assert torch.equal(back, buf.codes)
    want = oracle.entropy_encode_runs(buf.codes.cpu().numpy(), d, nseg)
    got, sizes = out.cpu().numpy(), nbytes.cpu().numpy()
    for r in range(nruns):
        assert sizes[r] == len(want[r])
        assert bytes(got[r, :sizes[r]]) == want[r]
    per_block = sum(len(s) for s in oracle.entropy_encode(buf.codes.cpu().numpy(), d))
    if nseg > 1:
        assert int(sizes.sum()) < per_block


@pytest.mark.gpu
@pytest.mark.parametrize("G,nseg,nb", [(128, 16, 40), (64, 4, 9)])
def test_run_coder_with_one_stream_far_above_four_bits_a_symbol(G, nseg, nb):
    """In the first run, stream 0 (entries 0, 32, 64, .. of each block) holds
    only rare symbols, so it needs far more than 4 bits a symbol while the run
    as a whole stays small; the other runs are ordinary.  Both kinds of run
    equal the oracle's slots byte for byte and decode back."""
    import torch
    from rate_adaptive_kv_block_b300 import kvq
    d = 32 * G
    e = np.arange(d)
    r = np.random.default_rng(11)
    sym = np.empty((nb, d), dtype=np.uint8)
    for b in range(nb):
        if b < nseg:
            sym[b] = np.where(e % 32 == 0, 1 + (e // 32 + b) % 15, 0)
        else:
            sym[b] = CASES["skewed"](r, d)
    codes_np = _pack(sym)
    want = oracle.entropy_encode_runs(codes_np, d, nseg)
    n = d // 32
    len0 = want[0][32 * nseg] | (want[0][32 * nseg + 1] << 8)
    assert len0 - 4 > n * nseg // 2 + 79          # well above 4 bits a symbol
    L = kvq.Layout(1, 32 * nb, G, G)
    assert L.nblocks == nb
    codes = torch.from_numpy(codes_np).cuda()
    nruns = -(-nb // nseg)
    cap = kvq.kvq_entropy_run_bytes(L, nseg)
    out = torch.zeros((nruns, cap), dtype=torch.uint8, device="cuda")
    nbytes = torch.zeros(nruns, dtype=torch.int32, device="cuda")
    kvq.kvq_entropy_encode_runs(codes, L, nseg, out, nbytes)
    back = torch.empty_like(codes)
    st = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    kvq.kvq_entropy_decode_runs(out, L, nseg, back, st)
    torch.cuda.synchronize()
    assert int(st.item()) == kvq.KVQ_OK
    assert torch.equal(back, codes)
    got, sizes = out.cpu().numpy(), nbytes.cpu().numpy()
    for rr in range(nruns):
        assert sizes[rr] == len(want[rr])
        assert bytes(got[rr, :sizes[rr]]) == want[rr]


@pytest.mark.gpu
def test_run_decode_reports_a_damaged_slot():
    import torch
    from rate_adaptive_kv_block_b300 import kvq, synth
    w = synth.workload("llama3_8b_layer", T=128, S=4)
    x = synth.make_torch(w, seed=5, device="cuda")
    L = kvq.Layout(w.S, w.T, w.D, w.G)
    buf = kvq.Buffers(L, 16)
    kvq.quantize(x, L, 2.5 * w.entries, 16, buf=buf)
    nseg = 4
    nruns = -(-L.nblocks // nseg)
    cap = kvq.kvq_entropy_run_bytes(L, nseg)
    out = torch.zeros((nruns, cap), dtype=torch.uint8, device="cuda")
    nbytes = torch.zeros(nruns, dtype=torch.int32, device="cuda")
    kvq.kvq_entropy_encode_runs(buf.codes, L, nseg, out, nbytes)
    torch.cuda.synchronize()
    back = torch.empty_like(buf.codes)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    h = 32 * nseg
    for damage in ("counts", "lengths", "stream", "short"):
        bad = out.clone()
        if damage == "counts":
            bad[1, 32 * 2] ^= 1                 # block 2's counts no longer add up to d
        elif damage == "lengths":
            bad[2, h + 1] = 0xFF                # a stream longer than the slot
        elif damage == "stream":
            bad[3, h] = 3                       # stream 0 shorter than its state
            bad[3, h + 1] = 0
        else:
            # stream 0 one byte short: it runs out just before the run's end
            n0 = int(bad[0, h]) | (int(bad[0, h + 1]) << 8)
            assert n0 > 4
            bad[0, h] = (n0 - 1) & 0xFF
            bad[0, h + 1] = (n0 - 1) >> 8
        kvq.kvq_entropy_decode_runs(bad, L, nseg, back, st)
        torch.cuda.synchronize()
        assert int(st.item()) == kvq.KVQ_ERR_CORRUPT, damage
