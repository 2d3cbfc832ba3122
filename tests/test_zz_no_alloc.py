"""kvq_allocate_static: kvq_allocate with the library's fixed device scratch,
for callers that cannot allocate device memory at the point of the call (a
caching allocator's own hooks, a serving process whose memory pool is fully
reserved, a C caller without an allocator).

Called through the C ABI, it must give exactly what kvq_allocate gives with a
caller-provided workspace, on two calls in a row (the second one reuses the
scratch the first one left behind).  The file is collected last, so these
tests run after the rest of the suite in the same process; one more test runs
the comparison in a fresh child process where kvq_allocate_static is the first
call that runs the library's per-device set-up.  The layout-size limit is
checked on the host.
"""
import os
import subprocess
import sys

import pytest
import torch

from rate_adaptive_kv_block_b300 import kvq, synth


def _outputs(L, s, device):
    nb = L.nblocks
    return dict(
        codebook=torch.full((nb, 16), float("nan"), dtype=torch.float32, device=device),
        k=torch.full((nb,), 255, dtype=torch.uint8, device=device),
        D_r=torch.full((nb,), float("nan"), dtype=torch.float32, device=device),
        H_r=torch.full((nb,), float("nan"), dtype=torch.float32, device=device),
        totals=torch.full((3,), float("nan"), dtype=torch.float64, device=device),
        lam=torch.zeros(1, dtype=torch.float64, device=device),
        status=torch.full((1,), -1, dtype=torch.int32, device=device),
    )


def _stats(x, L):
    stats = torch.empty(kvq.kvq_stats_bytes(L), dtype=torch.uint8, device=x.device)
    st = torch.zeros(1, dtype=torch.int32, device=x.device)
    kvq.kvq_stats(x, L, stats, st)
    return stats


def _same(a, b):
    for key in ("codebook", "k", "D_r", "H_r", "totals", "lam", "status"):
        assert torch.equal(a[key].view(torch.uint8) if a[key].dtype != torch.uint8 else a[key],
                           b[key].view(torch.uint8) if b[key].dtype != torch.uint8 else b[key]), key


CASES = [
    # (workload, T, S, budget bits/entry, mode, eta, lambda_in)
    ("llama3_8b_layer", 1024, 16, 2.5, kvq.KVQ_BISECT40, 0.0, 0.0),
    ("hadamard_groups", 512, 8, 2.0, kvq.KVQ_BISECT40, 0.0, 0.0),
    ("k_head_small", 256, 8, 3.0, kvq.KVQ_SUBGRADIENT, 1e-6, 0.02),
]


@pytest.mark.gpu
def test_static_scratch_matches_workspace_twice_in_a_row():
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    for seed in (11, 12):            # two calls in a row per case, new data each
        for name, T, S, bpe, mode, eta, lam0 in CASES:
            w = synth.workload(name, T=T, S=S)
            x = synth.make_torch(w, seed=seed, device="cuda")
            L = kvq.Layout(w.S, w.T, w.D, w.G)
            stats = _stats(x, L)
            budget = bpe * w.entries
            ref = _outputs(L, w.s, dev)
            ref["lam"].fill_(lam0)
            ws = torch.empty(kvq.kvq_workspace_bytes(L, w.s), dtype=torch.uint8, device=dev)
            kvq.kvq_allocate(stats, L, w.s, budget, mode, eta, ref["lam"], ws, ref["codebook"],
                             ref["k"], ref["D_r"], ref["H_r"], ref["totals"], ref["status"])
            got = _outputs(L, w.s, dev)
            got["lam"].fill_(lam0)
            kvq.kvq_allocate_static(stats, L, w.s, budget, mode, eta, got["lam"],
                                    got["codebook"], got["k"], got["D_r"], got["H_r"],
                                    got["totals"], got["status"])
            torch.cuda.synchronize()
            assert int(got["status"].item()) == kvq.KVQ_OK
            _same(ref, got)


@pytest.mark.gpu
def test_static_scratch_back_to_back_on_one_stream():
    """Two calls queued back to back with no host wait between them: the
    second one resets and reuses the scratch after the first one is done."""
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    w = synth.workload("llama3_8b_layer", T=2048, S=16)
    L = kvq.Layout(w.S, w.T, w.D, w.G)
    xs = [synth.make_torch(w, seed=sd, device="cuda") for sd in (21, 22)]
    stats = [_stats(x, L) for x in xs]
    budgets = [2.5 * w.entries, 2.0 * w.entries]
    ws = torch.empty(kvq.kvq_workspace_bytes(L, w.s), dtype=torch.uint8, device=dev)
    refs, gots = [], []
    for st, bud in zip(stats, budgets):
        r = _outputs(L, w.s, dev)
        kvq.kvq_allocate(st, L, w.s, bud, kvq.KVQ_BISECT40, 0.0, r["lam"], ws, r["codebook"],
                         r["k"], r["D_r"], r["H_r"], r["totals"], r["status"])
        refs.append(r)
    torch.cuda.synchronize()
    for st, bud in zip(stats, budgets):
        g = _outputs(L, w.s, dev)
        kvq.kvq_allocate_static(st, L, w.s, bud, kvq.KVQ_BISECT40, 0.0, g["lam"], g["codebook"],
                                g["k"], g["D_r"], g["H_r"], g["totals"], g["status"])
        gots.append(g)
    torch.cuda.synchronize()
    for r, g in zip(refs, gots):
        _same(r, g)


_FRESH = r"""
import sys, torch
sys.path.insert(0, sys.argv[1])
from rate_adaptive_kv_block_b300 import kvq, synth
torch.cuda.set_device(0)
w = synth.workload("llama3_8b_layer", T=1024, S=16)
x = synth.make_torch(w, seed=5, device="cuda")
L = kvq.Layout(w.S, w.T, w.D, w.G)
st = torch.zeros(1, dtype=torch.int32, device="cuda")
stats = torch.empty(kvq.kvq_stats_bytes(L), dtype=torch.uint8, device="cuda")
kvq.kvq_stats(x, L, stats, st)          # runs no per-device set-up
B = 2.5 * w.entries
def outs():
    nb = L.nblocks
    return [torch.full((nb, 16), float("nan"), device="cuda"),
            torch.full((nb,), 255, dtype=torch.uint8, device="cuda"),
            torch.full((nb,), float("nan"), device="cuda"),
            torch.full((nb,), float("nan"), device="cuda"),
            torch.full((3,), float("nan"), dtype=torch.float64, device="cuda"),
            torch.zeros(1, dtype=torch.float64, device="cuda"),
            torch.full((1,), -1, dtype=torch.int32, device="cuda")]
runs = []
for _ in range(2):                      # the set-up call, then a call on the set-up device
    cb, k, D, H, tot, lam, sts = outs()
    kvq.kvq_allocate_static(stats, L, w.s, B, kvq.KVQ_BISECT40, 0.0, lam, cb, k, D, H, tot, sts)
    runs.append([cb, k, D, H, tot, lam, sts])
cb, k, D, H, tot, lam, sts = outs()
ws = torch.empty(kvq.kvq_workspace_bytes(L, w.s), dtype=torch.uint8, device="cuda")
kvq.kvq_allocate(stats, L, w.s, B, kvq.KVQ_BISECT40, 0.0, lam, ws, cb, k, D, H, tot, sts)
torch.cuda.synchronize()
ref = [cb, k, D, H, tot, lam, sts]
assert int(sts.item()) == 0
for got in runs:
    for a, b in zip(ref, got):
        assert torch.equal(a.view(torch.uint8), b.view(torch.uint8))
print("FRESH_OK")
"""


@pytest.mark.gpu
def test_static_scratch_in_a_fresh_process():
    """In a new process the first kvq_allocate_static call runs the library's
    per-device set-up (module load, address look-up); it and the next call
    match kvq_allocate."""
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-c", _FRESH, root], capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0 and "FRESH_OK" in r.stdout, r.stdout[-2000:] + r.stderr[-2000:]


def test_static_scratch_limit_rejected_on_host():
    """Layouts over the fixed scratch size fail before any CUDA call."""
    lo, hi = 1, 1 << 20                  # largest number of 8-entry-wide blocks that fits
    while lo < hi:
        m = (lo + hi + 1) // 2
        if kvq.kvq_workspace_bytes(kvq.Layout(1, 32 * m, 8, 8), 16) <= kvq.KVQ_STATIC_WORKSPACE_BYTES:
            lo = m
        else:
            hi = m - 1
    assert 29000 <= lo <= 30000          # the limit the header states
    big = kvq.Layout(1, 32 * (lo + 1), 8, 8)
    assert kvq.kvq_workspace_bytes(big, 16) > kvq.KVQ_STATIC_WORKSPACE_BYTES
    rc = kvq.lib().kvq_allocate_static(None, big.c(), 16, 1.0, kvq.KVQ_BISECT40, 0.0, None,
                                       None, None, None, None, None, None, None)
    assert rc == kvq.KVQ_ERR_TOO_LARGE
    assert "static workspace" in kvq.kvq_status_string(rc)
    with pytest.raises(kvq.KvqError):
        kvq.kvq_allocate_static(None, big, 16, 1.0, kvq.KVQ_BISECT40, 0.0, None, None, None,
                                None, None, None, None, stream=_NoStream())


class _NoStream:
    cuda_stream = 0
