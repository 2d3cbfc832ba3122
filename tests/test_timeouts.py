"""The error paths of the kernels' bounded waits, run without a fault or a
hang: with KVQ_TEST_WAIT_LIMIT_NS set, the search kernel's grid hand-over
waits give up after a nanosecond and the quantize and attention kernels' waits
for their bulk copies without polling.  Each call must return (no hang), report
KVQ_ERR_TIMEOUT in its device status, and leave the buffers usable: the next
call without the limit, on the same buffers, gives exactly the results of a
call on fresh buffers.  The copies still in flight when a kernel leaves are
waited for with the normal limit, so no copy lands in released shared
memory."""
import math

import numpy as np
import pytest
import torch

from rate_adaptive_kv_block_b300 import kvq, synth

pytestmark = pytest.mark.gpu

ENV = "KVQ_TEST_WAIT_LIMIT_NS"


def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _same(a, b, keys):
    for key in keys:
        x, y = getattr(a, key), getattr(b, key)
        assert torch.equal(x.view(torch.uint8), y.view(torch.uint8)), key


@pytest.mark.parametrize("fused", [False, True])
def test_allocate_and_quantize_time_out_then_recover(monkeypatch, fused):
    _need_gpu()
    w = synth.workload("llama3_8b_layer", T=2048)
    x = synth.make_torch(w, seed=61)
    L = kvq.Layout(w.S, w.T, w.D, w.G)
    B = w.budgets[0] * w.entries
    buf = kvq.Buffers(L, w.s)
    buf.status_quant.zero_()
    monkeypatch.setenv(ENV, "1")
    kvq.quantize(x, L, B, w.s, seed=3, buf=buf, fused=fused)
    torch.cuda.synchronize()                          # returned: no hang
    assert int(buf.status.item()) == kvq.KVQ_ERR_TIMEOUT
    if not fused:
        assert int(buf.status_quant.item()) == kvq.KVQ_ERR_TIMEOUT
    monkeypatch.delenv(ENV)
    buf.status_quant.zero_()
    kvq.quantize(x, L, B, w.s, seed=3, buf=buf, fused=fused)
    ref = kvq.Buffers(L, w.s)
    ref.status_quant.zero_()
    kvq.quantize(x, L, B, w.s, seed=3, buf=ref, fused=fused)
    torch.cuda.synchronize()
    assert int(buf.status.item()) == 0 and int(buf.status_quant.item()) == 0
    _same(buf, ref, ("codebook", "k", "D_r", "H_r", "totals", "lam", "status", "codes"))


def test_decode_attention_times_out_then_recovers(monkeypatch):
    _need_gpu()
    w = synth.workload("llama3_8b_layer", T=1024)
    x = synth.make_torch(w, seed=62)
    L = kvq.Layout(w.S, w.T, w.D, w.G)
    buf = kvq.quantize(x, L, w.budgets[0] * w.entries, w.s, seed=1)
    S_kv = w.S // 2
    half = S_kv * (w.T // 32)
    Lk = kvq.Layout(S_kv, w.T, w.D, w.G)
    g = torch.Generator(device="cpu").manual_seed(3)
    q = torch.randn((S_kv * 4, w.D), generator=g).cuda()
    ws = torch.empty(kvq.kvq_attention_workspace_bytes(Lk, 4), dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")

    def call(out):
        kvq.kvq_decode_attention(q, 4, Lk, buf.codes[:half], buf.codebook[:half], buf.codes[half:],
                                 buf.codebook[half:], w.T, 1 / math.sqrt(w.D), ws, out, st)
    out = torch.empty_like(q)
    monkeypatch.setenv(ENV, "1")
    call(out)
    torch.cuda.synchronize()
    assert int(st.item()) == kvq.KVQ_ERR_TIMEOUT
    monkeypatch.delenv(ENV)
    st.zero_()
    call(out)
    ref = torch.empty_like(q)
    call(ref)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.equal(out, ref) and torch.isfinite(out).all()
