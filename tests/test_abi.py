"""The C-ABI library loads, exports every entry point include/kvq.h declares,
and rejects bad arguments on the host before touching the GPU (no compute
call runs here)."""
import ctypes as C
import os
import re

import pytest

from rate_adaptive_kv_block_b300 import build as kbuild
from rate_adaptive_kv_block_b300 import kvq

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    src = open(os.path.join(ROOT, "include", "kvq.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(kvq_[a-z_]+)\s*\(", src)))


def test_library_builds_and_exports_every_declared_symbol():
    path = kbuild.build()
    lib = C.CDLL(path)
    names = declared_functions()
    assert {"kvq_stats", "kvq_allocate", "kvq_quantize", "kvq_dequantize"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n


def test_sizes_and_layout_validation():
    L = kvq.Layout(16, 8192, 128, 128)
    assert kvq.kvq_num_blocks(L) == 4096
    assert kvq.kvq_stats_bytes(L) == 256 + 4096 * 4800
    assert kvq.kvq_workspace_bytes(L, 16) > 4096 * 32 * 8
    assert kvq.kvq_workspace_bytes(L, 1) == 0 and kvq.kvq_workspace_bytes(L, 17) == 0
    assert kvq.kvq_num_blocks(kvq.Layout(16, 8200, 128, 128)) == -1      # T % 32
    assert kvq.kvq_num_blocks(kvq.Layout(16, 8192, 128, 48)) == -1       # group
    assert kvq.kvq_num_blocks(kvq.Layout(16, 8192, 96, 64)) == -1        # D % group
    assert kvq.kvq_num_blocks(kvq.Layout(1, 32, 8 * 33, 8)) == -1        # > 32 groups
    assert kvq.kvq_num_blocks(kvq.Layout(0, 32, 128, 32)) == 0
    assert kvq.kvq_status_string(3) == "non-finite input entry"
    assert kvq.kvq_status_string(kvq.KVQ_ERR_BAD_WEIGHT) == "negative or non-finite distortion weight"


class _Fake:
    """Stands in for a device tensor: only data_ptr() is used by the binding."""
    def __init__(self, p):
        self.p = p

    def data_ptr(self):
        return self.p


class _Stream:
    cuda_stream = 0


def test_host_validation_rejects_bad_arguments():
    L = kvq.Layout(2, 64, 128, 128)
    p, odd = _Fake(1 << 20), _Fake((1 << 20) + 8)
    s = _Stream()
    bad = kvq.KVQ_ERR_INVALID_ARG
    lib = kvq.lib()
    st = kvq._stream
    assert lib.kvq_stats(C.c_void_p(p.p), L.c(), 16, C.c_void_p(p.p), C.c_void_p(p.p), st(s)) == bad
    assert lib.kvq_stats(C.c_void_p(odd.p), L.c(), 17, C.c_void_p(p.p), C.c_void_p(p.p), st(s)) == bad
    assert lib.kvq_stats(C.c_void_p(p.p), L.c(), 17, C.c_void_p(p.p), None, st(s)) == bad
    v = C.c_void_p(p.p)
    assert lib.kvq_stats_weighted(v, None, L.c(), 17, v, v, st(s)) == bad            # no weights
    assert lib.kvq_stats_weighted(v, C.c_void_p(odd.p), L.c(), 17, v, v, st(s)) == bad
    assert lib.kvq_stats_weighted(v, v, L.c(), 16, v, v, st(s)) == bad
    assert lib.kvq_stats_weighted(v, v, kvq.Layout(2, 65, 128, 128).c(), 17, v, v, st(s)) == bad
    args = [C.c_void_p(p.p)] * 9
    for s_, B, mode, eta in [(1, 1.0, 0, 0.0), (17, 1.0, 0, 0.0), (8, -1.0, 0, 0.0),
                             (8, float("nan"), 0, 0.0), (8, 1.0, 2, 0.0), (8, 1.0, 1, -1.0)]:
        assert lib.kvq_allocate(C.c_void_p(p.p), L.c(), s_, B, mode, eta, *args, st(s)) == bad
    for base in (1, 2, 6):                                                     # base % 4 != 0
        assert lib.kvq_quantize(C.c_void_p(p.p), L.c(), C.c_void_p(p.p), C.c_void_p(p.p), 0,
                                base, C.c_void_p(p.p), None, st(s)) == bad
    assert lib.kvq_quantize(C.c_void_p(p.p), L.c(), C.c_void_p(p.p), C.c_void_p(p.p), 0,
                            (1 << 40) - 1000, C.c_void_p(p.p), None, st(s)) == bad   # 2^40 cap
    assert lib.kvq_dequantize(None, C.c_void_p(p.p), L.c(), C.c_void_p(p.p), st(s)) == bad
    with pytest.raises(kvq.KvqError):
        kvq.kvq_stats(p, L, p, p, m=16, stream=s)
    # the binding checks the weights' type and size before any call
    import torch
    for wbad in (torch.zeros((2, 64, 128), dtype=torch.float16),
                 torch.zeros((2, 64, 64), dtype=torch.float32),
                 torch.zeros((2, 128, 64), dtype=torch.float32).transpose(1, 2)):
        with pytest.raises(kvq.KvqError, match="weights"):
            kvq.kvq_stats_weighted(p, wbad, L, p, p, stream=s)


def test_decode_attention_host_validation():
    """kvq_decode_attention rejects unsupported shapes and bad arguments on
    the host; its workspace size is one partial result per KV head, split
    and query head."""
    L = kvq.Layout(8, 8192, 128, 128)
    assert kvq.kvq_attention_workspace_bytes(L, 4) == 8 * 64 * 4 * 130 * 4
    assert kvq.kvq_attention_workspace_bytes(kvq.Layout(8, 8192, 64, 64), 4) == 0   # D != 128
    assert kvq.kvq_attention_workspace_bytes(L, 3) == 0                             # n_rep
    p, odd = _Fake(1 << 20), _Fake((1 << 20) + 8)
    s = _Stream()
    bad = kvq.KVQ_ERR_INVALID_ARG
    lib = kvq.lib()
    st = kvq._stream
    v = C.c_void_p(p.p)

    def call(q=v, n_rep=4, lay=L, T_valid=8192, scale=0.088, ws=v, out=v, kc=v):
        return lib.kvq_decode_attention(q, n_rep, lay.c(), kc, v, v, v, T_valid, scale, ws, out,
                                        None, st(s))
    assert call(n_rep=3) == bad
    assert call(lay=kvq.Layout(8, 8192, 256, 128)) == bad
    assert call(T_valid=8193) == bad and call(T_valid=-1) == bad
    assert call(scale=float("nan")) == bad and call(scale=float("inf")) == bad
    assert call(q=None) == bad and call(ws=None) == bad and call(out=C.c_void_p(odd.p)) == bad
    assert call(kc=None) == bad and call(kc=C.c_void_p(odd.p)) == bad
    with pytest.raises(kvq.KvqError):
        kvq.kvq_decode_attention(p, 3, L, p, p, p, p, 8192, 0.088, p, p, stream=s)


def test_encode_host_validation():
    """kvq_encode_host checks every argument of its three calls before it
    issues anything (no GPU is touched: each case is rejected on the host)."""
    L = kvq.Layout(2, 64, 128, 128)
    lib = kvq.lib()
    bad = kvq.KVQ_ERR_INVALID_ARG
    v, odd = C.c_void_p(1 << 20), C.c_void_p((1 << 20) + 8)

    def call(x_host=v, L_=L, s=8, B=1.0, seed=0, base=0, x_dev=v, stats=v, lam=v, ws=v, cb=v,
             k=v, Dr=v, Hr=v, tot=v, codes=v, status=v):
        return lib.kvq_encode_host(x_host, L_.c(), s, B, seed, base, x_dev, stats, lam, ws, cb, k,
                                   Dr, Hr, tot, codes, status, None, None, None, None,
                                   kvq._stream(_Stream()))

    assert call(L_=kvq.Layout(2, 65, 128, 128)) == bad          # T % 32
    assert call(s=1) == bad and call(s=17) == bad
    assert call(B=-1.0) == bad and call(B=float("inf")) == bad
    assert call(base=2) == bad                                   # index_base % 4
    assert call(x_host=None) == bad and call(x_dev=None) == bad
    assert call(x_dev=odd) == bad and call(codes=odd) == bad and call(stats=odd) == bad
    assert call(status=None) == bad and call(lam=None) == bad and call(tot=None) == bad
    assert call(ws=None) == bad and call(cb=None) == bad
