"""Python binding of libkvq (include/kvq.h): argument marshalling only.

Every function has the name of the C entry point it calls and takes torch
tensors that live on the current CUDA device; it passes their data pointers,
the layout and torch's current stream, and raises on a non-OK return code.
All work happens in the CUDA kernels; there is no CPU fallback: if the
library is missing or cannot be loaded the first call raises.
"""
import ctypes as C
import os
from dataclasses import dataclass

import torch

_LIB = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libkvq.so")
_lib = None

KVQ_OK = 0
KVQ_ERR_INVALID_ARG = 1
KVQ_ERR_CUDA = 2
KVQ_ERR_NONFINITE = 3
KVQ_ERR_INFEASIBLE = 4
KVQ_ERR_TOO_LARGE = 5
KVQ_ERR_TIMEOUT = 6
KVQ_ERR_CORRUPT = 7
KVQ_ERR_BAD_WEIGHT = 8
KVQ_STATIC_WORKSPACE_BYTES = 8 << 20
KVQ_BISECT40 = 0
KVQ_SUBGRADIENT = 1
# kvq_stats output: a 256-byte header, then per block a 4800-byte record whose
# first 96 floats are the stats row (candidates, m', flags, d, atom moments)
STATS_HEADER_BYTES = 256
STATS_RECORD_FLOATS = 1200
STATS_ROW_FLOATS = 96


class _Layout(C.Structure):
    _fields_ = [("S", C.c_int64), ("T", C.c_int64), ("D", C.c_int32), ("group", C.c_int32)]


@dataclass(frozen=True)
class Layout:
    """[S, T, D] binary16 tensor cut into blocks of 32 tokens x `group`
    features."""
    S: int
    T: int
    D: int
    group: int

    def c(self):
        return _Layout(self.S, self.T, self.D, self.group)

    @property
    def d(self) -> int:
        return 32 * self.group

    @property
    def nblocks(self) -> int:
        return self.S * (self.T // 32) * (self.D // self.group)


class _Report(C.Structure):
    _fields_ = [("rounds", C.c_int32), ("steps", C.c_int32), ("active", C.c_uint32 * 16),
                ("lambda_", C.c_double), ("xa", C.c_double), ("xb", C.c_double),
                ("t_start", C.c_uint64), ("t_end", C.c_uint64), ("t_dp", C.c_uint64 * 16),
                ("t_ctl", C.c_uint64 * 16)]


class KvqError(RuntimeError):
    pass


def library_path() -> str:
    return _LIB


def lib():
    """Load libkvq.so (building it first if it is absent)."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB):
            from . import build as _b
            _b.build()
        L = C.CDLL(_LIB)
        vp, i32, i64, u64, dbl = C.c_void_p, C.c_int32, C.c_int64, C.c_uint64, C.c_double
        L.kvq_num_blocks.restype = i64
        L.kvq_num_blocks.argtypes = [_Layout]
        L.kvq_stats_bytes.restype = C.c_size_t
        L.kvq_stats_bytes.argtypes = [_Layout]
        L.kvq_workspace_bytes.restype = C.c_size_t
        L.kvq_workspace_bytes.argtypes = [_Layout, C.c_int]
        L.kvq_stats.restype = C.c_int
        L.kvq_stats.argtypes = [vp, _Layout, C.c_int, vp, vp, vp]
        L.kvq_stats_weighted.restype = C.c_int
        L.kvq_stats_weighted.argtypes = [vp, vp, _Layout, C.c_int, vp, vp, vp]
        L.kvq_allocate.restype = C.c_int
        L.kvq_allocate.argtypes = [vp, _Layout, C.c_int, dbl, C.c_int, dbl, vp, vp, vp, vp,
                                   vp, vp, vp, vp, vp]
        L.kvq_allocate_quantize.restype = C.c_int
        L.kvq_allocate_quantize.argtypes = [vp, vp, _Layout, C.c_int, dbl, C.c_int, dbl, vp, vp,
                                            vp, vp, vp, vp, vp, u64, u64, vp, vp, vp]
        L.kvq_allocate_static.restype = C.c_int
        L.kvq_allocate_static.argtypes = [vp, _Layout, C.c_int, dbl, C.c_int, dbl, vp, vp, vp,
                                          vp, vp, vp, vp, vp]
        L.kvq_allocate_fixed_rate.restype = C.c_int
        L.kvq_allocate_fixed_rate.argtypes = [vp, _Layout, C.c_int, dbl, vp, vp, vp, vp, vp, vp,
                                              vp, vp]
        L.kvq_search_state_bytes.restype = C.c_size_t
        L.kvq_search_state_bytes.argtypes = []
        L.kvq_search_begin.restype = C.c_int
        L.kvq_search_begin.argtypes = [dbl, dbl, vp]
        L.kvq_search_probes.restype = C.c_int
        L.kvq_search_probes.argtypes = [vp, vp]
        L.kvq_search_advance.restype = C.c_int
        L.kvq_search_advance.argtypes = [vp, vp, dbl]
        L.kvq_search_result.restype = C.c_int
        L.kvq_search_result.argtypes = [vp, vp, vp]
        L.kvq_stats_hi0.restype = C.c_int
        L.kvq_stats_hi0.argtypes = [vp, vp]
        L.kvq_rate_sums.restype = C.c_int
        L.kvq_rate_sums.argtypes = [vp, _Layout, C.c_int, vp, C.c_int, vp, vp]
        L.kvq_quantize.restype = C.c_int
        L.kvq_quantize.argtypes = [vp, _Layout, vp, vp, u64, u64, vp, vp, vp]
        L.kvq_dequantize.restype = C.c_int
        L.kvq_dequantize.argtypes = [vp, vp, _Layout, vp, vp]
        L.kvq_encode_host.restype = C.c_int
        L.kvq_encode_host.argtypes = [vp, _Layout, C.c_int, dbl, u64, u64, vp, vp, vp, vp, vp, vp,
                                      vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]
        L.kvq_uniform_codebook.restype = C.c_int
        L.kvq_uniform_codebook.argtypes = [vp, _Layout, vp, vp, vp, vp]
        L.kvq_quantize_nearest.restype = C.c_int
        L.kvq_quantize_nearest.argtypes = [vp, _Layout, vp, vp, vp, vp, vp]
        L.kvq_entropy_slot_bytes.restype = C.c_size_t
        L.kvq_entropy_slot_bytes.argtypes = [_Layout]
        L.kvq_entropy_encode.restype = C.c_int
        L.kvq_entropy_encode.argtypes = [vp, _Layout, vp, vp, vp]
        L.kvq_entropy_decode.restype = C.c_int
        L.kvq_entropy_decode.argtypes = [vp, _Layout, vp, vp, vp]
        L.kvq_entropy_run_bytes.restype = C.c_size_t
        L.kvq_entropy_run_bytes.argtypes = [_Layout, C.c_int]
        L.kvq_entropy_encode_runs.restype = C.c_int
        L.kvq_entropy_encode_runs.argtypes = [vp, _Layout, C.c_int, vp, vp, vp]
        L.kvq_entropy_decode_runs.restype = C.c_int
        L.kvq_entropy_decode_runs.argtypes = [vp, _Layout, C.c_int, vp, vp, vp]
        L.kvq_attention_workspace_bytes.restype = C.c_size_t
        L.kvq_attention_workspace_bytes.argtypes = [_Layout, C.c_int]
        L.kvq_decode_attention.restype = C.c_int
        L.kvq_decode_attention.argtypes = [vp, C.c_int, _Layout, vp, vp, vp, vp, i64, C.c_float,
                                           vp, vp, vp, vp]
        L.kvq_allocate_report.restype = C.c_int
        L.kvq_allocate_report.argtypes = [vp, C.POINTER(_Report)]
        L.kvq_status_string.restype = C.c_char_p
        L.kvq_status_string.argtypes = [C.c_int]
        _lib = L
    return _lib


def _ptr(t):
    return None if t is None else C.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return C.c_void_p(stream.cuda_stream)


def _check(rc: int, what: str):
    if rc != KVQ_OK:
        raise KvqError("%s: %s" % (what, kvq_status_string(rc)))


def kvq_status_string(status: int) -> str:
    return lib().kvq_status_string(int(status)).decode()


def kvq_num_blocks(L: Layout) -> int:
    return lib().kvq_num_blocks(L.c())


def kvq_stats_bytes(L: Layout) -> int:
    return lib().kvq_stats_bytes(L.c())


def kvq_workspace_bytes(L: Layout, s: int) -> int:
    return lib().kvq_workspace_bytes(L.c(), int(s))


def kvq_stats(x, L: Layout, stats, status, m: int = 17, stream=None):
    _check(lib().kvq_stats(_ptr(x), L.c(), int(m), _ptr(stats), _ptr(status), _stream(stream)),
           "kvq_stats")


def kvq_stats_weighted(x, w, L: Layout, stats, status, m: int = 17, stream=None):
    """kvq_stats with per-entry distortion weights w (float32 CUDA tensor of
    x's shape)."""
    if isinstance(w, torch.Tensor) and (w.dtype != torch.float32 or not w.is_contiguous()
                                        or w.numel() != L.S * L.T * L.D):
        raise KvqError("kvq_stats_weighted: the weights must be a contiguous float32 tensor "
                       "with one entry per element of x")
    _check(lib().kvq_stats_weighted(_ptr(x), _ptr(w), L.c(), int(m), _ptr(stats), _ptr(status),
                                    _stream(stream)), "kvq_stats_weighted")


def kvq_allocate(stats, L: Layout, s: int, budget_bits: float, mode: int, eta: float, lam,
                 workspace, codebook, k, D_r, H_r, totals, status, stream=None):
    _check(lib().kvq_allocate(_ptr(stats), L.c(), int(s), float(budget_bits), int(mode),
                              float(eta), _ptr(lam), _ptr(workspace), _ptr(codebook), _ptr(k),
                              _ptr(D_r), _ptr(H_r), _ptr(totals), _ptr(status),
                              _stream(stream)), "kvq_allocate")


def kvq_allocate_quantize(stats, x, L: Layout, s: int, budget_bits: float, mode: int, eta: float,
                          lam, workspace, codebook, k, D_r, H_r, totals, seed: int,
                          index_base: int, codes, status, stream=None):
    """kvq_allocate and kvq_quantize in one launch (same results)."""
    _check(lib().kvq_allocate_quantize(_ptr(stats), _ptr(x), L.c(), int(s), float(budget_bits),
                                       int(mode), float(eta), _ptr(lam), _ptr(workspace),
                                       _ptr(codebook), _ptr(k), _ptr(D_r), _ptr(H_r),
                                       _ptr(totals), int(seed), int(index_base), _ptr(codes),
                                       _ptr(status), _stream(stream)), "kvq_allocate_quantize")


def kvq_allocate_static(stats, L: Layout, s: int, budget_bits: float, mode: int, eta: float,
                        lam, codebook, k, D_r, H_r, totals, status, stream=None):
    """kvq_allocate with the library's fixed device scratch instead of a
    caller-provided workspace, for callers that cannot allocate device memory
    at the call.  Layouts needing more than KVQ_STATIC_WORKSPACE_BYTES of
    scratch raise KvqError (KVQ_ERR_TOO_LARGE); calls that overlap in time on
    one device share the scratch and must be serialised."""
    _check(lib().kvq_allocate_static(_ptr(stats), L.c(), int(s), float(budget_bits), int(mode),
                                     float(eta), _ptr(lam), _ptr(codebook), _ptr(k), _ptr(D_r),
                                     _ptr(H_r), _ptr(totals), _ptr(status), _stream(stream)),
           "kvq_allocate_static")


def kvq_allocate_fixed_rate(stats, L: Layout, s: int, bits_per_entry: float, codebook, k, D_r,
                            H_r, lambda_r, totals, status, stream=None):
    _check(lib().kvq_allocate_fixed_rate(_ptr(stats), L.c(), int(s), float(bits_per_entry),
                                         _ptr(codebook), _ptr(k), _ptr(D_r), _ptr(H_r),
                                         _ptr(lambda_r), _ptr(totals), _ptr(status),
                                         _stream(stream)), "kvq_allocate_fixed_rate")


class SearchState:
    """Host state of the global lambda search driven round by round
    (kvq_search_* in include/kvq.h)."""

    def __init__(self, hi0: float, budget_bits: float):
        self.buf = (C.c_char * lib().kvq_search_state_bytes())()
        self.budget = float(budget_bits)
        _check(lib().kvq_search_begin(float(hi0), self.budget, self.buf), "kvq_search_begin")

    def probes(self):
        lam = (C.c_double * 32)()
        n = lib().kvq_search_probes(self.buf, lam)
        if n < 0:
            raise KvqError("kvq_search_probes: bad argument")
        return list(lam)[:n]

    def advance(self, rate_sums):
        arr = (C.c_int64 * 32)(*[int(v) for v in list(rate_sums)[:32]] +
                               [0] * (32 - min(32, len(rate_sums))))
        _check(lib().kvq_search_advance(self.buf, arr, self.budget), "kvq_search_advance")

    def result(self):
        lam = C.c_double(0.0)
        rounds = C.c_int32(0)
        st = lib().kvq_search_result(self.buf, C.byref(lam), C.byref(rounds))
        if st == KVQ_ERR_INVALID_ARG:
            raise KvqError("kvq_search_result: the search is not done")
        return lam.value, st, rounds.value


def kvq_stats_hi0(stats) -> float:
    v = C.c_double(0.0)
    rc = lib().kvq_stats_hi0(_ptr(stats), C.byref(v))
    if rc not in (KVQ_OK, KVQ_ERR_NONFINITE):
        _check(rc, "kvq_stats_hi0")
    return v.value


def kvq_rate_sums(stats, L: Layout, s: int, lambdas, sums, stream=None):
    """sums: device int64 [32]; lambdas: up to 32 host floats."""
    lam = (C.c_double * 32)(*list(lambdas)[:32])
    _check(lib().kvq_rate_sums(_ptr(stats), L.c(), int(s), lam, len(lambdas), _ptr(sums),
                               _stream(stream)), "kvq_rate_sums")


def kvq_quantize(x, L: Layout, codebook, k, seed: int, index_base: int, codes, status=None,
                 stream=None):
    _check(lib().kvq_quantize(_ptr(x), L.c(), _ptr(codebook), _ptr(k), int(seed),
                              int(index_base), _ptr(codes), _ptr(status), _stream(stream)),
           "kvq_quantize")


def kvq_dequantize(codes, codebook, L: Layout, y, stream=None):
    _check(lib().kvq_dequantize(_ptr(codes), _ptr(codebook), L.c(), _ptr(y), _stream(stream)),
           "kvq_dequantize")


def kvq_encode_host(x_host, L: Layout, s: int, budget_bits: float, seed: int, index_base: int,
                    x_dev, buf: "Buffers", status, codes_host=None, codebook_host=None,
                    k_host=None, totals_host=None, stream=None):
    """The write path from host memory (see include/kvq.h): x_host a pinned
    [S,T,D] float16 CPU tensor, x_dev its device destination, buf the device
    buffers, status a device int32 [3]; the *_host outputs are pinned CPU
    tensors or None."""
    _check(lib().kvq_encode_host(
        _ptr(x_host), L.c(), int(s), float(budget_bits), int(seed), int(index_base), _ptr(x_dev),
        _ptr(buf.stats), _ptr(buf.lam), _ptr(buf.workspace), _ptr(buf.codebook), _ptr(buf.k),
        _ptr(buf.D_r), _ptr(buf.H_r), _ptr(buf.totals), _ptr(buf.codes), _ptr(status),
        _ptr(codes_host), _ptr(codebook_host), _ptr(k_host), _ptr(totals_host), _stream(stream)),
        "kvq_encode_host")


def kvq_uniform_codebook(x, L: Layout, codebook, k, status, stream=None):
    """Uniform comparator codebooks (see include/kvq.h)."""
    _check(lib().kvq_uniform_codebook(_ptr(x), L.c(), _ptr(codebook), _ptr(k), _ptr(status),
                                      _stream(stream)), "kvq_uniform_codebook")


def kvq_quantize_nearest(x, L: Layout, codebook, k, codes, status=None, stream=None):
    """Round every entry to the nearest level of its block's codebook."""
    _check(lib().kvq_quantize_nearest(_ptr(x), L.c(), _ptr(codebook), _ptr(k), _ptr(codes),
                                      _ptr(status) if status is not None else None,
                                      _stream(stream)), "kvq_quantize_nearest")


def kvq_entropy_slot_bytes(L: Layout) -> int:
    return int(lib().kvq_entropy_slot_bytes(L.c()))


def kvq_entropy_encode(codes, L: Layout, out, nbytes, stream=None):
    """Entropy-code every block's codes into its fixed-capacity slot."""
    _check(lib().kvq_entropy_encode(_ptr(codes), L.c(), _ptr(out), _ptr(nbytes), _stream(stream)),
           "kvq_entropy_encode")


def kvq_entropy_decode(inp, L: Layout, codes, status, stream=None):
    """Decode the slots of kvq_entropy_encode back into packed codes."""
    _check(lib().kvq_entropy_decode(_ptr(inp), L.c(), _ptr(codes), _ptr(status), _stream(stream)),
           "kvq_entropy_decode")


def kvq_entropy_run_bytes(L: Layout, nseg: int) -> int:
    return lib().kvq_entropy_run_bytes(L.c(), int(nseg))


def kvq_entropy_encode_runs(codes, L: Layout, nseg: int, out, nbytes, stream=None):
    _check(lib().kvq_entropy_encode_runs(_ptr(codes), L.c(), int(nseg), _ptr(out), _ptr(nbytes),
                                         _stream(stream)), "kvq_entropy_encode_runs")


def kvq_entropy_decode_runs(inp, L: Layout, nseg: int, codes, status, stream=None):
    _check(lib().kvq_entropy_decode_runs(_ptr(inp), L.c(), int(nseg), _ptr(codes), _ptr(status),
                                         _stream(stream)), "kvq_entropy_decode_runs")


def kvq_attention_workspace_bytes(L: Layout, n_rep: int) -> int:
    return int(lib().kvq_attention_workspace_bytes(L.c(), n_rep))


def kvq_decode_attention(q, n_rep: int, L: Layout, k_codes, k_codebook, v_codes, v_codebook,
                         T_valid: int, scale: float, workspace, out, status=None, stream=None):
    """Attention of one decoding step read from the codes (see include/kvq.h);
    q and out are fp32 [L.S * n_rep, 128] device tensors."""
    _check(lib().kvq_decode_attention(_ptr(q), n_rep, L.c(), _ptr(k_codes), _ptr(k_codebook),
                                      _ptr(v_codes), _ptr(v_codebook), int(T_valid),
                                      float(scale), _ptr(workspace), _ptr(out),
                                      _ptr(status) if status is not None else None,
                                      _stream(stream)), "kvq_decode_attention")


def stats_rows(stats):
    """View of the per-block stats rows inside a kvq_stats buffer: a
    [nblocks, 96] float32 tensor (same device)."""
    recs = stats[STATS_HEADER_BYTES:].view(torch.float32).view(-1, STATS_RECORD_FLOATS)
    return recs[:, :STATS_ROW_FLOATS]


def kvq_allocate_report(workspace) -> dict:
    r = _Report()
    _check(lib().kvq_allocate_report(_ptr(workspace), C.byref(r)), "kvq_allocate_report")
    n = max(r.rounds, 0)
    t0 = r.t_start
    us = lambda t: (t - t0) / 1e3 if t and t0 else None
    return {"rounds": r.rounds, "steps": r.steps, "active": list(r.active)[:n],
            "lambda": r.lambda_, "xa": r.xa, "xb": r.xb,
            "dp_done_us": [us(t) for t in list(r.t_dp)[:n]],
            "control_done_us": [us(t) for t in list(r.t_ctl)[:n]],
            "end_us": us(r.t_end)}


class Buffers:
    """Device buffers of one quantization of a layout (torch allocations)."""

    def __init__(self, L: Layout, s: int, device="cuda"):
        nb = L.nblocks
        dev = torch.device(device)
        self.L, self.s = L, s
        self.stats = torch.empty(kvq_stats_bytes(L), dtype=torch.uint8, device=dev)
        self.workspace = torch.empty(max(kvq_workspace_bytes(L, s), 16), dtype=torch.uint8,
                                     device=dev)
        self.codebook = torch.empty((nb, 16), dtype=torch.float32, device=dev)
        self.k = torch.empty(nb, dtype=torch.uint8, device=dev)
        self.D_r = torch.empty(nb, dtype=torch.float32, device=dev)
        self.H_r = torch.empty(nb, dtype=torch.float32, device=dev)
        self.totals = torch.zeros(3, dtype=torch.float64, device=dev)
        self.lam = torch.zeros(1, dtype=torch.float64, device=dev)
        self.status_stats = torch.zeros(1, dtype=torch.int32, device=dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.status_quant = torch.zeros(1, dtype=torch.int32, device=dev)
        self.codes = torch.empty((nb, 16 * L.group), dtype=torch.uint8, device=dev)


def quantize(x, L: Layout, budget_bits: float, s: int, seed: int = 0, index_base: int = 0,
             mode: int = KVQ_BISECT40, eta: float = 0.0, buf: Buffers = None, stream=None,
             fused: bool = False, weights=None):
    """kvq_stats (kvq_stats_weighted when per-entry distortion weights are
    given) + kvq_allocate + kvq_quantize on x (a [S,T,D] float16 CUDA tensor);
    fused: kvq_allocate_quantize instead of the last two.  Returns the Buffers
    (codes, codebook, k, D_r, H_r, totals, lambda, statuses), all still on the
    device."""
    if buf is None:
        buf = Buffers(L, s, x.device)
    if weights is None:
        kvq_stats(x, L, buf.stats, buf.status_stats, stream=stream)
    else:
        kvq_stats_weighted(x, weights, L, buf.stats, buf.status_stats, stream=stream)
    if fused:
        kvq_allocate_quantize(buf.stats, x, L, s, budget_bits, mode, eta, buf.lam, buf.workspace,
                              buf.codebook, buf.k, buf.D_r, buf.H_r, buf.totals, seed,
                              index_base, buf.codes, buf.status, stream=stream)
        return buf
    kvq_allocate(buf.stats, L, s, budget_bits, mode, eta, buf.lam, buf.workspace, buf.codebook,
                 buf.k, buf.D_r, buf.H_r, buf.totals, buf.status, stream=stream)
    kvq_quantize(x, L, buf.codebook, buf.k, seed, index_base, buf.codes, buf.status_quant,
                 stream=stream)
    return buf
