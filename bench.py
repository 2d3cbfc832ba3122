"""Throughput of the write-time KV-cache quantizer on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step = kvq_stats + kvq_allocate (40-step lambda bisection) + kvq_quantize
over one [S, T, D] binary16 K/V tensor already resident in HBM: the
Llama-3-8B-shaped single-layer prefill (K and V, 8 KV heads each, 8192
tokens, head dim 128; blocks of one head x 32 tokens; s = 16; B = 2.5 bits per
entry).  The step is captured once as a CUDA graph and replayed; L2 is
flushed before every timed step, outside the timed interval (a 256 MB write,
then a 256 MB read so the write's dirty lines are written back before timing
starts).  The metric is binary16 input bytes quantized per second.  The same
step launched eagerly is timed too, with per-kernel events.

Also reported on the same line: per-kernel times, the roofline of the dominant
kernel (algorithmic bytes / measured time / measured HBM peak), an end-to-end
figure through the C ABI with pinned host buffers (host->device copy of the
input and device->host copy of codes, codebooks, k and totals inside the timed
region, pipelined over three streams), the number of our kernel launches, SM clocks sampled during the
timed region, and the CPU oracle timed on a bounded sample (cpu_baseline).

Multi-GPU (torchrun): every rank quantizes its own independent tensor
(replicas: the method has no cross-tensor exchange); value = all ranks' bytes
/ the slowest rank's time.

--impl reference times the CPU oracle (the only reference implementation: the
method's pages publish no code) on the host cores, on bounded samples of the
same workload.
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "fp16 KV GB/s quantized at budget B (1 B300) and fraction of HBM roofline"
# DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum) of the
# layer workload's search and quantize kernels from one ncu capture each
# (cache control on: cold L2), as summarised in
# profiles/kernels_llama3_8b_layer.md; to be taken again whenever either
# kernel changes
SEARCH_DRAM_BYTES = 18524416
QUANT_DRAM_BYTES = 33873408 + 1024000
TRAFFIC_NOTE = "bytes per launch, ncu capture with a cold L2"
WORKLOAD = "llama3_8b_layer"
WORKLOAD_DESC = ("Llama-3-8B-shaped single-layer prefill: K and V, 8 KV heads x 8192 tokens x "
                 "128 dims fp16 (S=16 streams); K = N(0,1) x per-channel lognormal(0,0.5) with 4 "
                 "outlier channels x10, V = Student-t(5); blocks = head x 32 tokens (4096 blocks "
                 "of 4096), s=16, B=2.5 bits/entry, seed 0")
CPU_SAMPLE_BLOCKS = 4096


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6400.0, "fallback"


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        import tempfile
        self.path = tempfile.mktemp(prefix="kvq_clocks_", suffix=".csv")
        try:
            # nvidia-smi writes each sample line itself (-f), so nothing is
            # lost in a pipe buffer when it is stopped
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100", "-f", self.path],
                stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            try:
                with open(self.path) as f:
                    self.lines = [ln.strip() for ln in f if ln.strip()]
                os.unlink(self.path)
            except OSError:
                pass

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def cpu_model() -> str:
    """The host CPU's model name (from /proc/cpuinfo), or "unknown"."""
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


def cpu_baseline(w, x_np, budget_per_entry, nblocks=CPU_SAMPLE_BLOCKS, seed=0):
    """The oracle, as it stands, on a bounded sample: `nblocks` whole blocks
    (half from K streams, half from V streams), full path (stats, 40-step
    bisection at the same bits/entry, quantize).  Returns (GB/s, seconds,
    threads, description)."""
    import numpy as np
    import oracle
    nTB = w.T // 32
    per = nblocks // 2
    half = w.S // 2
    sel = []
    for s0 in (0, half):
        for i in range(per):
            sel.append((s0 + i % half, i // half))
    sl = np.stack([x_np[h, 32 * tb:32 * tb + 32, :] for h, tb in sel])   # [n, 32, D]
    threads = oracle.set_threads(0)
    t0 = time.perf_counter()
    oracle.stats(sl, w.G)
    r = oracle.allocate_bisect(sl, w.G, w.s, budget_per_entry * sl.size)
    oracle.quantize(sl, w.G, r["codebook"], r["k"], seed, 0)
    dt = time.perf_counter() - t0
    return sl.nbytes / dt / 1e9, dt, threads, (
        "%d blocks (%d K + %d V slabs of 32 tokens x 128; all of them when %d) of the workload, "
        "full path (stats, 40-step bisection at the same bits/entry, quantize); %d bytes"
        % (len(sel), per, per, w.nblocks, sl.nbytes))


def step_config(world):
    """The bench step's workload and launch, the same object on both arms."""
    return {"workload": WORKLOAD_DESC,
            "l2": "flushed before each step (256 MB write then 256 MB read, outside the timed "
                  "interval)",
            "launch": "whole step as one CUDA graph replay",
            "parallelism": "replicas" if world > 1 else "single"}


def run_reference(args, rank, world):
    """Reference arm: the CPU oracle on bounded samples (rank 0 only)."""
    if rank != 0:
        return
    import numpy as np
    from rate_adaptive_kv_block_b300 import synth
    w = synth.workload(WORKLOAD)
    x = synth.make_numpy(w, seed=0)
    B = w.budgets[0]
    for _ in range(args.warmup):
        cpu_baseline(w, x, B, nblocks=32)
    vals, secs = [], []
    for _ in range(args.steps):
        gbs, dt, thr, desc = cpu_baseline(w, x, B, nblocks=args.ref_blocks)
        vals.append(gbs)
        secs.append(dt)
    value = sum(args.ref_blocks * 8192 for _ in vals) / sum(secs) / 1e9
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * sum(secs) / len(secs),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "impl": "reference",
        "config": step_config(world),
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": thr, "kind": "oracle",
                         "sample": desc, "cpu_model": cpu_model()},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def comparator_bench(w, L, x, buf, flush_l2, graph_of, device_ms, t_flush, nrep, dev):
    """The page's comparators on the same layer: uniform INT4 (16 equally
    spaced levels from the block's minimum to its maximum, nearest level) and
    uniform stochastic quantization (same levels, unbiased interpolation),
    against the rate-adaptive quantizer at its budget and at the rate the
    INT4 codes would take entropy-coded per block.  Distortion = mean squared
    error of the binary16 decode; rates in bits per entry (entropies of the
    codes' empirical frequencies per block for the uniform ones, sum d_r H_r
    for the rate-adaptive one).  Kernel times with L2 flushed."""
    import torch
    from rate_adaptive_kv_block_b300 import kvq
    nb, d = L.nblocks, 32 * w.G
    xf = x.float()
    y = torch.empty_like(x)

    def mse(codes, cb):
        kvq.kvq_dequantize(codes, cb, L, y)
        return float(((y.float() - xf) ** 2).mean())

    def code_entropy(codes):
        c = torch.stack([codes & 15, codes >> 4], dim=-1).reshape(nb, d).long()
        idx = c + 16 * torch.arange(nb, device=dev).unsqueeze(1)
        n = torch.bincount(idx.reshape(-1), minlength=16 * nb).reshape(nb, 16).double()
        p = n / d
        h = -(torch.where(n > 0, p * torch.log2(p), torch.zeros_like(p))).sum(dim=1)
        return float(h.mean())

    ucb = torch.empty((nb, 16), dtype=torch.float32, device=dev)
    uk = torch.empty(nb, dtype=torch.uint8, device=dev)
    ust = torch.zeros(1, dtype=torch.int32, device=dev)
    ucodes = torch.empty_like(buf.codes)
    g_u = graph_of(lambda: (flush_l2(1), kvq.kvq_uniform_codebook(x, L, ucb, uk, ust),
                            kvq.kvq_quantize_nearest(x, L, ucb, uk, ucodes)))
    device_ms(g_u, 2)
    t_u = device_ms(g_u, nrep) - t_flush
    mse_near = mse(ucodes, ucb)
    h_near = code_entropy(ucodes)
    kvq.kvq_quantize(x, L, ucb, uk, 0, 0, ucodes)
    mse_sto = mse(ucodes, ucb)
    h_sto = code_entropy(ucodes)
    mse_ecasq = mse(buf.codes, buf.codebook)
    rate_ecasq = float(buf.totals[0].item()) / x.numel()
    # the rate-adaptive quantizer at the entropy-coded rate of the INT4 codes
    b2 = kvq.Buffers(L, w.s, dev)
    kvq.quantize(x, L, h_near * x.numel(), w.s, buf=b2)
    torch.cuda.synchronize()
    mse_eq = mse(b2.codes, b2.codebook)
    # fixed-rate: every block at the same bits per entry (its own lambda_r),
    # the same total budget; its kernel time (L2 flushed)
    bpe = w.budgets[0]
    bf_ = kvq.Buffers(L, w.s, dev)
    lam_r = torch.empty(nb, dtype=torch.float64, device=dev)
    bf_.stats.copy_(buf.stats)

    def fixed():
        kvq.kvq_allocate_fixed_rate(bf_.stats, L, w.s, bpe, bf_.codebook, bf_.k, bf_.D_r, bf_.H_r,
                                    lam_r, bf_.totals, bf_.status)
    fixed()
    kvq.kvq_quantize(x, L, bf_.codebook, bf_.k, 0, 0, bf_.codes)
    torch.cuda.synchronize()
    g_f = graph_of(lambda: (flush_l2(1), fixed()))
    device_ms(g_f, 2)
    t_f = device_ms(g_f, max(3, nrep // 4)) - t_flush
    mse_fixed = mse(bf_.codes, bf_.codebook)
    n = x.numel()
    fixed_budget = {"rate_bits": float(bf_.totals[0].item()) / n,
                    "expected_distortion_per_entry": float(bf_.totals[1].item()) / n}
    # the same comparator at equal total rate: the per-block budget b' raised
    # (bisection, 14 steps) until the blocks' total rate is the rate-adaptive
    # allocation's (each block's rate moves in steps, so a cap of b leaves part
    # of b unspent)
    target = float(buf.totals[0].item())
    lo_b, hi_b = bpe, 4.0
    for _ in range(14):
        mid_b = 0.5 * (lo_b + hi_b)
        kvq.kvq_allocate_fixed_rate(bf_.stats, L, w.s, mid_b, bf_.codebook, bf_.k, bf_.D_r,
                                    bf_.H_r, lam_r, bf_.totals, bf_.status)
        if float(bf_.totals[0].item()) <= target:
            lo_b = mid_b
        else:
            hi_b = mid_b
    kvq.kvq_allocate_fixed_rate(bf_.stats, L, w.s, lo_b, bf_.codebook, bf_.k, bf_.D_r, bf_.H_r,
                                lam_r, bf_.totals, bf_.status)
    kvq.kvq_quantize(x, L, bf_.codebook, bf_.k, 0, 0, bf_.codes)
    torch.cuda.synchronize()
    fixed_equal = {"what": "every block at <= b' bits/entry on its own lambda, b' raised until the "
                           "total rate equals the rate-adaptive allocation's",
                   "block_budget_bits": lo_b, "mse": mse(bf_.codes, bf_.codebook),
                   "rate_bits": float(bf_.totals[0].item()) / n,
                   "expected_distortion_per_entry": float(bf_.totals[1].item()) / n,
                   "status": int(bf_.status.item())}
    return {"what": "mean squared error of the binary16 decode and rate in bits/entry on this "
                    "layer; uniform = 16 equally spaced levels per block from its minimum to its "
                    "maximum; uniform rates are the per-block entropies of the codes",
            "uniform_int4_nearest": {"mse": mse_near, "rate_bits": h_near, "stored_bits": 4.0},
            "uniform_stochastic": {"mse": mse_sto, "rate_bits": h_sto, "stored_bits": 4.0},
            "rate_adaptive_at_budget": {"mse": mse_ecasq, "rate_bits": rate_ecasq, "stored_bits": 4.0},
            "rate_adaptive_at_int4_rate": {"mse": mse_eq,
                                           "rate_bits": float(b2.totals[0].item()) / x.numel(),
                                           "stored_bits": 4.0},
            "fixed_rate_at_budget": {"what": "every block at <= %.2f bits/entry on its own lambda "
                                             "(kvq_allocate_fixed_rate): the same total budget as "
                                             "the rate-adaptive allocation" % bpe,
                                     "mse": mse_fixed,
                                     "rate_bits": fixed_budget["rate_bits"],
                                     "expected_distortion_per_entry":
                                         fixed_budget["expected_distortion_per_entry"],
                                     "rate_adaptive_expected_distortion_per_entry":
                                         float(buf.totals[1].item()) / n,
                                     "allocate_ms": t_f},
            "fixed_rate_at_equal_rate": fixed_equal,
            "uniform_int4_ms": t_u,
            "uniform_int4_GBps": (x.numel() * 2 + x.numel() // 2 + nb * 65) / (t_u * 1e-3) / 1e9}


def weighted_bench(w, L, x, buf, flush_l2, graph_of, device_ms, t_flush, nrep, dev):
    """D_r weighted by attention sensitivity (kvq_stats_weighted) on the same
    layer at the same budget: seeded synthetic sensitivities (keys per
    feature, values per token, each stream's mean 1), the weighted stats
    kernel and the whole weighted step with L2 flushed, and the weighted and
    plain squared error of the binary16 decode for the weighted allocation and
    for the unweighted one (buf)."""
    import torch
    from rate_adaptive_kv_block_b300 import kvq, synth
    s, B = w.s, w.budgets[0] * x.numel()
    Wt = synth.weights_torch(w, seed=7, device=dev)
    bw = kvq.Buffers(L, s, dev)

    def stats_w():
        kvq.kvq_stats_weighted(x, Wt, L, bw.stats, bw.status_stats)

    def step_w():
        stats_w()
        kvq.kvq_allocate(bw.stats, L, s, B, kvq.KVQ_BISECT40, 0.0, bw.lam, bw.workspace,
                         bw.codebook, bw.k, bw.D_r, bw.H_r, bw.totals, bw.status)
        kvq.kvq_quantize(x, L, bw.codebook, bw.k, 0, 0, bw.codes, bw.status_quant)

    step_w()
    torch.cuda.synchronize()
    if int(bw.status_stats.item()) != 0 or int(bw.status.item()) != 0:
        raise SystemExit("weighted path status %d / %d" % (int(bw.status_stats.item()),
                                                          int(bw.status.item())))
    g_sw = graph_of(lambda: (flush_l2(1), stats_w()))
    g_stw = graph_of(lambda: (flush_l2(1), step_w()))
    device_ms(g_sw, 2)
    device_ms(g_stw, 2)
    t_sw = device_ms(g_sw, nrep) - t_flush
    t_stw = device_ms(g_stw, nrep) - t_flush
    xf = x.float()
    y = torch.empty_like(x)

    def errs(b):
        kvq.kvq_dequantize(b.codes, b.codebook, L, y)
        e2 = (y.float() - xf) ** 2
        return float((Wt * e2).sum() / Wt.sum()), float(e2.mean())

    we_w, mse_w = errs(bw)
    we_u, mse_u = errs(buf)
    n = x.numel()
    return {"what": "distortion weighted per entry by synthetic attention sensitivities "
                    "(keys: per feature, values: per token); errors of one stochastic "
                    "decode, weighted error = sum w e^2 / sum w",
            "stats_weighted_ms": t_sw,
            "stats_weighted_GBps": (n * 6 + L.nblocks * 4800) / (t_sw * 1e-3) / 1e9,
            "step_weighted_ms": t_stw,
            "lambda": float(bw.lam.item()),
            "weighted_allocation": {"weighted_err": we_w, "mse": mse_w,
                                    "rate_bits": float(bw.totals[0].item()) / n},
            "unweighted_allocation": {"weighted_err": we_u, "mse": mse_u,
                                      "rate_bits": float(buf.totals[0].item()) / n}}


def entropy_bench(w, L, x, buf, flush_l2, graph_of, device_ms, t_flush, nrep, dev):
    """The layer's codes entropy-coded (kvq_entropy_encode): stored bits per
    entry against the rate the allocation targets, and the coder's times
    (L2 flushed before each launch)."""
    import torch
    from rate_adaptive_kv_block_b300 import kvq
    nb = L.nblocks
    cap = kvq.kvq_entropy_slot_bytes(L)
    out = torch.zeros((nb, cap), dtype=torch.uint8, device=dev)
    nbytes = torch.zeros(nb, dtype=torch.int32, device=dev)
    back = torch.empty_like(buf.codes)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    g_e = graph_of(lambda: (flush_l2(1), kvq.kvq_entropy_encode(buf.codes, L, out, nbytes)))
    g_d = graph_of(lambda: (flush_l2(1), kvq.kvq_entropy_decode(out, L, back, st)))
    device_ms(g_e, 2)
    device_ms(g_d, 2)
    t_e = device_ms(g_e, nrep) - t_flush
    t_d = device_ms(g_d, nrep) - t_flush
    torch.cuda.synchronize()
    assert torch.equal(back, buf.codes) and int(st.item()) == 0
    stored = float(nbytes.double().sum())
    n = x.numel()
    # coding across adjacent blocks: runs of 16 consecutive blocks
    nseg = 16
    nruns = -(-nb // nseg)
    rcap = kvq.kvq_entropy_run_bytes(L, nseg)
    rout = torch.zeros((nruns, rcap), dtype=torch.uint8, device=dev)
    rbytes = torch.zeros(nruns, dtype=torch.int32, device=dev)
    rback = torch.empty_like(buf.codes)
    g_re = graph_of(lambda: (flush_l2(1), kvq.kvq_entropy_encode_runs(buf.codes, L, nseg, rout, rbytes)))
    g_rd = graph_of(lambda: (flush_l2(1), kvq.kvq_entropy_decode_runs(rout, L, nseg, rback, st)))
    device_ms(g_re, 2)
    device_ms(g_rd, 2)
    t_re = device_ms(g_re, nrep) - t_flush
    t_rd = device_ms(g_rd, nrep) - t_flush
    torch.cuda.synchronize()
    assert torch.equal(rback, buf.codes) and int(st.item()) == 0
    rstored = float(rbytes.double().sum())
    return {"what": "the layer's 4-bit codes entropy-coded per block (rANS, exact counts, 32 "
                    "streams per block); bits per entry include the 96-byte block headers, not "
                    "the 64-byte codebooks",
            "stored_bits_per_entry": stored * 8 / n, "rate_target_bits": float(buf.totals[0]) / n,
            "runs_of_adjacent_blocks": {"blocks_per_run": nseg,
                                        "stored_bits_per_entry": rstored * 8 / n,
                                        "encode_ms": t_re, "decode_ms": t_rd,
                                        "what": "32 rANS streams per run of 16 consecutive blocks, "
                                                "states carried across the blocks; counts "
                                                "(32 B) per block, states and lengths per run"},
            "packed_bits_per_entry": 4.0,
            "encode_ms": t_e, "decode_ms": t_d,
            "encode_GBps_of_codes": (n / 2) / (t_e * 1e-3) / 1e9,
            "decode_GBps_of_codes": (n / 2) / (t_d * 1e-3) / 1e9}


def attention_bench(w, L, buf, flush_l2, graph_of, device_ms, t_flush, nrep, hbm, src, dev):
    """kvq_decode_attention on the quantized layer, L2 flushed before every
    launch: its time (by subtraction of flush-only replays), the bytes it must read
    (codes, codebooks, queries) and the fraction of the HBM roofline;
    PyTorch's attention on the binary16 decode of the same cache, timed the
    same way, for comparison."""
    import math
    import torch
    import torch.nn.functional as F
    from rate_adaptive_kv_block_b300 import kvq
    S_kv, D, n_rep = w.S // 2, w.D, 4
    half = S_kv * (w.T // 32) * (w.D // w.G)          # blocks of the K streams
    L_kv = kvq.Layout(S_kv, w.T, w.D, w.G)
    g = torch.Generator(device="cpu").manual_seed(1)
    qa = torch.randn((S_kv * n_rep, D), generator=g).to(dev)
    out = torch.empty_like(qa)
    ws = torch.empty(kvq.kvq_attention_workspace_bytes(L_kv, n_rep), dtype=torch.uint8, device=dev)
    kc, vc = buf.codes[:half], buf.codes[half:]
    kcb, vcb = buf.codebook[:half], buf.codebook[half:]
    scale = 1.0 / math.sqrt(D)

    def run():
        kvq.kvq_decode_attention(qa, n_rep, L_kv, kc, kcb, vc, vcb, w.T, scale, ws, out)

    # a call this short is timed by subtraction over many replays: a graph of
    # (L2 flush, call) and a graph of the flush alone, each replayed 200
    # times between events, five times over; the median of the differences
    # (events around one short replay move in 2.048 us steps on this GPU)
    def median_cold_ms(fn, n):
        gf = graph_of(lambda: flush_l2(0))
        gk = graph_of(lambda: (flush_l2(0), fn()))
        device_ms(gk, 3)
        ts = sorted(device_ms(gk, n) - device_ms(gf, n) for _ in range(5))
        return ts[len(ts) // 2]
    t_att = median_cold_ms(run, 200)
    nbytes = 2 * half * 16 * w.G + 2 * half * 64 + 2 * qa.numel() * 4
    res = {"what": "one decoding step: %d query heads, %d KV heads x %d tokens x %d, read from "
                   "the 4-bit codes" % (S_kv * n_rep, S_kv, w.T, D),
           "ms": t_att, "bytes": nbytes, "GBps": nbytes / (t_att * 1e-3) / 1e9,
           "roofline": {"bound": "hbm", "achieved": nbytes / (t_att * 1e-3) / 1e9, "peak": hbm,
                        "unit": "GB/s", "frac": nbytes / (t_att * 1e-3) / 1e9 / hbm,
                        "peak_source": src},
           "kernels_per_call": 2}
    try:
        y16 = torch.empty((w.S, w.T, D), dtype=torch.float16, device=dev)
        kvq.kvq_dequantize(buf.codes, buf.codebook, L, y16)
        Kf, Vf = y16[:S_kv].unsqueeze(0), y16[S_kv:].unsqueeze(0)
        qh = qa.half().view(1, S_kv * n_rep, 1, D)
        ref = {}

        def sdpa():
            ref["o"] = F.scaled_dot_product_attention(qh, Kf, Vf, scale=scale, enable_gqa=True)
        sdpa()
        t_sdpa = median_cold_ms(sdpa, 200)
        run()
        torch.cuda.synchronize()
        diff = (ref["o"].view(-1, D).float() - out).abs().max().item()
        res["torch_sdpa_fp16"] = {"ms": t_sdpa, "bytes": 2 * S_kv * w.T * D * 2,
                                  "max_abs_diff_vs_ours": diff}
    except Exception as e:                          # the comparison is context only
        res["torch_sdpa_fp16"] = {"unavailable": str(e)[:200]}
    return res


def other_configs_bench(dev, hbm, src):
    """The other synthetic workloads, each resident in HBM and larger than
    L2 (no flush needed between steps), timed with CUDA events:
      * full_model_cache: 32 layers x {K, V} x 8 heads x 32768 tokens x 128
        (4.3 GB), one global lambda at B = 2.0: the whole path
        (stats + allocate + quantize) per step;
      * decode_admission: per step 64 sequences x 32 layers x {K, V} x 8
        heads append one 32-token block (268 MB); lambda from the bisection
        at step 0, then one subgradient step per call (eta = 1e-6, B = 2.5);
        64 timed steps cycling 8 pre-drawn step tensors: per-step latency
        (median, p99) and the lambda trace;
      * hadamard_groups: 8 heads x 131072 tokens x 128 after the 128-point
        Hadamard rotation, 32-feature groups: stats once, then allocate +
        quantize for each budget 1.5 / 2 / 3 / 4 bits per entry."""
    import torch
    from rate_adaptive_kv_block_b300 import kvq, synth
    stream = torch.cuda.current_stream()
    out = {}

    def ev():
        return torch.cuda.Event(enable_timing=True)

    # ---- full model cache
    w = synth.workload("full_model_cache")
    x = synth.make_torch(w, seed=0, device=dev)
    L = kvq.Layout(w.S, w.T, w.D, w.G)
    B = w.budgets[0] * w.entries
    buf = kvq.Buffers(L, w.s, dev)

    def step3():
        kvq.kvq_stats(x, L, buf.stats, buf.status_stats)
        kvq.kvq_allocate(buf.stats, L, w.s, B, kvq.KVQ_BISECT40, 0.0, buf.lam, buf.workspace,
                         buf.codebook, buf.k, buf.D_r, buf.H_r, buf.totals, buf.status)
        kvq.kvq_quantize(x, L, buf.codebook, buf.k, 0, 0, buf.codes, buf.status_quant)
    for _ in range(2):
        step3()
    torch.cuda.synchronize()
    assert int(buf.status.item()) == 0
    ts = []
    for _ in range(5):
        a, b = ev(), ev()
        a.record(stream)
        step3()
        b.record(stream)
        torch.cuda.synchronize()
        ts.append(a.elapsed_time(b))
    ms = statistics.median(ts)
    rep = kvq.kvq_allocate_report(buf.workspace)
    out["full_model_cache"] = {
        "workload": "32 layers x {K,V} x 8 heads x 32768 tokens x 128 fp16 (4.3 GB), 524288 "
                    "blocks of 4096, s=16, B=2.0 bits/entry",
        "ms_per_step_median": ms, "GBps": x.numel() * 2 / (ms * 1e-3) / 1e9,
        "tokens_per_s": w.T / (ms * 1e-3), "lambda": float(buf.lam.item()),
        "rate_bits_per_entry": float(buf.totals[0].item()) / w.entries,
        "search_rounds": rep["rounds"], "search_active_blocks": rep["active"],
        "l2": "input 34x larger than L2: no flush"}
    del x, buf
    torch.cuda.empty_cache()

    # ---- decode admission: subgradient steps
    w = synth.workload("decode_admission")
    L = kvq.Layout(w.S, w.T, w.D, w.G)
    B = w.budgets[0] * w.entries
    xs = [synth.make_torch(w, seed=1000 + i, device=dev) for i in range(8)]
    buf = kvq.Buffers(L, w.s, dev)

    def step4(xt, t, mode):
        kvq.kvq_stats(xt, L, buf.stats, buf.status_stats)
        kvq.kvq_allocate(buf.stats, L, w.s, B, mode, w.eta if mode == kvq.KVQ_SUBGRADIENT else 0.0,
                         buf.lam, buf.workspace, buf.codebook, buf.k, buf.D_r, buf.H_r, buf.totals,
                         buf.status)
        kvq.kvq_quantize(xt, L, buf.codebook, buf.k, t, 0, buf.codes, buf.status_quant)
    step4(xs[0], 0, kvq.KVQ_BISECT40)                  # step 0: the bisection warm start
    torch.cuda.synchronize()
    lam0 = float(buf.lam.item())
    for t in range(1, 4):                               # warm-up subgradient steps
        step4(xs[t % 8], t, kvq.KVQ_SUBGRADIENT)
    torch.cuda.synchronize()
    n = 64
    evs = [(ev(), ev()) for _ in range(n)]
    trace = []
    lam_dev = torch.empty(n, dtype=torch.float64, device=dev)
    for i in range(n):
        evs[i][0].record(stream)
        step4(xs[(4 + i) % 8], 4 + i, kvq.KVQ_SUBGRADIENT)
        evs[i][1].record(stream)
        lam_dev[i:i + 1].copy_(buf.lam)
    torch.cuda.synchronize()
    lat = sorted(a.elapsed_time(b) for a, b in evs)
    trace = [lam0] + lam_dev.cpu().tolist()
    med = statistics.median(lat)
    out["decode_admission"] = {
        "workload": "per step 64 sequences x 32 layers x {K,V} x 8 heads x 32 tokens x 128 fp16 "
                    "(268 MB, 32768 blocks of 4096), s=16, B=2.5 bits/entry, subgradient eta=1e-6 "
                    "after a bisection warm start; 8 pre-drawn step tensors cycled",
        "steps": n, "ms_per_step_median": med, "ms_per_step_p99": lat[min(n - 1, int(0.99 * n))],
        "ms_per_step_min": lat[0], "GBps_median": xs[0].numel() * 2 / (med * 1e-3) / 1e9,
        "tokens_per_s_median": 64 / (med * 1e-3),
        "lambda_trace": trace[:17], "lambda_trace_every": "step 0 (bisection), then steps 4..",
        "l2": "each step's input (268 MB) is larger than L2: no flush"}
    del xs, buf
    torch.cuda.empty_cache()

    # ---- Hadamard-rotated groups: budget sweep on one stats result
    w = synth.workload("hadamard_groups")
    L = kvq.Layout(w.S, w.T, w.D, w.G)
    x = synth.make_torch(w, seed=0, device=dev)
    buf = kvq.Buffers(L, w.s, dev)
    a, b = ev(), ev()
    kvq.kvq_stats(x, L, buf.stats, buf.status_stats)   # warm
    torch.cuda.synchronize()
    a.record(stream)
    kvq.kvq_stats(x, L, buf.stats, buf.status_stats)
    b.record(stream)
    torch.cuda.synchronize()
    t_stats = a.elapsed_time(b)
    sweep = []
    for bpe in w.budgets:
        Bb = bpe * w.entries

        def aq():
            kvq.kvq_allocate(buf.stats, L, w.s, Bb, kvq.KVQ_BISECT40, 0.0, buf.lam, buf.workspace,
                             buf.codebook, buf.k, buf.D_r, buf.H_r, buf.totals, buf.status)
            kvq.kvq_quantize(x, L, buf.codebook, buf.k, 0, 0, buf.codes, buf.status_quant)
        aq()
        torch.cuda.synchronize()
        ta, tq = [], []
        for _ in range(5):
            e0, e1, e2 = ev(), ev(), ev()
            e0.record(stream)
            kvq.kvq_allocate(buf.stats, L, w.s, Bb, kvq.KVQ_BISECT40, 0.0, buf.lam, buf.workspace,
                             buf.codebook, buf.k, buf.D_r, buf.H_r, buf.totals, buf.status)
            e1.record(stream)
            kvq.kvq_quantize(x, L, buf.codebook, buf.k, 0, 0, buf.codes, buf.status_quant)
            e2.record(stream)
            torch.cuda.synchronize()
            ta.append(e0.elapsed_time(e1))
            tq.append(e1.elapsed_time(e2))
        assert int(buf.status.item()) == 0
        rep = kvq.kvq_allocate_report(buf.workspace)
        ma, mq = statistics.median(ta), statistics.median(tq)
        qb = x.numel() * 2.5 + L.nblocks * 65
        sweep.append({"bits_per_entry": bpe, "allocate_ms": ma, "quantize_ms": mq,
                      "quantize_frac_hbm": qb / (mq * 1e-3) / 1e9 / hbm,
                      "GBps_allocate_quantize": x.numel() * 2 / ((ma + mq) * 1e-3) / 1e9,
                      "lambda": float(buf.lam.item()),
                      "rate_bits_per_entry": float(buf.totals[0].item()) / w.entries,
                      "search_rounds": rep["rounds"]})
    out["hadamard_groups"] = {
        "workload": "8 heads x 131072 tokens x 128 fp16 after a 128-point Hadamard rotation "
                    "(268 MB), 32-feature groups: 131072 blocks of 1024, s=16",
        "stats_ms": t_stats, "stats_GBps": x.numel() * 2 / (t_stats * 1e-3) / 1e9,
        "sweep": sweep, "peak_source": src, "l2": "input (268 MB) larger than L2: no flush"}
    del x, buf
    torch.cuda.empty_cache()
    return out


def run_sharded(args, rank, world, local):
    """Several GPUs on one tensor under one global lambda: rank r holds the
    layer-shaped shard r (the same workload, drawn with seed r), the total
    budget is 2.5 bits per entry over every shard, and the lambda search runs
    in rounds with one all-reduce of 32 integer rate sums per round
    (sharded.allocate); stats, the final choice and quantize are local.  The
    step is timed eagerly (host round trips between rounds), L2 flushed
    before it, between barriers; value = all ranks' bytes / the slowest
    rank's time."""
    import numpy as np
    import torch
    import torch.distributed as dist
    from rate_adaptive_kv_block_b300 import kvq, sharded, synth
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    use_dist = world > 1 or "RANK" in os.environ     # torchrun: NCCL even for one rank
    if use_dist and not dist.is_initialized():
        dist.init_process_group("nccl")
    w = synth.workload(WORKLOAD)
    x_np = synth.make_numpy(w, seed=rank)
    x = torch.from_numpy(x_np.view(np.int16)).view(torch.float16).to(dev)
    L = kvq.Layout(w.S, w.T, w.D, w.G)
    B = w.budgets[0] * w.entries * world
    buf = kvq.Buffers(L, w.s, dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    in_bytes = x.numel() * 2

    def step(xin):
        kvq.kvq_stats(xin, L, buf.stats, buf.status_stats)
        lam, st, rounds = sharded.allocate(buf.stats, L, w.s, B, buf)
        kvq.kvq_quantize(xin, L, buf.codebook, buf.k, 0, 0, buf.codes, buf.status_quant)
        return lam, st, rounds

    def barrier():
        if use_dist:
            dist.barrier()

    for i in range(args.warmup):
        flush.fill_(i & 0xff)
        info = step(x)
    torch.cuda.synchronize()
    if info[1] != 0 or int(buf.status.item()) != 0:
        raise SystemExit("sharded allocation status %d / %d" % (info[1], int(buf.status.item())))
    with ClockSampler(local) as clk:
        ts = []
        for i in range(args.steps):
            flush.fill_(i & 0xff)
            torch.cuda.synchronize()
            barrier()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            info = step(x)
            b.record(stream)
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(b))
        # end to end: the input from pinned host memory, the codes, codebooks,
        # k and totals back, inside the timed interval
        x_host = torch.from_numpy(x_np.view(np.int16)).view(torch.float16).pin_memory()
        xe = torch.empty_like(x)
        outs = dict(codes=torch.empty(buf.codes.shape, dtype=torch.uint8).pin_memory(),
                    codebook=torch.empty(buf.codebook.shape, dtype=torch.float32).pin_memory(),
                    k=torch.empty(buf.k.shape, dtype=torch.uint8).pin_memory(),
                    totals=torch.empty(3, dtype=torch.float64).pin_memory())
        te = []
        for i in range(args.steps):
            flush.fill_(i & 0xff)
            torch.cuda.synchronize()
            barrier()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            xe.copy_(x_host, non_blocking=True)
            step(xe)
            for key, t in outs.items():
                t.copy_(getattr(buf, key), non_blocking=True)
            b.record(stream)
            torch.cuda.synchronize()
            te.append(a.elapsed_time(b))
    tot = torch.tensor([sum(ts), sum(te)], dtype=torch.float64, device=dev)
    if use_dist:
        dist.all_reduce(tot, op=dist.ReduceOp.MAX)
    tot_ms, tot_e2e = float(tot[0].item()), float(tot[1].item())
    value = world * args.steps * in_bytes / (tot_ms * 1e-3) / 1e9
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        gbs, dt, thr, desc = cpu_baseline(w, x_np, w.budgets[0])
        cpu = {"value": gbs, "unit": "GB/s", "cores": thr, "kind": "oracle", "sample": desc,
               "seconds": dt, "cpu_model": cpu_model()}
    if rank == 0:
        h2d = x_host.numel() * 2
        d2h = sum(t.numel() * t.element_size() for t in outs.values())
        line = {
            "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": tot_ms / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic",
            "config": {"workload": WORKLOAD_DESC + "; rank r holds shard r (seed r), one global "
                                                   "lambda over all shards",
                       "l2": "flushed before each step (256 MB write, outside the timed interval)",
                       "launch": "eager (the lambda search's rounds return to the host)",
                       "parallelism": "sharded lambda over %d GPUs (all-reduce of 32 int64 "
                                      "rate sums per search round)" % world},
            "tokens_per_s": world * args.steps * w.T / (tot_ms * 1e-3),
            "lambda": info[0], "search_rounds": info[2],
            "e2e": {"value": world * args.steps * in_bytes / (tot_e2e * 1e-3) / 1e9,
                    "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "how": "C-ABI calls with the input copied from pinned host memory and the "
                           "codes, codebooks, k and totals copied back inside each step"},
            "gpu_launches": args.steps * (4 + info[2]),   # stats, a rate-sum kernel per round, control init + search kernel, quantize
            "clocks": clk.summary(),
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)
    if use_dist:
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ref-blocks", type=int, default=CPU_SAMPLE_BLOCKS)
    ap.add_argument("--no-other-configs", action="store_true")
    ap.add_argument("--sharded", action="store_true",
                    help="the multi-GPU mode (one global lambda over every rank's shard) also "
                         "at one GPU")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if world > 1 or args.sharded:
        run_sharded(args, rank, world, local)
        return

    import numpy as np
    import torch
    from rate_adaptive_kv_block_b300 import kvq, synth

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
        pg = dist

    w = synth.workload(WORKLOAD)
    x_np = synth.make_numpy(w, seed=rank)
    x = torch.from_numpy(x_np.view(np.int16)).view(torch.float16).to(dev)
    L = kvq.Layout(w.S, w.T, w.D, w.G)
    B = w.budgets[0] * w.entries
    s = w.s
    buf = kvq.Buffers(L, s, dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    flush_r = torch.ones(64 << 20, dtype=torch.float32, device=dev)
    sink = torch.empty(1, dtype=torch.float32, device=dev)

    def flush_l2(i):
        # write 256 MB (evicts the input), then read 256 MB so the dirty lines
        # of the write are written back before the timed interval starts
        flush.fill_(i & 0xff)
        torch.sum(flush_r, dim=0, keepdim=True, out=sink)
    stream = torch.cuda.current_stream()
    in_bytes = x.numel() * 2
    nb = L.nblocks

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        kvq.kvq_stats(x, L, buf.stats, buf.status_stats)
        if ev is not None:
            ev[1].record(stream)
        kvq.kvq_allocate(buf.stats, L, s, B, kvq.KVQ_BISECT40, 0.0, buf.lam, buf.workspace,
                         buf.codebook, buf.k, buf.D_r, buf.H_r, buf.totals, buf.status)
        if ev is not None:
            ev[2].record(stream)
        kvq.kvq_quantize(x, L, buf.codebook, buf.k, 0, 0, buf.codes, buf.status_quant)
        if ev is not None:
            ev[3].record(stream)

    # the whole step captured once as a CUDA graph (the C-ABI calls are
    # stream-ordered and capture-safe after their first call on a device)
    for _ in range(args.warmup):
        flush_l2(0)
        step()
    torch.cuda.synchronize()
    st = int(buf.status.item())
    if st != 0:
        raise SystemExit("allocation status %d (%s)" % (st, kvq.kvq_status_string(st)))
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    torch.cuda.synchronize()

    def timed(run, n):
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(n)]
        for i in range(n):
            flush_l2(i)
            ev[i][0].record(stream)
            run()
            ev[i][1].record(stream)
        torch.cuda.synchronize()
        return [a.elapsed_time(b) for a, b in ev]

    with ClockSampler(local) as clk:
        for i in range(args.warmup):
            flush_l2(i)
            graph.replay()
        if pg:
            pg.barrier()
        torch.cuda.synchronize()
        t_step = timed(graph.replay, args.steps)
        # the same step launched eagerly, with per-kernel events
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
        for i in range(args.steps):
            flush_l2(i)
            step(evs[i])
        torch.cuda.synchronize()
    st = int(buf.status.item())
    if st != 0:
        raise SystemExit("allocation status %d (%s)" % (st, kvq.kvq_status_string(st)))
    t_stats = [e[0].elapsed_time(e[1]) for e in evs]
    t_alloc = [e[1].elapsed_time(e[2]) for e in evs]
    t_quant = [e[2].elapsed_time(e[3]) for e in evs]
    t_eager = [e[0].elapsed_time(e[3]) for e in evs]
    tot_ms = sum(t_step)
    if pg:
        t = torch.tensor([tot_ms], device=dev, dtype=torch.float64)
        pg.all_reduce(t, op=pg.ReduceOp.MAX)
        tot_ms = float(t.item())
    value = world * args.steps * in_bytes / (tot_ms * 1e-3) / 1e9

    # Each kernel alone with a cold L2, in its own launch configuration: one
    # graph runs (L2 flush, kernel), another the flush alone; N back-to-back
    # replays of each are timed on the device and the difference per replay
    # is the kernel's time (no host launch overhead inside it).
    def graph_of(fn):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        return g

    def device_ms(g, n):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        a.record(stream)
        for _ in range(n):
            g.replay()
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / n

    g_flush = graph_of(lambda: flush_l2(1))
    g_stats = graph_of(lambda: (flush_l2(1), kvq.kvq_stats(x, L, buf.stats, buf.status_stats)))
    g_alloc = graph_of(lambda: (flush_l2(1), kvq.kvq_allocate(
        buf.stats, L, s, B, kvq.KVQ_BISECT40, 0.0, buf.lam, buf.workspace, buf.codebook, buf.k,
        buf.D_r, buf.H_r, buf.totals, buf.status)))
    g_quant = graph_of(lambda: (flush_l2(1), kvq.kvq_quantize(x, L, buf.codebook, buf.k, 0, 0,
                                                              buf.codes, buf.status_quant)))
    # the same search with emit and quantize fused into its persistent kernel
    # (kvq_allocate_quantize), reported beside the separate calls
    g_fused = graph_of(lambda: (flush_l2(1), kvq.kvq_allocate_quantize(
        buf.stats, x, L, s, B, kvq.KVQ_BISECT40, 0.0, buf.lam, buf.workspace, buf.codebook, buf.k,
        buf.D_r, buf.H_r, buf.totals, 0, 0, buf.codes, buf.status)))
    nrep = max(args.steps, 10)
    for g_ in (g_flush, g_stats, g_alloc, g_quant, g_fused):
        device_ms(g_, 2)
    t_flush = device_ms(g_flush, nrep)
    t_scold = device_ms(g_stats, nrep) - t_flush
    t_acold = device_ms(g_alloc, nrep) - t_flush
    rep_cold = kvq.kvq_allocate_report(buf.workspace)     # the last replay: cold L2
    t_qcold = device_ms(g_quant, nrep) - t_flush
    t_fcold = device_ms(g_fused, nrep) - t_flush

    # decode attention over this layer's stored cache (kvq_decode_attention):
    # 32 query heads (4 per KV head) on the 8 K and 8 V streams, every token;
    # beside it PyTorch's scaled_dot_product_attention on the binary16 decode
    # of the same cache (a library kernel, for context)
    att = attention_bench(w, L, buf, flush_l2, graph_of, device_ms, t_flush, nrep, *peaks(), dev)
    comp = comparator_bench(w, L, x, buf, flush_l2, graph_of, device_ms, t_flush, nrep, dev)
    ent = entropy_bench(w, L, x, buf, flush_l2, graph_of, device_ms, t_flush, nrep, dev)
    wtd = weighted_bench(w, L, x, buf, flush_l2, graph_of, device_ms, t_flush, nrep, dev)
    others = None if args.no_other_configs else other_configs_bench(dev, *peaks())

    # End to end through the C ABI from pinned host memory: one
    # kvq_encode_host call per step (the input copied in by four copy
    # engines at once, the three kernels, the codes, codebooks, k and totals
    # copied out), steps alternating between two streams and two sets of
    # buffers the way a serving loop would run them, so that step i's copy in
    # overlaps step i-1's kernels and result copy.  The L2 flush runs on the
    # step's stream before its call, inside the timed interval.
    x_host = torch.from_numpy(x_np.view(np.int16)).view(torch.float16).pin_memory()
    bufs = [buf, kvq.Buffers(L, s, dev)]
    xes = [torch.empty_like(x), torch.empty_like(x)]
    sts = [torch.zeros(3, dtype=torch.int32, device=dev) for _ in range(2)]
    outs_h = [dict(codes=torch.empty(buf.codes.shape, dtype=torch.uint8).pin_memory(),
                   codebook=torch.empty(buf.codebook.shape, dtype=torch.float32).pin_memory(),
                   k=torch.empty(buf.k.shape, dtype=torch.uint8).pin_memory(),
                   totals=torch.empty(3, dtype=torch.float64).pin_memory()) for _ in range(2)]
    h2d = x_host.numel() * 2
    d2h = sum(t.numel() * t.element_size() for t in outs_h[0].values())
    e2e_streams = [torch.cuda.Stream(dev), torch.cuda.Stream(dev)]

    def e2e_run(n):
        torch.cuda.synchronize()
        cur = torch.cuda.current_stream()
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(cur)
        for st_ in e2e_streams:
            st_.wait_event(t0)
        for i in range(n):
            j = i & 1
            st_, oh = e2e_streams[j], outs_h[j]
            with torch.cuda.stream(st_):
                flush_l2(i)
                kvq.kvq_encode_host(x_host, L, s, B, 0, 0, xes[j], bufs[j], sts[j], oh["codes"],
                                    oh["codebook"], oh["k"], oh["totals"], stream=st_)
        for st_ in e2e_streams:
            cur.wait_stream(st_)
        t1.record(cur)                                # after the last result copy
        torch.cuda.synchronize()
        return t0.elapsed_time(t1)

    ref_codes = buf.codes.cpu()
    e2e_run(args.warmup)
    t_e2e = e2e_run(args.steps)
    if pg:
        t = torch.tensor([t_e2e], device=dev, dtype=torch.float64)
        pg.all_reduce(t, op=pg.ReduceOp.MAX)
        t_e2e = float(t.item())
    e2e_val = world * args.steps * in_bytes / (t_e2e * 1e-3) / 1e9
    if not torch.equal(outs_h[(args.steps - 1) & 1]["codes"], ref_codes):
        raise SystemExit("end-to-end codes differ from the device-resident run")
    if any(v != 0 for st_ in sts for v in st_.tolist()):
        raise SystemExit("end-to-end statuses %s" % [st_.tolist() for st_ in sts])

    hbm, src = peaks()
    mean = lambda v: sum(v) / len(v)
    # algorithmic bytes per launch (per entry / per block figures)
    q_bytes = in_bytes + in_bytes // 4 + nb * (64 + 1)
    s_bytes = in_bytes + nb * 384
    kern = {
        "step_ms_graph_median": statistics.median(t_step), "step_ms_graph_min": min(t_step),
        "step_ms_eager_mean": mean(t_eager), "step_ms_eager_median": statistics.median(t_eager),
        "eager_stats_ms": mean(t_stats), "eager_allocate_ms": mean(t_alloc),
        "eager_quantize_ms": mean(t_quant),
        "stats_cold_ms": t_scold, "quantize_cold_ms": t_qcold, "allocate_cold_ms": t_acold,
        "fused_allocate_quantize_cold_ms": t_fcold,
        "decode_attention": att,
        "comparators": comp,
        "entropy_coding": ent,
        "weighted_distortion": wtd,
        "other_configs": others,
        "cold_method": "graph (L2 flush + kernel) minus graph (L2 flush), device-timed",
        "stats_cold_GBps": s_bytes / (t_scold * 1e-3) / 1e9,
        "quantize_cold_GBps": q_bytes / (t_qcold * 1e-3) / 1e9,
    }
    kern["quantize_cold_frac_hbm"] = kern["quantize_cold_GBps"] / hbm
    kern["stats_cold_frac_hbm"] = kern["stats_cold_GBps"] / hbm
    # the quantize kernel against the HBM roofline (2.5 B per entry + 65 B per block)
    kern["quantize_roofline"] = {"bound": "hbm", "achieved": kern["quantize_cold_GBps"],
                                 "peak": hbm, "unit": "GB/s",
                                 "frac": kern["quantize_cold_GBps"] / hbm,
                                 "traffic": QUANT_DRAM_BYTES, "traffic_unit": TRAFFIC_NOTE,
                                 "peak_source": src}
    shares = {"stats": t_scold, "allocate": t_acold, "quantize": t_qcold}
    dominant = max(shares, key=shares.get)
    clk = clk_summary = clk.summary()
    sm_mhz = clk_summary["sm_mhz"] or 2032.0
    rep = kvq.kvq_allocate_report(buf.workspace)
    kern["search_rounds"] = rep["rounds"]
    kern["search_active_blocks"] = rep["active"]
    kern["search_timeline_us"] = {"what": "device clock from the search kernel's start, after "
                                          "a cold-L2 replay: each round's evaluations all in, "
                                          "its control published; end = emit and totals done",
                                  "dp_done": rep_cold["dp_done_us"],
                                  "control_done": rep_cold["control_done_us"],
                                  "end": rep_cold["end_us"]}
    # exact DP of one block at one lambda: 680 (i < j < l) level triples, one
    # fp32 multiply-add and one min each
    dp_ops = sum(rep["active"]) * 32 * 680 * 2
    n_sm = torch.cuda.get_device_properties(dev).multi_processor_count
    if dominant == "allocate":
        peak = n_sm * 128 * sm_mhz * 1e6 / 1e12         # fp32 lane ops, T/s
        a = dp_ops / (t_acold * 1e-3) / 1e12
        roof = {"kernel": "kvq_allocate (search rounds)", "bound": "alu", "achieved": a,
                "peak": peak, "unit": "T fp32 lane-op/s", "frac": a / peak,
                "traffic": SEARCH_DRAM_BYTES, "traffic_unit": TRAFFIC_NOTE,
                "work": "%d DP block-lambda evaluations x 680 triples x 2 ops" % (sum(rep["active"]) * 32),
                "peak_source": "%d SMs x 128 fp32 lanes x median SM clock" % n_sm}
    elif dominant == "stats":
        a = kern["stats_cold_GBps"]
        roof = {"kernel": "kvq_stats", "bound": "hbm", "achieved": a, "peak": hbm, "unit": "GB/s",
                "frac": a / hbm, "traffic": None, "peak_source": src}
    else:
        a = kern["quantize_cold_GBps"]
        roof = {"kernel": "kvq_quantize", "bound": "hbm", "achieved": a, "peak": hbm,
                "unit": "GB/s", "frac": a / hbm, "traffic": None, "peak_source": src}

    # kvq_stats 1; kvq_allocate: control init + the persistent search kernel; kvq_quantize 1
    launches_per_step = 1 + 2 + 1
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        gbs, dt, thr, desc = cpu_baseline(w, x_np, w.budgets[0])
        cpu = {"value": gbs, "unit": "GB/s", "cores": thr, "kind": "oracle", "sample": desc,
               "seconds": dt, "cpu_model": cpu_model()}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": tot_ms / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic",
            "config": step_config(world),
            "tokens_per_s": world * args.steps * w.T / (tot_ms * 1e-3),
            "lambda": float(buf.lam.item()), "rate_bits_per_entry": float(buf.totals[0].item()) / w.entries,
            "kernels": kern,
            "roofline": roof,
            "e2e": {"value": e2e_val, "unit": "GB/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h,
                    "how": "kvq_encode_host per step from pinned host memory (input copied in "
                           "4 pieces on 4 copy streams, codes / codebooks / k / totals copied "
                           "out), steps alternating over 2 streams, L2 flush inside each step"},
            "gpu_launches": launches_per_step * args.steps,
            "clocks": clk_summary,
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)
    if pg:
        pg.destroy_process_group()


if __name__ == "__main__":
    main()
