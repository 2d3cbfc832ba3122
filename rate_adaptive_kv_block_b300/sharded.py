"""One global lambda over a tensor whose blocks are split across ranks
("Rate-adaptive KV-cache quantizer", "Mathematical statement": the blocks
are coupled only through lambda).

Each rank holds some of the blocks (any split: streams, layers, sequences)
and runs kvq_stats on them.  The 40-step bisection of kvq_allocate then runs
in rounds: every rank takes the round's lambdas from the shared search state
(kvq_search_probes), evaluates its own blocks there (kvq_rate_sums: the exact
DP, rates in fixed point), the 32 integer sums are all-reduced (the one
exchange; integer adds are exact, so the result does not depend on how the
blocks are split), and every rank advances the same state
(kvq_search_advance).  At the end each rank takes its blocks' choice at the
common lambda (kvq_allocate in subgradient mode with eta = 0).  The collective
goes through torch.distributed (NCCL on GPUs; gloo moves the sums through
host memory).  Without an initialised process group the same code runs on
one rank.
"""
import torch

from . import kvq


def _dist():
    import torch.distributed as dist
    return dist if dist.is_available() and dist.is_initialized() else None


def _all_reduce(t, op, group):
    """All-reduce of a small tensor; gloo takes it through host memory."""
    dist = _dist()
    if dist is None:
        return t
    backend = dist.get_backend(group)
    if backend == "gloo" and t.device.type != "cpu":
        c = t.cpu()
        dist.all_reduce(c, op=op, group=group)
        t.copy_(c)
        return t
    dist.all_reduce(t, op=op, group=group)
    return t


def search(hi0_local, budget_bits, evaluate, group=None, device="cpu"):
    """Drive the global search.  hi0_local: this rank's largest
    (c_max - c_min)^2; budget_bits: the total budget over all ranks;
    evaluate(lambdas) returns this rank's 32 fixed-point rate sums (int64
    tensor on `device`; entries past len(lambdas) are 0).  Returns (lambda,
    status, rounds), the same on every rank."""
    dist = _dist()
    h = torch.tensor([float(hi0_local)], dtype=torch.float64, device=device)
    if dist is not None:
        _all_reduce(h, dist.ReduceOp.MAX, group)
    state = kvq.SearchState(float(h.item()), budget_bits)
    while True:
        lam = state.probes()
        if not lam:
            break
        sums = evaluate(lam)
        if dist is not None:
            _all_reduce(sums, dist.ReduceOp.SUM, group)
        state.advance(sums.cpu().tolist())
    return state.result()


def allocate(stats, L: kvq.Layout, s: int, budget_bits: float, buf: kvq.Buffers, group=None,
             stream=None):
    """This rank's blocks (stats: their kvq_stats record, on the GPU) under
    the global lambda of every rank's blocks and the total budget
    budget_bits.  Writes buf's codebook, k, D_r, H_r, totals (this rank's
    sums), lam and status; returns (lambda, search status, rounds)."""
    dev = stats.device
    sums = torch.zeros(32, dtype=torch.int64, device=dev)

    def evaluate(lam):
        kvq.kvq_rate_sums(stats, L, s, lam, sums, stream=stream)
        return sums
    hi0 = kvq.kvq_stats_hi0(stats)
    lam, st, rounds = search(hi0, budget_bits, evaluate, group=group, device=dev)
    buf.lam.fill_(lam)
    kvq.kvq_allocate(stats, L, s, 0.0, kvq.KVQ_SUBGRADIENT, 0.0, buf.lam, buf.workspace,
                     buf.codebook, buf.k, buf.D_r, buf.H_r, buf.totals, buf.status, stream=stream)
    return lam, st, rounds
