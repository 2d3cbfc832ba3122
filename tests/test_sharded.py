"""One global lambda over blocks split across ranks (sharded search).

CPU, world size 2 (gloo, spawned processes): each rank holds half of the
streams of one tensor and evaluates its blocks with an oracle-based evaluator
(the oracle's per-block rates at binary32 lambda, in the library's fixed
point); the library's host search control and the all-reduce of the 32
integer sums are the product path.  Two half-tensors must give the lambda of
one rank holding every block bit for bit, the same codebooks, and the oracle's
40-step bisection lambda within 1e-4.

GPU (world size 1, marked gpu): sharded.allocate with the library's rate sums
gives kvq_allocate's lambda within 1e-4 (the same bisection and rate sums,
evaluated at other probes) and the same codebooks on 99.9 % of the blocks.
"""
import os
import socket

import numpy as np
import pytest
import torch

import oracle
from rate_adaptive_kv_block_b300 import kvq, sharded, synth

W = synth.workload("llama3_8b_layer", T=128)   # 16 streams: 64 blocks of 4096
S_BITS = 2.5


def _x():
    return synth.make_numpy(W, seed=9)


def _evaluator(x):
    """This rank's fixed-point rate sums at binary32 lambda (the oracle's
    per-block rates, each rounded once to 2^-20 bit)."""
    d = 32 * W.G

    def evaluate(lams):
        out = torch.zeros(32, dtype=torch.int64)
        for p, lam in enumerate(lams):
            at = oracle.allocate_at(x, W.G, W.s, float(np.float32(lam)))
            out[p] = int(np.sum(np.rint(at["H_r"] * d * 1048576.0).astype(np.int64)))
        return out
    return evaluate


def _hi0(x):
    st = oracle.stats(x, W.G)
    return max((c[m - 1] - c[0]) ** 2 for c, m in zip(st["cand"], st["mprime"]))


def _rank_main(rank, world, port, x_all, out_path):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    half = x_all.shape[0] // world
    x = np.ascontiguousarray(x_all[rank * half:(rank + 1) * half])
    lam, st, rounds = sharded.search(_hi0(x), S_BITS * x_all.size, _evaluator(x))
    at = oracle.allocate_at(x, W.G, W.s, float(np.float32(lam)))
    np.savez(out_path % rank, lam=lam, st=st, rounds=rounds, cb=at["codebook"], k=at["k"])
    dist.barrier()
    dist.destroy_process_group()


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def test_two_ranks_give_the_single_rank_lambda(tmp_path):
    x = _x()
    lam1, st1, rounds1 = sharded.search(_hi0(x), S_BITS * x.size, _evaluator(x))
    assert st1 == kvq.KVQ_OK and rounds1 > 1
    ref = oracle.allocate_bisect(x, W.G, W.s, S_BITS * x.size)
    assert abs(lam1 - ref["lambda"]) <= 1e-4 * ref["lambda"]
    out = str(tmp_path / "rank%d.npz")
    ctx = torch.multiprocessing.get_context("spawn")
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, x, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=600)
        assert p.exitcode == 0
    at1 = oracle.allocate_at(x, W.G, W.s, float(np.float32(lam1)))
    half = x.shape[0] // 2
    nbh = half * (W.T // 32)
    for r in range(2):
        z = np.load(out % r)
        assert float(z["lam"]) == lam1 and int(z["st"]) == st1 and int(z["rounds"]) == rounds1
        assert np.array_equal(z["cb"], at1["codebook"][r * nbh:(r + 1) * nbh])
        assert np.array_equal(z["k"], at1["k"][r * nbh:(r + 1) * nbh])


def test_search_state_host_api():
    st = kvq.SearchState(4.0, 100.0)
    lam = st.probes()
    assert len(lam) == 32 and lam[0] == 0.0 and lam[1] == 4.0
    with pytest.raises(kvq.KvqError):
        st.result()                                  # not done yet
    # every probe feasible: lambda = 0 after one round
    st.advance([0] * 32)
    assert st.probes() == []
    assert st.result()[0] == 0.0 and st.result()[1] == kvq.KVQ_OK


@pytest.mark.gpu
def test_sharded_allocate_on_one_gpu_equals_kvq_allocate():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    w = synth.workload("llama3_8b_layer", T=2048)
    xd = synth.make_torch(w, seed=12)
    L = kvq.Layout(w.S, w.T, w.D, w.G)
    B = w.budgets[0] * w.entries
    ref = kvq.quantize(xd, L, B, w.s)
    buf = kvq.Buffers(L, w.s)
    kvq.kvq_stats(xd, L, buf.stats, buf.status_stats)
    lam, st, rounds = sharded.allocate(buf.stats, L, w.s, B, buf)
    torch.cuda.synchronize()
    assert st == kvq.KVQ_OK and int(buf.status.item()) == 0
    # the same bisection and rate sums at other probes: the window each search
    # infers from depends on its probes wherever the binary32 DP's rate sum is
    # not monotone near a switch, so the two agree within the parity rule
    # (each is within 1e-4 of the oracle's)
    assert abs(lam - float(ref.lam.item())) <= 1e-4 * float(ref.lam.item())
    assert float(buf.totals[0].item()) <= B
    same = (buf.codebook == ref.codebook).all(dim=1) & (buf.k == ref.k)
    assert float(same.float().mean().item()) >= 0.999
