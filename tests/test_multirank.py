"""bench.py's multi-GPU path on CPU: two gloo ranks.

Requests are independent, so the path shards by request with no collective
on the data path.  Each rank verifies its own batch (weak scaling); the step
time is the maximum over ranks, and the positions are summed.  These tests
run bench.py's own rank plumbing on two CPU processes with the gloo
backend: process-group setup, barrier, max/sum reductions, per-rank seeds,
and the reference arm's rank-0-only rule.
"""
import os
import socket
import types

import torch
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    from draft_verification_row_gb300 import workloads as W
    w, r, _ = bench.dist_setup()
    try:
        mx = bench.max_over_ranks(1.5 * (r + 1), w)
        sm = bench.sum_over_ranks(float(10 + r), w)
        bench.barrier(w)
        seed = bench.rank_seed(W.HEADLINE, r)
        batch = W.make(W.HEADLINE, "cpu", seed=seed, B=3, K=2, L=2, V=64)
        pos = batch.positions
        tot = bench.sum_over_ranks(pos, w)
        # the reference arm runs on rank 0 only: other ranks return at once
        args = types.SimpleNamespace(workload=None, B=3, cpu_requests=4, warmup=0, steps=1, mode="token")
        ref_ran = None
        if r != 0:
            ref_ran = bench.run_reference(args, w, r)
        q.put((r, w, mx, sm, seed, pos, tot, int(batch.tokens.sum().item()), ref_ran))
    finally:
        torch.distributed.destroy_process_group()


def test_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    try:
        res = sorted(q.get(timeout=180) for _ in range(2))
    finally:
        for p in procs:
            p.join(timeout=60)
    assert [p.exitcode for p in procs] == [0, 0]
    (r0, w0, mx0, sm0, s0, p0, t0, k0, _), (r1, w1, mx1, sm1, s1, p1, t1, k1, ref1) = res
    assert (r0, r1) == (0, 1) and w0 == w1 == 2
    assert mx0 == mx1 == 3.0          # the step time is the slowest rank's
    assert sm0 == sm1 == 21.0         # whole-job sums
    assert s0 != s1 and k0 != k1      # each rank has its own requests
    assert t0 == t1 == p0 + p1        # positions of the whole job
    assert ref1 is None               # no reference work off rank 0
