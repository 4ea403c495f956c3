"""The oracle across host cores (oracle.pool) gives the single-process
oracle's outputs: requests are independent, so splitting a batch into
per-process shares changes nothing."""
import numpy as np
import pytest

import oracle
from oracle import pool
from draft_verification_row_gb300 import workloads as W


def _arrays(batch):
    def np_(t):
        import torch
        t = t.cpu()
        return (t.view(torch.int16) if t.dtype == torch.bfloat16 else t).numpy()
    return {k: np_(getattr(batch, k)) for k in ("target", "draft", "tokens", "lengths", "accept_u", "sample_u")}


@pytest.mark.parametrize("mode,procs", [("multidraft", 3), ("token", 2), ("greedy", 4)])
def test_all_cores_matches_one_process(mode, procs):
    batch = W.make("mixed-B256-K8-L8-V151936-bf16", "cpu", B=7, K=3, L=3, V=503)
    ref = oracle.verify(mode, oracle.Problem(batch.target, batch.draft, batch.tokens, batch.lengths,
                                             batch.accept_u, batch.sample_u, batch.temperature, V=batch.V))
    out, dt, used = pool.verify_all_cores(_arrays(batch), mode, batch.temperature, batch.V, procs=procs)
    assert used == procs and dt > 0
    for k in ("accept_len", "accept_draft", "out_token"):
        np.testing.assert_array_equal(out[k], ref[k], err_msg=k)


def test_more_processes_than_requests():
    batch = W.make("mixed-B256-K8-L8-V151936-bf16", "cpu", B=2, K=2, L=2, V=101)
    out, dt, used = pool.verify_all_cores(_arrays(batch), "multidraft", batch.temperature, batch.V, procs=8)
    assert used == 2 and out["accept_len"].shape == (2,)


def test_refuses_when_shared_memory_is_too_small(monkeypatch):
    # a tmpfs written past its size would kill the process: the pool checks
    # the room first and raises instead
    import os

    class Small:
        f_bavail, f_frsize = 1024, 4096  # 4 MiB free

    monkeypatch.setattr(os, "statvfs", lambda path: Small())
    batch = W.make("mixed-B256-K8-L8-V151936-bf16", "cpu", B=2, K=2, L=2, V=101)
    with pytest.raises(RuntimeError, match="/dev/shm"):
        pool.verify_all_cores(_arrays(batch), "token", batch.temperature, batch.V, procs=2)


@pytest.mark.parametrize("mode", ["multidraft", "token", "greedy", "kseq"])
def test_threads_match_one_call(mode):
    """verify_threads splits the requests over host threads: every output,
    floats and residual rows included, equals one call's, and its decision
    counts are those of the trace."""
    batch = W.make("mixed-B256-K8-L8-V151936-bf16", "cpu", B=9, K=3, L=3, V=301)
    prob = oracle.Problem(batch.target, batch.draft, batch.tokens, batch.lengths, batch.accept_u,
                          batch.sample_u, batch.temperature, V=batch.V)
    ref = oracle.verify(mode, prob, residual_out=True, trace_cap=1 << 16)
    out = oracle.verify_threads(mode, prob, threads=4, residual_out=True)
    for k in ("accept_len", "accept_draft", "out_token", "accept_prob", "residual_mass", "margin", "req_status",
              "residual_out"):
        np.testing.assert_array_equal(out[k], ref[k], err_msg=k)
    assert int(out["decisions"].sum()) == len(ref["trace"])
    dec, near = oracle.trace_counts(prob, ref["trace"])
    np.testing.assert_array_equal(out["decisions"], dec)
    np.testing.assert_array_equal(out["near_margin"], near)
    if mode != "greedy":
        assert (dec >= 1).all()


def test_trace_counts_margins():
    """A decision is near its threshold when |u - threshold| < 1e-5 (an
    accept test) or u lies within 1e-5 of its CDF interval's ends (a draw)."""
    class Pb:
        B, K, L = 2, 1, 2
        accept_u = np.array([[[0.5, 0.3]], [[0.1, 0.2]]])
        sample_u = np.array([[[0.7, 0.1, 0.2]], [[0.4, 0.5, 0.6]]])
    trace = [(0, 0, 0.500005, 0.500005), (0, 1, 0.9, 0.9), (1, 2, 0.1, 0.3),
             (0, 2, 0.1, 0.1), (1, 4, 0.499995, 0.7)]
    dec, near = oracle.trace_counts(Pb, trace)
    assert dec.tolist() == [3, 2]
    assert near.tolist() == [1, 2]
