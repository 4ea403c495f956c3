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
