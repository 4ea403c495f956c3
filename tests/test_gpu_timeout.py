"""Bounded device waits run out without a fault (needs a GB300).

Every wait in the library gives up after a limit and reports
SDV_DEV_TIMEOUT instead of hanging.  The test hook
sdv_testing_verify_without_roots (include/sdv_testing.h) takes the trie
roots out of the node kernel's work list, so that the nodes below them wait
for weights nothing writes, and each request's decision waits for node
records that never come: a flag that nothing sets.  With the limit cut to
20 ms the call must come back with every request marked invalid, and the
next ordinary call on the same stream must be correct."""
import ctypes

import numpy as np
import pytest
import torch

from draft_verification_row_gb300 import binding
from draft_verification_row_gb300 import workloads as W
from tests import parity as P

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    return binding.lib()


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


@pytest.mark.parametrize("mode,name,kw", [
    ("multidraft", "multidraft-B32-K4-L4-V32000-f32", dict(B=6, V=3001)),
    ("block", "block-B128-K1-L5-V128256-bf16", dict(B=5, V=4099)),
])
def test_waits_run_out_and_the_next_call_is_correct(lib, mode, name, kw):
    batch = W.make(name, DEV, temperature=0.7, **kw)
    out = binding.Outputs(mode, batch.B, batch.K, batch.L, batch.V, torch.device(DEV))
    stream = torch.cuda.current_stream()
    assert lib.sdv_testing_set_wait_limit(20_000_000) == 0
    try:
        rc = lib.sdv_testing_verify_without_roots(
            binding.MODES[mode], batch.B, batch.K, batch.L, batch.V, batch.stride, binding._dtype_code(batch.target),
            batch.temperature, _p(batch.target), _p(batch.draft), _p(batch.tokens), _p(batch.lengths),
            _p(batch.accept_u), _p(batch.sample_u), _p(out.accept_len), _p(out.accept_draft), _p(out.out_token),
            _p(out.accept_prob), _p(out.residual_mass), _p(out.device_status), _p(out.workspace),
            out.workspace.numel(), ctypes.c_void_p(stream.cuda_stream))
        torch.cuda.synchronize()
    finally:
        assert lib.sdv_testing_set_wait_limit(0) == 0
    assert rc == 0
    st = int(out.device_status.item())
    assert st & binding.DEV_TIMEOUT, st
    lens = batch.lengths.cpu().numpy()
    assert (lens >= 1).all()
    assert (out.accept_len.cpu().numpy() == 0).all()
    assert (out.accept_draft.cpu().numpy() == 0).all()
    assert (out.out_token.cpu().numpy() == -1).all()
    assert not out.accept_prob.cpu().numpy().any() and not out.residual_mass.cpu().numpy().any()
    # the same stream, the default limit again: an ordinary call is correct
    P.compare(P.gpu_run(mode, batch), P.oracle_run(mode, batch), f"after timeout/{mode}")


def test_only_block_rules_take_the_hook(lib):
    args = [0, 1, 0, 1, 8, 0, 1.0] + [None] * 13 + [0, None]
    assert lib.sdv_testing_verify_without_roots(binding.MODES["token"], *args) == 1
