"""One-GPU PSD emulation (MineDraft pages, section 2) on the GPU: the
overlapped schedule gives the same results as the same phases run one after
the other, and each phase agrees with the oracle."""
import numpy as np
import pytest
import torch

import oracle
from draft_verification_row_gb300 import psd, workloads as W
from tests import parity as P

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
WL = "mixed-B256-K8-L8-V151936-bf16"


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _emu(seed=3):
    batch = W.make(WL, DEV, B=8, V=12011, seed=seed)
    return psd.PsdEmulator(batch, steps=4, seed=7), batch


def test_overlapped_equals_sequential():
    a, _ = _emu()
    b, _ = _emu()
    for s in range(3):
        a.step_overlapped(s)
        b.step_sequential(s)
    torch.cuda.synchronize()
    for h in range(2):
        ra, rb = a.results(h), b.results(h)
        assert ra["device_status"] == 0 and rb["device_status"] == 0
        for key in ("accept_len", "accept_draft", "out_token", "tokens"):
            assert torch.equal(ra[key], rb[key]), (h, key)


def test_draft_phase_samples_each_depth_row():
    emu, batch = _emu()
    emu.draft(1, 2, torch.cuda.current_stream())
    torch.cuda.synchronize()
    x = emu.halves[1]
    n = emu.B * emu.K
    for j in range(emu.L):
        rows = x.draft[:, :, j, :].reshape(n, x.draft.shape[-1]).cpu()
        ref = oracle.sample_rows(rows, 1, x.draft_u[2, j].cpu().double().numpy(), emu.T, V=emu.V)
        got = x.tokens[:, :, j].reshape(n, 1).cpu().numpy()
        diff = got != ref["tokens"]
        assert (ref["margin"][diff] < 1e-5).all() and diff.sum() <= 1, j


def test_verify_phase_matches_the_oracle():
    emu, batch = _emu(seed=5)
    emu.step_overlapped(0)   # half 1 drafts
    emu.step_overlapped(1)   # half 1 verifies its new drafts
    torch.cuda.synchronize()
    x = emu.halves[1]

    class Half:
        pass
    h = Half()
    h.target, h.draft, h.tokens, h.lengths = x.target, x.draft, x.tokens, x.lengths
    h.accept_u, h.sample_u, h.temperature, h.V, h.B = x.accept_u, x.sample_u, emu.T, emu.V, emu.B
    gpu = {k: getattr(x.out, k).cpu().numpy() for k in ("accept_len", "accept_draft", "out_token", "accept_prob",
                                                            "residual_mass", "device_status")}
    P.compare(gpu, P.oracle_run("multidraft", h), "psd verify")
