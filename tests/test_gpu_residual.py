"""residual_out: the normalised distribution each request's correction (or
bonus) token was drawn from (the end node's residual after the target
adjustment, "SpecTr-GBV: Multi-Draft Block Verification Accelerating
Speculative Decoding", section 2, steps 4-5), compared element by element
with the oracle's fp64 row within 1e-5 (sdv_verify_residual, through the
C-ABI; needs a GB300)."""
import numpy as np
import pytest
import torch

from draft_verification_row_gb300 import workloads as W
from tests import parity as P

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _end_holds_dominant_token(batch, gpu, b):
    """Does request b's end node (an inner node) have a shared dominant
    token x*: the unique maximum of its target row equal to the unique
    maximum of its draft row?"""
    j, k = int(gpu["accept_len"][b]), int(gpu["accept_draft"][b])
    Lb = int(batch.lengths[b])
    if j >= Lb:
        return False
    t = batch.target[b, k, j, :batch.V].float().cpu().numpy()
    d = batch.draft[b, k, j, :batch.V].float().cpu().numpy()
    it, idr = int(t.argmax()), int(d.argmax())
    return it == idr and (t == t[it]).sum() == 1 and (d == d[idr]).sum() == 1


def _check(mode, batch, requests=None, what="", **kw):
    gpu = P.gpu_run(mode, batch, residual_out=True, **kw)
    ref = P.oracle_run(mode, batch, requests, residual_out=True)
    P.compare(gpu, ref, what)
    worst, n = P.compare_residual_rows(gpu, ref, what)
    assert n > 0
    # every valid row sums to one
    for b in ref["requests"]:
        if int(gpu["out_token"][b]) >= 0:
            assert abs(float(gpu["residual_out"][b].astype(np.float64).sum()) - 1.0) < 1e-4
    return gpu, ref, worst


@pytest.mark.parametrize("mode", ["token", "block", "multidraft", "greedy", "kseq"])
def test_token_workload_all_rules(mode):
    """The token workload at full size (B=4, K=1, L=4, V=1024, fp32, T=1)."""
    _check(mode, W.make("token-B4-K1-L4-V1024-f32", DEV), what=f"c1/{mode}")


@pytest.mark.parametrize("T", [0.1, 0.4, 0.7])
@pytest.mark.parametrize("mode,ap", [("multidraft", True), ("multidraft", False), ("token", True)])
def test_multidraft_workload_every_temperature(mode, ap, T):
    """The multi-draft workload at full size (B=32, K=4, L=4, V=32000, fp32)
    at each of its temperatures, every request; among the end nodes some
    hold a shared dominant token x*, whose residual the node kernel carries
    in closed form."""
    batch = W.make("multidraft-B32-K4-L4-V32000-f32", DEV, temperature=T)
    gpu, ref, worst = _check(mode, batch, what=f"c4/{mode}/T={T}", accept_prob=ap)
    if mode == "multidraft":
        assert any(_end_holds_dominant_token(batch, gpu, b) for b in range(batch.B))


def test_mixed_batch_sample():
    """The mixed batch at full size (the bench's launch configuration),
    SpecTr-GBV and token-level, on a sample of requests that includes end
    nodes holding x*."""
    batch = W.make(W.HEADLINE, DEV)
    sample = [0, 1, 2, 3, 37, 64, 101, 128, 190, 200, 233, 255]
    for mode in ("multidraft", "token"):
        gpu = P.gpu_run(mode, batch, residual_out=True)
        xs = [b for b in range(batch.B) if _end_holds_dominant_token(batch, gpu, b)]
        req = sorted(set(sample + xs[:4]))
        ref = P.oracle_run(mode, batch, req, residual_out=True)
        P.compare(gpu, ref, f"c5/{mode}", workload=W.HEADLINE)
        worst, n = P.compare_residual_rows(gpu, ref, f"c5/{mode}")
        assert n >= len(req) - 2
        if mode == "multidraft":
            assert xs, "no end node of the mixed batch holds x*"


@pytest.mark.parametrize("mode", ["token", "multidraft", "greedy", "kseq"])
def test_invalid_requests_get_zero_rows_and_leaves_their_bonus_row(mode):
    """Invalid requests get rows of zeros; requests that accept everything
    end at a leaf, whose row is P (the bonus draw); the rest are unchanged
    against a call without residual_out."""
    batch = W.make("multidraft-B32-K4-L4-V32000-f32", DEV, B=8, K=3, L=3, V=1999, temperature=0.7)
    batch.accept_u[:3] = 0.0
    batch.target[4, 0, 0, 5] = float("nan")
    batch.tokens[5, 1, 0] = batch.V
    plain = P.gpu_run(mode, batch)
    gpu, ref, worst = _check(mode, batch, what=f"invalid/{mode}")
    for key in ("accept_len", "accept_draft", "out_token", "accept_prob", "residual_mass", "device_status"):
        np.testing.assert_array_equal(plain[key], gpu[key], err_msg=key)
    assert not gpu["residual_out"][4].any() and not gpu["residual_out"][5].any()


@pytest.mark.parametrize("V,dtype", [(1, "f32"), (7, "bf16"), (8193, "bf16"), (4097, "f32")])
def test_vocabulary_edges(V, dtype):
    batch = W.make("mixed-B256-K8-L8-V151936-bf16", DEV, B=4, K=3, L=3, V=V, dtype=dtype, temperature=0.9)
    for mode in ("token", "multidraft", "kseq"):
        _check(mode, batch, what=f"V={V}/{dtype}/{mode}")
