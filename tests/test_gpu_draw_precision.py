"""How close the GPU's inverse-CDF draws come to the oracle's, over seeds the
rest of the suite does not use.

A draw takes the first token whose running sum of masses exceeds u times the
total ("SpecTr-GBV: Multi-Draft Block Verification Accelerating Speculative
Decoding", section 2, step 4, for the correction; section 1 for the draft
tokens).  The GPU forms the masses in fp32 and their running sums over
segments in double; the oracle works in fp64.  A draw can therefore come out
differently only where u lies within the fp32 error of the masses of an
interval's end: the property checked here is that every such flip has the
oracle's u within 2^-22 (two fp32 ulps of 1) of the chosen token's interval.
An accept test (u <= threshold) may flip only within 1e-5 of its threshold.

The flip rates are printed, not asserted: on vocabularies of 128K-152K tokens
a few draws in 10^4 land within fp32 resolution of an interval end (most of
them on tokens of probability below 1e-7), so any fp32 implementation flips
some of them.
"""
import numpy as np
import pytest
import torch

import draft_verification_row_gb300 as sdv
import oracle
from draft_verification_row_gb300 import workloads as W
from tests import parity as P

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
DRAW_BOUND = 2.0 ** -22  # two fp32 ulps of 1
ACCEPT_BOUND = 1e-5


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _path_margins(mode, batch, b):
    """The oracle's decisions for request b: the smallest margin among its
    inverse-CDF draws and among its accept tests."""
    sub = P.oracle_run(mode, batch, requests=[b])
    one = oracle.verify(mode, sub["prob"], trace_cap=4096)
    au = sub["prob"].accept_u.reshape(-1)
    su = sub["prob"].sample_u.reshape(-1)
    draw, acc = np.inf, np.inf
    for kind, idx, lo, hi in one["trace"]:
        if kind == 0:
            acc = min(acc, abs(float(au[idx]) - lo))
        else:
            draw = min(draw, float(su[idx]) - lo, hi - float(su[idx]))
    return draw, acc


@pytest.mark.parametrize("mode", ["block", "token"])
def test_verification_flips_lie_within_fp32_resolution(mode):
    name = "block-B128-K1-L5-V128256-bf16"
    flips = decisions = 0
    for seed in range(200, 206):
        batch = W.make(name, DEV, seed=seed)
        ref = P.oracle_run(mode, batch)
        got = P.gpu_run(mode, batch)
        decisions += int(np.maximum(ref["decisions"], 1).sum())
        for b in range(batch.B):
            same = (got["accept_len"][b] == ref["accept_len"][b] and got["accept_draft"][b] == ref["accept_draft"][b]
                    and got["out_token"][b] == ref["out_token"][b])
            if same:
                continue
            flips += 1
            draw, acc = _path_margins(mode, batch, b)
            assert draw < DRAW_BOUND or acc < ACCEPT_BOUND, (
                f"{name} seed {seed} {mode} request {b}: differs, but its smallest draw margin is {draw:.3g} "
                f"and its smallest accept margin {acc:.3g}")
        del batch
        torch.cuda.empty_cache()
    print(f"\n{name} {mode}, seeds 200-205: {flips} flips in {decisions} decisions")


def test_sampler_flips_lie_within_fp32_resolution():
    flips = draws = 0
    T = float(np.float32(0.7))
    for seed in range(200, 204):
        batch = W.make(W.HEADLINE, DEV, seed=seed, B=64)
        rows = batch.draft[:, :, 0, :].reshape(batch.B * batch.K, batch.stride).contiguous()
        V = batch.V
        del batch
        g = torch.Generator(device=DEV)
        g.manual_seed(seed)
        u = torch.rand((rows.shape[0], 4), generator=g, device=DEV)
        tokens, status = sdv.sample_rows(rows, 4, u, T, V=V)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        ref = oracle.sample_rows(rows.cpu(), 4, u.cpu(), T, V=V)
        bad = tokens.cpu().numpy() != ref["tokens"]
        draws += bad.size
        flips += int(bad.sum())
        if bad.any():
            worst = float(ref["margin"][bad].max())
            assert worst < DRAW_BOUND, f"seed {seed}: a draw differs {worst:.3g} from its interval end"
        del rows
        torch.cuda.empty_cache()
    print(f"\nsampler, 4 x 512 depth-0 draft rows of the mixed batch: {flips} flips in {draws} draws")


@pytest.mark.parametrize("T", [0.1, 1.0])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_sampler_flips_on_peaked_and_flat_rows(dtype, T):
    # rows of N(0, 9) logits: at T = 0.1 a few tokens hold nearly all the
    # mass, so any error in how a segment is rescaled to the row maximum
    # moves every later interval end by that much
    V, n = 32000, 1024
    g = torch.Generator(device=DEV)
    g.manual_seed(V)
    x = torch.randn((n, V), generator=g, device=DEV) * 3.0
    x = x.to(torch.bfloat16 if dtype == "bf16" else torch.float32)
    u = torch.rand((n, 4), generator=g, device=DEV)
    Tf = float(np.float32(T))
    tokens, status = sdv.sample_rows(x, 4, u, Tf, V=V)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref = oracle.sample_rows(x.cpu(), 4, u.cpu(), Tf, V=V)
    bad = tokens.cpu().numpy() != ref["tokens"]
    if bad.any():
        worst = float(ref["margin"][bad].max())
        assert worst < DRAW_BOUND, f"{dtype} T={T}: a draw differs {worst:.3g} from its interval end"
    print(f"\nrandom rows V={V} {dtype} T={T}: {int(bad.sum())} flips in {bad.size} draws")
