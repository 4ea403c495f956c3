"""GPU draft-token sampling (sdv_sample_rows, through the C-ABI) against the
oracle's sampler.

Draft tokens are drawn from softmax(d / T) ("SpecTr-GBV: Multi-Draft Block
Verification Accelerating Speculative Decoding", section 1) by the inverse
CDF.  Tokens must equal the oracle's except at draws whose uniform lies
within 1e-5 of a CDF boundary (the oracle reports that margin); such flips
are counted and stay at one per comparison or under 1e-4 of the draws.
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
MARGIN = 1e-5


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _rows(n, V, dtype, seed, std=2.5, stride_pad=0):
    g = torch.Generator(device=DEV)
    g.manual_seed(seed)
    stride = (V + 7) // 8 * 8 + stride_pad
    x = torch.full((n, stride), float("nan"), device=DEV)
    x[:, :V] = torch.randn((n, V), generator=g, device=DEV) * std
    return x.to(torch.bfloat16 if dtype == "bf16" else torch.float32)


def _uniforms(n, s, seed):
    g = torch.Generator(device=DEV)
    g.manual_seed(seed)
    return torch.rand((n, s), generator=g, device=DEV)


def _check(logits, n_samples, u, T, V=None, what=""):
    T = float(np.float32(T))  # the value the library's float argument holds
    tokens, status = sdv.sample_rows(logits, n_samples, u, T, V=V)
    torch.cuda.synchronize()
    got = tokens.cpu().numpy()
    ref = oracle.sample_rows(logits.cpu(), n_samples, None if u is None else u.cpu(), T, V=V)
    assert ref["rc"] == 0
    diff = got != ref["tokens"]
    if diff.any():
        assert (ref["margin"][diff] < MARGIN).all(), (
            f"{what}: {int(diff.sum())} draws differ, margins {ref['margin'][diff][:5]}")
    assert diff.sum() <= max(1.0, 1e-4 * got.size), f"{what}: {int(diff.sum())} near-margin flips of {got.size}"
    expect_status = 4 if (ref["row_status"] != 0).any() else 0
    assert int(status.item()) == expect_status, what
    return got, ref


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("V", [1, 2, 7, 8, 9, 33, 1000, 4097])
def test_vocabulary_edges(dtype, V):
    logits = _rows(6, V, dtype, 11 + V)
    _check(logits, 5, _uniforms(6, 5, V), 0.7, V=V, what=f"V={V}/{dtype}")


# a segment is 256 units (2048 bf16 or 1024 fp32 logits), a step 16 segments
@pytest.mark.parametrize("V,dtype", [(2047, "bf16"), (2048, "bf16"), (2049, "bf16"), (32767, "bf16"),
                                     (32768, "bf16"), (32769, "bf16"), (151936, "bf16"), (16383, "f32"),
                                     (16384, "f32"), (16385, "f32"), (262144, "f32")])
def test_segment_and_step_boundaries(V, dtype):
    logits = _rows(4, V, dtype, 5)
    _check(logits, 8, _uniforms(4, 8, 6), 1.0, V=V, what=f"V={V}/{dtype}")


@pytest.mark.parametrize("T", [0.0, 0.1, 1.0, 2.5])
def test_temperatures(T):
    logits = _rows(8, 32000, "bf16", 21, std=3.0)
    u = None if T == 0.0 else _uniforms(8, 6, 22)
    got, ref = _check(logits, 6, u, T, V=32000, what=f"T={T}")
    if T == 0.0:
        am = logits.float().argmax(dim=1).cpu().numpy()
        assert (got == am[:, None]).all()


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_degenerate_and_masked_rows(dtype):
    V = 40007
    stride = (V + 7) // 8 * 8
    logits = torch.full((7, stride), float("nan"), device=DEV)
    for k in range(7):
        logits[k, :V] = P.pattern_row(k, V).to(DEV)
    logits = logits.to(torch.bfloat16 if dtype == "bf16" else torch.float32)
    for T in (0.0, 0.7):
        u = None if T == 0.0 else _uniforms(7, 16, 31)
        _check(logits, 16, u, T, V=V, what=f"degenerate/{dtype}/T={T}")


def test_invalid_rows_are_isolated():
    logits = _rows(5, 5000, "f32", 41)
    logits[1, 17] = float("nan")
    logits[2, 4000] = float("inf")
    logits[3, :5000] = float("-inf")
    tokens, status = sdv.sample_rows(logits, 3, _uniforms(5, 3, 42), 0.9, V=5000)
    torch.cuda.synchronize()
    t = tokens.cpu().numpy()
    assert (t[1:4] == -1).all() and (t[[0, 4]] >= 0).all()
    assert int(status.item()) == 4
    _check(logits, 3, _uniforms(5, 3, 42), 0.9, V=5000, what="invalid rows")


def test_many_draws_per_row_and_padding():
    logits = _rows(3, 7000, "bf16", 51, stride_pad=24)  # NaN padding past V must never be read
    _check(logits, 64, _uniforms(3, 64, 52), 0.8, V=7000, what="64 draws")


def test_deterministic():
    logits = _rows(16, 20011, "bf16", 61)
    u = _uniforms(16, 4, 62)
    a, _ = sdv.sample_rows(logits, 4, u, 0.6, V=20011)
    b, _ = sdv.sample_rows(logits, 4, u, 0.6, V=20011)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


def test_draws_follow_the_exact_law():
    """Chi-square of 200k GPU draws from one row against its exact
    probabilities (numpy softmax of the stored logits)."""
    from scipy.stats import chi2
    V, n_rows, S = 200, 3125, 64
    one = _rows(1, V, "f32", 71, std=1.5)
    logits = one.expand(n_rows, -1).contiguous()
    u = _uniforms(n_rows, S, 72)
    tokens, _ = sdv.sample_rows(logits, S, u, 1.3, V=V)
    torch.cuda.synchronize()
    counts = np.bincount(tokens.cpu().numpy().ravel(), minlength=V).astype(np.float64)
    z = one[0, :V].double().cpu().numpy() / 1.3
    p = np.exp(z - z.max())
    p /= p.sum()
    expected = p * counts.sum()
    keep = expected >= 5
    stat = np.sum((counts[keep] - expected[keep]) ** 2 / expected[keep])
    pval = chi2.sf(stat, keep.sum() - 1)
    assert pval > 1e-6, f"chi-square p = {pval:.3g}"


def test_full_size_draft_rows():
    """The mixed batch's depth-0 draft rows: 2048 rows of 151936 bf16 logits,
    one draw each (the oracle checks every row)."""
    batch = W.make(W.HEADLINE, DEV)
    rows = batch.draft[:, :, 0, :].reshape(batch.B * batch.K, batch.stride).contiguous()
    u = _uniforms(rows.shape[0], 1, 81)
    _check(rows, 1, u, batch.temperature, V=batch.V, what="full size")


def test_rejects_bad_arguments():
    logits = _rows(2, 100, "f32", 91)
    u = _uniforms(2, 65, 92)
    with pytest.raises(sdv.SDVError):
        sdv.sample_rows(logits, 65, u, 1.0, V=100)  # more than SDV_MAX_SAMPLES draws
    with pytest.raises(sdv.SDVError):
        sdv.sample_rows(logits, 1, None, 1.0, V=100)  # uniforms are needed for T > 0
    with pytest.raises(sdv.SDVError):
        sdv.sample_rows(logits, 1, _uniforms(2, 1, 93), -0.5, V=100)
