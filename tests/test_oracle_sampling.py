"""Pins of the oracle's draft-token sampler (oracle.sample_rows).

Draft tokens are drawn from the draft model's distribution softmax(d / T)
("SpecTr-GBV: Multi-Draft Block Verification Accelerating Speculative
Decoding", section 1).  The sampler is the inverse CDF the verification
oracle uses for its correction draws: the first token in index order whose
running sum exceeds u * S, else the last token of nonzero mass; T = 0 gives
the argmax, lowest index on ties.  These tests fix it against hand-derived
values, an independent numpy softmax and the verification oracle itself.
"""
import numpy as np
import pytest
import torch

import oracle


def _bf16_bits(a):
    return torch.as_tensor(np.asarray(a, np.float32)).to(torch.bfloat16).view(torch.int16).numpy()


def test_hand_derived_cdf():
    # P = (0.1, 0.2, 0.3, 0.4) at T = 1; CDF ends 0.1, 0.3, 0.6, 1.0
    lg = np.log(np.array([[0.1, 0.2, 0.3, 0.4]], np.float64)).astype(np.float32)
    u = np.array([[0.0, 0.05, 0.15, 0.35, 0.65, 0.999]])
    o = oracle.sample_rows(lg, u.shape[1], u, 1.0)
    assert o["rc"] == 0
    assert o["tokens"].tolist() == [[0, 0, 1, 2, 3, 3]]
    # T = 0.5 squares the probabilities: (1, 4, 9, 16) / 30; CDF ends
    # 1/30, 5/30, 14/30, 1
    u = np.array([[0.03, 0.034, 0.16, 0.17, 0.46, 0.47]])
    o = oracle.sample_rows(lg, u.shape[1], u, 0.5)
    assert o["tokens"].tolist() == [[0, 1, 1, 2, 2, 3]]


def test_strict_inequality_at_a_boundary():
    # four equal logits: CDF ends 0.25, 0.5, 0.75, 1.  A uniform exactly at a
    # boundary belongs to the next token (running sum must exceed u * S).
    lg = np.zeros((1, 4), np.float32)
    u = np.array([[0.25, 0.5, 0.75]])
    o = oracle.sample_rows(lg, 3, u, 1.0)
    assert o["tokens"].tolist() == [[1, 2, 3]]
    np.testing.assert_allclose(o["margin"], 0.0, atol=1e-15)


def test_masked_tokens_are_never_drawn():
    lg = np.array([[-np.inf, 0.0, -np.inf, 0.0, -np.inf]], np.float32)
    u = np.linspace(0.0, 0.999, 41)[None, :]
    o = oracle.sample_rows(lg, u.shape[1], u, 0.7)
    assert set(o["tokens"].ravel().tolist()) == {1, 3}
    assert (o["tokens"][0, :20] == 1).all() and (o["tokens"][0, 21:] == 3).all()


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("T", [0.3, 1.0, 2.5])
def test_grid_frequencies_match_an_independent_softmax(dtype, T):
    """On a uniform grid of N points the share of each token is its
    probability to within 1/N: pins the mapping against numpy's softmax."""
    rng = np.random.default_rng(7)
    V, N = 37, 20000
    rows = rng.normal(0, 2.0, (3, V)).astype(np.float32)
    rows[1, 5] = -np.inf
    if dtype == "bf16":
        bits = _bf16_bits(rows)
        vals = torch.as_tensor(bits).view(torch.bfloat16).float().numpy().astype(np.float64)
        lg = bits
    else:
        vals = rows.astype(np.float64)
        lg = rows
    grid = (np.arange(N) + 0.5) / N
    u = np.tile(grid, (3, 1))
    o = oracle.sample_rows(lg, N, u, T)
    assert o["rc"] == 0
    for r in range(3):
        z = vals[r] / T
        p = np.exp(z - np.max(z))
        p /= p.sum()
        share = np.bincount(o["tokens"][r], minlength=V) / N
        assert np.max(np.abs(share - p)) <= 1.0 / N + 1e-12


def test_zero_temperature_is_argmax_lowest_index():
    lg = np.array([[0.0, 3.0, 1.0, 3.0], [-1.0, -1.0, -1.0, -1.0]], np.float32)
    o = oracle.sample_rows(lg, 3, None, 0.0)
    assert o["tokens"].tolist() == [[1, 1, 1], [0, 0, 0]]


def test_invalid_rows_are_isolated():
    lg = np.zeros((4, 6), np.float32)
    lg[1, 2] = np.nan
    lg[2, 0] = np.inf
    lg[3, :] = -np.inf
    u = np.full((4, 2), 0.55)
    o = oracle.sample_rows(lg, 2, u, 1.0)
    assert o["row_status"].tolist() == [0, 4, 4, 4]
    assert o["tokens"][1:].ravel().tolist() == [-1] * 6
    assert o["tokens"][0].tolist() == [3, 3]  # six equal logits: CDF ends k/6, u = 0.55 -> index 3


def test_padding_columns_are_not_read():
    lg = np.full((2, 8), np.nan, np.float32)
    lg[:, :5] = np.array([0.0, 1.0, 2.0, 1.0, 0.0], np.float32)
    u = np.array([[0.1, 0.9], [0.5, 0.6]])
    o = oracle.sample_rows(lg, 2, u, 1.0, V=5)
    assert o["rc"] == 0 and (o["row_status"] == 0).all()
    assert ((o["tokens"] >= 0) & (o["tokens"] < 5)).all()


def test_agrees_with_the_bonus_draw_of_verification():
    """With L = 0 verification returns a token drawn from P_0 with
    sample_u[b][0][0]: the sampler must give the same token."""
    rng = np.random.default_rng(3)
    B, V = 12, 53
    tgt = rng.normal(0, 1.5, (B, 1, 1, V)).astype(np.float32)
    sample_u = rng.random((B, 1, 1)).astype(np.float32)
    prob = oracle.Problem(tgt, np.zeros((B, 1, 0, V), np.float32), np.zeros((B, 1, 0), np.int32), None,
                          np.zeros((B, 1, 0), np.float32), sample_u, 0.8)
    ref = oracle.verify("token", prob)
    o = oracle.sample_rows(tgt.reshape(B, V), 1, sample_u.reshape(B, 1).astype(np.float64), 0.8)
    assert o["tokens"][:, 0].tolist() == ref["out_token"].tolist()


def test_rejects_bad_arguments():
    lg = np.zeros((1, 4), np.float32)
    assert oracle.sample_rows(lg, 1, np.zeros((1, 1)), -1.0)["rc"] == 1
    assert oracle.sample_rows(lg, 1, np.zeros((1, 1)), float("inf"))["rc"] == 1
