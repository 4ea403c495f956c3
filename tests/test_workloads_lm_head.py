"""The LM-head input generator (workloads.make_lm_head), on the CPU.

The generator builds the inputs the fused LM-head calls and the oracle both
take: hidden rows that depend only on a draft's prefix (drafts sharing a
prefix share its row), drafted tokens in range, seeded reproducibility, the
integer mode's value range, and NaN in exactly the rows no rule reads.
"""
import numpy as np
import torch

from draft_verification_row_gb300 import workloads as W

WL = W.LM_HEAD_HEADLINE


def _owner(tokens, b, k, j):
    """Lowest draft sharing draft k's first j tokens."""
    return min(k2 for k2 in range(tokens.shape[1]) if (tokens[b, k2, :j] == tokens[b, k, :j]).all())


def test_rows_follow_the_trie_and_tokens_are_in_range():
    b = W.make_lm_head(WL, "cpu", B=6, K=4, L=4, V=211, d=16)
    tok = b.tokens.numpy()
    lens = b.lengths.numpy()
    h = b.hidden.float().numpy()
    assert b.hidden.dtype == torch.bfloat16 and b.lm_head.shape == (211, 16)
    assert ((lens >= 1) & (lens <= 4)).all()
    for r in range(6):
        for k in range(4):
            assert ((tok[r, k, :lens[r]] >= 0) & (tok[r, k, :lens[r]] < 211)).all()
            for j in range(5):
                o = _owner(tok, r, k, j)
                np.testing.assert_array_equal(h[r, k, j], h[r, o, j])
    # drafts do share prefixes (the trie is not trivial) and do diverge
    shared = sum(_owner(tok, r, k, 1) != k for r in range(6) for k in range(4))
    assert 0 < shared < 6 * 4


def test_seeded_and_reproducible():
    a = W.make_lm_head(WL, "cpu", B=3, K=2, L=3, V=101, d=8, seed=7)
    b = W.make_lm_head(WL, "cpu", B=3, K=2, L=3, V=101, d=8, seed=7)
    c = W.make_lm_head(WL, "cpu", B=3, K=2, L=3, V=101, d=8, seed=8)
    for name in ("hidden", "lm_head", "tokens", "lengths"):
        assert torch.equal(getattr(a, name).view(-1).float(), getattr(b, name).view(-1).float()), name
    assert not torch.equal(a.hidden.float(), c.hidden.float())


def test_integer_mode_draws_small_integers():
    b = W.make_lm_head(WL, "cpu", B=2, K=2, L=2, V=50, d=8, integer=2)
    for t in (b.hidden, b.lm_head):
        v = t.float()
        assert torch.equal(v, v.round()) and v.abs().max() <= 2


def test_poison_marks_exactly_the_unread_rows():
    b = W.make_lm_head(WL, "cpu", B=5, K=3, L=3, V=97, d=8, lengths=[3, 1, 0, 2, 3], poison_unread=True)
    tok = b.tokens.numpy()
    nan = torch.isnan(b.hidden.float()).any(dim=-1).numpy()  # [B][K][L+1]
    for r, Lb in enumerate([3, 1, 0, 2, 3]):
        for k in range(3):
            for j in range(4):
                read = j <= Lb and _owner(tok, r, k, j) == k
                assert nan[r, k, j] == (not read), (r, k, j)
        assert (tok[r, :, Lb:] == -1).all()
