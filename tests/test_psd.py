"""Host logic of the one-GPU PSD emulation (MineDraft pages, section 2:
two batches alternate drafting and verification)."""
import pytest

from draft_verification_row_gb300 import psd


def test_roles_alternate():
    # batch 0 verifies first; every step swaps the two roles
    assert [psd.roles(s) for s in range(4)] == [(0, 1), (1, 0), (0, 1), (1, 0)]


@pytest.mark.parametrize("d,v,seq,par,want", [
    (1.0, 3.0, 4.0, 4.0, 0.0),    # no overlap at all
    (1.0, 3.0, 4.0, 3.0, 1.0),    # the shorter phase fully hidden
    (2.0, 2.0, 4.0, 3.0, 0.5),
    (0.0, 2.0, 2.0, 2.0, 0.0),    # nothing to hide
])
def test_hidden_fraction(d, v, seq, par, want):
    assert psd.hidden_fraction(d, v, seq, par) == pytest.approx(want)
