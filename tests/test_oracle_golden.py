"""The oracle against hand-derived worked examples (tests/golden/)."""
import numpy as np
import pytest

import oracle
from tests import goldens

CASES = goldens.cases()


@pytest.mark.parametrize("case", CASES, ids=[c["name"] for c in CASES])
def test_worked_example(case):
    prob = oracle.Problem(case["target"], case["draft"], case["tokens"], case["lengths"],
                          case["accept_u"], case["sample_u"], case["T"])
    o = oracle.verify(case["mode"], prob)
    e = case["expected"]
    assert o["rc"] == 0
    assert o["req_status"][0] == 0
    assert o["accept_len"][0] == e["accept_len"]
    assert o["accept_draft"][0] == e["accept_draft"]
    assert o["out_token"][0] == e["out_token"]
    np.testing.assert_allclose(o["accept_prob"][0], np.asarray(e["accept_prob"]), atol=1e-6)
    assert abs(o["residual_mass"][0] - e["residual_mass"]) < 1e-6
