"""The GPU-versus-oracle comparison rules themselves, on the CPU (no GPU):
the per-workload ledger of near-margin mismatches, and the K-SEQ search
ends that fp32 rounding can reach (tests/parity.py)."""
import numpy as np
import pytest

import oracle
from draft_verification_row_gb300 import workloads as W
from tests import parity as P


def _fake_gpu(ref):
    g = {k: ref[k].copy() for k in ("accept_len", "accept_draft", "out_token", "accept_prob")}
    g["residual_mass"] = ref["residual_mass"].astype(np.float32)
    g["device_status"] = np.array([int(np.bitwise_or.reduce(ref["req_status"]))], np.int32)
    return g


def _multi_draw_nodes(prob):
    for i in range(prob.B):
        tok = prob.tokens[i]
        for j in range(int(prob.lengths[i])):
            groups = {}
            for k in range(prob.K):
                o = min(k2 for k2 in range(prob.K) if (tok[k2, :j] == tok[k, :j]).all())
                groups.setdefault(o, []).append(k)
            for o, ks in groups.items():
                if len(ks) > 1:
                    yield i, j, o, ks


@pytest.mark.parametrize("T", [0.1, 0.7])
def test_kseq_search_ends_hold_the_oracles_rho(T):
    """The oracle's own acceptance probabilities follow from one of the
    search ends kseq_reachable lists, at every node with several draws; a
    rho that no search end is (here n, the top of the range, whenever the
    search stops below it) is refused."""
    batch = W.make("multidraft-B32-K4-L4-V32000-f32", "cpu", B=6, V=2003, temperature=T)
    ref = P.oracle_run("kseq", batch)
    prob = ref["prob"]
    checked = refused = 0
    for i, j, o, ks in _multi_draw_nodes(prob):
        a_ref = [float(ref["accept_prob"][i, k, j]) for k in ks]
        P._kseq_node_ok(prob, i, j, ks, a_ref, "oracle")
        checked += 1
        Pr = P._softmax64(prob.target[i, o, j, :prob.V], T)
        Qr = P._softmax64(prob.draft[i, o, j, :prob.V], T)
        n = len(ks)
        ends = P.kseq_reachable(Pr, Qr, n)
        ys = [int(prob.tokens[i, k, j]) for k in ks]
        a_top = [min(1.0, Pr[y] / (n * Qr[y])) for y in ys]
        if max(ends) < n * (1 - 1e-3) and max(abs(x - y) for x, y in zip(a_top, a_ref)) > 10 * P.TOL:
            with pytest.raises(AssertionError):
                P._kseq_node_ok(prob, i, j, ks, a_top, "planted")
            refused += 1
    assert checked >= 5 and refused >= 1


def test_kseq_reachable_without_ambiguity_is_the_search():
    """With eps = 0 no test goes both ways: the one end is the plain fp64
    search (rho = 1 when gamma(1) <= 1; n = 1 always gives rho = 1)."""
    rng = np.random.default_rng(3)
    P_ = rng.random(50); P_ /= P_.sum()
    Q_ = rng.random(50); Q_ /= Q_.sum()
    assert P.kseq_reachable(P_, Q_, 1, eps=0.0) == [1.0]
    ends = P.kseq_reachable(P_, Q_, 4, eps=0.0)
    assert len(ends) == 1 and 1.0 <= ends[0] <= 4.0
    g = P.kseq_gamma(np.minimum(Q_, P_ / ends[0]).sum(), 4)
    assert g <= ends[0]


def test_ledger_counts_and_bar():
    batch = W.make("multidraft-B32-K4-L4-V32000-f32", "cpu", B=5, K=3, L=3, V=501, temperature=0.7)
    ref = P.oracle_run("multidraft", batch)
    P.LEDGER.pop("rules-test", None)
    assert P.compare(_fake_gpu(ref), ref, "same", workload="rules-test") == 0
    e = P.LEDGER["rules-test"]
    assert e["requests"] == 5 and e["decisions"] == int(np.maximum(ref["decisions"], 1).sum())
    assert e["decisions"] >= 5 and e["mismatches"] == 0
    assert "rules-test" not in P.ledger_violations()
    e["mismatches"] = 1  # one mismatch against fewer than 10000 decisions is over the bar
    assert "rules-test" in P.ledger_violations()
    P.LEDGER.pop("rules-test")


def test_a_mismatch_far_from_every_threshold_fails():
    batch = W.make("token-B4-K1-L4-V1024-f32", "cpu", B=4)
    ref = P.oracle_run("token", batch)
    g = _fake_gpu(ref)
    b = int(np.argmax(ref["margin"]))
    assert ref["margin"][b] >= P.MARGIN
    g["out_token"][b] = (g["out_token"][b] + 1) % batch.V
    with pytest.raises(AssertionError, match="margin"):
        P.compare(g, ref, "planted", workload="rules-test-2")
    P.LEDGER.pop("rules-test-2", None)
