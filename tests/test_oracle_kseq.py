"""Pins of the oracle's K-SEQ mode (SpecTr's per-position multi-draft rule
with its search for the scaling factor rho; the SpecTr-GBV page names it,
sections 3-4, and the rule follows its published definition).

* Validity: the emitted stream followed by target sampling is distributed
  exactly as the target, checked by integrating the oracle over all drafts
  and uniforms of prefix-consistent toy models.  This holds for any rho
  with gamma(rho) <= rho, so it pins the acceptance rule and the residual
  whatever the search finds.
* K = 1: rho = 1 and the rule is token-level speculative sampling, equal
  to the oracle's token mode on the same inputs.
* The search: the rho it returns satisfies gamma(rho) <= rho, and no point
  a quarter-step below it on its last grid does (minimality up to the
  search's resolution).
* Planted mistakes in a copy of the oracle are caught by the validity pin.
"""
import os
import shutil
import subprocess
import tempfile
import ctypes

import numpy as np
import pytest

import oracle
from tests import toymodel as tm

TOL = 1e-12


@pytest.mark.parametrize("K,L,V,T", [(1, 3, 3, 1.0), (2, 2, 3, 1.0), (2, 3, 3, 0.7), (3, 2, 3, 1.0),
                                     (3, 2, 2, 0.5), (4, 2, 2, 1.0)])
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_stream_is_target_distributed(K, L, V, T, seed):
    sp, tp, P, Q = tm.exact("kseq", V, K, L, seed, T)
    assert abs(sp.sum() - 1.0) < TOL
    assert tm.completed_stream_error(sp, P, V, L) < TOL


def test_stream_property_with_peaked_draft():
    sp, tp, P, Q = tm.exact("kseq", 3, 3, 2, 5, 1.0, scale=3.0, noise=3.0)
    assert tm.completed_stream_error(sp, P, 3, 2) < TOL


def _random_problem(B, K, L, V, seed, T=0.9):
    rng = np.random.default_rng(seed)
    tgt = rng.normal(0, 2, (B, K, L + 1, V)).astype(np.float32)
    dft = (tgt[:, :, :L] + rng.normal(0, 1, (B, K, L, V))).astype(np.float32)
    tok = rng.integers(0, V, (B, K, L)).astype(np.int32)
    lengths = rng.integers(0, L + 1, B).astype(np.int32)
    return oracle.Problem(tgt, dft, tok, lengths, rng.random((B, K, L)), rng.random((B, K, L + 1)), T)


@pytest.mark.parametrize("seed", range(4))
def test_single_draft_is_token_level_sampling(seed):
    prob = _random_problem(6, 1, 4, 23, seed)
    a, b = oracle.verify("kseq", prob, residual_out=True), oracle.verify("token", prob, residual_out=True)
    for key in ("accept_len", "accept_draft", "out_token", "req_status"):
        np.testing.assert_array_equal(a[key], b[key])
    np.testing.assert_allclose(a["accept_prob"], b["accept_prob"], atol=1e-7)
    np.testing.assert_allclose(a["residual_mass"], b["residual_mass"], atol=1e-12)


def _kseq_quantities(P, Q, n, rho):
    beta = np.minimum(Q, P / rho).sum()
    gamma = (1 - (1 - beta) ** n) / beta if beta > 0 else n
    return beta, gamma


@pytest.mark.parametrize("seed", range(6))
def test_search_finds_a_valid_and_near_minimal_rho(seed):
    """Re-run the search's arithmetic from the accept probabilities the
    oracle reports: a = min(1, P(y) / (rho Q(y))) gives rho back whenever
    a < 1; that rho must satisfy gamma <= rho, and rho minus the last
    grid's quarter-step must not (unless rho = 1)."""
    rng = np.random.default_rng(100 + seed)
    V, K = 40, 4
    lt = rng.normal(0, 1.5, V)
    ld = lt + rng.normal(0, 1.0, V)
    P = np.exp(lt - lt.max()); P /= P.sum()
    Q = np.exp(ld - ld.max()); Q /= Q.sum()
    ys = rng.choice(V, size=K, p=Q)
    tgt = np.tile(lt.astype(np.float32), (1, K, 2, 1))
    dft = np.tile(ld.astype(np.float32), (1, K, 1, 1))
    tok = ys.reshape(1, K, 1).astype(np.int32)
    tok[:] = ys.reshape(1, K, 1)
    prob = oracle.Problem(tgt, dft, tok, None, np.full((1, K, 1), 0.999), np.full((1, K, 2), 0.5), 1.0)
    # all K drafts share depth 0 (one node with K draws); P, Q in float64 from the stored float32 logits
    Pd = np.exp(lt.astype(np.float32).astype(np.float64) - lt.astype(np.float32).max()); Pd /= Pd.sum()
    Qd = np.exp(ld.astype(np.float32).astype(np.float64) - ld.astype(np.float32).max()); Qd /= Qd.sum()
    o = oracle.verify("kseq", prob)
    ap = o["accept_prob"][0, :, 0]
    cands = [Pd[y] / (a * Qd[y]) for y, a in zip(ys, ap) if a < 1.0]
    if not cands:
        return
    rho = cands[0]
    for c in cands:
        assert abs(c - rho) < 1e-6 * rho
    beta, gamma = _kseq_quantities(Pd, Qd, K, rho)
    assert gamma <= rho * (1 + 1e-9)
    step = (K - 1) / 4 ** 10
    if rho > 1 + 2 * step:
        b2, g2 = _kseq_quantities(Pd, Qd, K, rho - step)
        assert g2 > rho - step


# planted mistakes, caught by the validity pin (same machinery as the
# other modes' sensitivity test)
MUTANTS = {
    "residual_without_gamma": ("fmax(r->P[x] - r->gam[j][o] * fmin(r->Q[x], r->P[x] / r->rho[j][o]), 0.0)",
                               "fmax(r->P[x] - fmin(r->Q[x], r->P[x] / r->rho[j][o]), 0.0)"),
    "accept_without_rho": ("double den = hi * r->Q[y];", "double den = r->Q[y];"),
    "gamma_power_off_by_one": ("-expm1((double)n * log1p(-beta)) / beta", "-expm1((double)(n + 1) * log1p(-beta)) / beta"),
    "rho_from_lower_end": ("    r->rho[j][o] = hi;", "    r->rho[j][o] = lo;"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, monkeypatch):
    here = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle")
    src = open(os.path.join(here, "sdv_oracle.c")).read()
    old, new = MUTANTS[name]
    assert src.count(old) == 1, name
    with tempfile.TemporaryDirectory() as tmp:
        open(os.path.join(tmp, "sdv_oracle.c"), "w").write(src.replace(old, new))
        shutil.copy(os.path.join(here, "sdv_oracle.h"), tmp)
        shutil.copy(os.path.join(here, "exact.c"), tmp)
        so = os.path.join(tmp, "libm.so")
        subprocess.run(["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-o", so, os.path.join(tmp, "sdv_oracle.c"),
                        os.path.join(tmp, "exact.c"), "-lm"], check=True)
        mlib = ctypes.CDLL(so)
        mlib.sdvo_exact_streams.restype = ctypes.c_int
        monkeypatch.setattr(oracle, "_lib", mlib)
        errs = []
        for K, L, V, seed in [(2, 2, 3, 0), (3, 2, 3, 1), (2, 3, 2, 2), (4, 2, 2, 0)]:
            sp, tp, P, Q = tm.exact("kseq", V, K, L, seed, 1.0)
            errs.append(tm.completed_stream_error(sp, P, V, L))
        assert max(errs) > 1e-9, f"mutant {name} not caught"
