"""Pins of the CPU oracle against what the mathematics fixes (no GPU).

* Validity: for every sampling mode, the emitted stream followed by target
  sampling is distributed exactly as the target (the distribution-preserving
  guarantee stated on the SpecTr-GBV page, section 3 "theoretical
  guarantees", and the defining property of speculative sampling).  Checked
  exactly by integrating the oracle over all drafts and uniforms of
  prefix-consistent toy models.
* Acceptance invariants from the SpecTr-GBV page (section 2 "theoretical
  basis": optimality and monotonicity in K; section 4 ablation over K):
  E[tau] of SpecTr-GBV is non-decreasing in K, at least the per-position
  multi-draft rule's, and equals greedy block verification at K = 1.
* Closed forms: token-level acceptance tails, the block-verification tail
  identity P(tau >= i) = E[p_i], the residual correction law.
"""
import itertools
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

STREAM_CASES = [
    # mode, K, L, V, T
    ("token", 1, 3, 3, 1.0),
    ("token", 2, 2, 3, 1.0),
    ("token", 3, 2, 3, 0.5),
    ("token", 4, 2, 2, 1.0),
    ("block", 1, 3, 3, 1.0),
    ("block", 1, 3, 4, 0.7),
    ("multidraft", 1, 3, 3, 1.0),
    ("multidraft", 2, 2, 4, 1.0),
    ("multidraft", 2, 3, 3, 0.7),
    ("multidraft", 3, 2, 3, 1.0),
    ("multidraft", 4, 2, 2, 1.0),
    ("multidraft", 3, 3, 2, 0.4),
]


@pytest.mark.parametrize("mode,K,L,V,T", STREAM_CASES)
@pytest.mark.parametrize("seed", [0, 1])
def test_stream_is_target_distributed(mode, K, L, V, T, seed):
    sp, tp, P, Q = tm.exact(mode, V, K, L, seed, T)
    assert abs(tp.sum() - 1.0) < TOL
    assert abs(sp.sum() - 1.0) < TOL
    assert tm.completed_stream_error(sp, P, V, L) < TOL


@pytest.mark.parametrize("seed", [2, 3])
def test_stream_property_with_peaked_draft(seed):
    # a draft far from the target exercises long residual recursions
    sp, tp, P, Q = tm.exact("multidraft", 3, 3, 2, seed, 1.0, scale=3.0, noise=3.0)
    assert tm.completed_stream_error(sp, P, 3, 2) < TOL
    sp, tp, P, Q = tm.exact("token", 3, 3, 2, seed, 1.0, scale=3.0, noise=3.0)
    assert tm.completed_stream_error(sp, P, 3, 2) < TOL


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_multidraft_monotone_in_K_and_dominates(seed):
    V, L = 3, 2
    e_md, e_tok = [], []
    for K in (1, 2, 3, 4):
        _, tp, _, _ = tm.exact("multidraft", V, K, L, seed)
        e_md.append(tm.expected_tau(tp))
        _, tp, _, _ = tm.exact("token", V, K, L, seed)
        e_tok.append(tm.expected_tau(tp))
    for a, b in zip(e_md, e_md[1:]):
        assert b >= a - TOL, e_md
    # the optimal acceptance bound grows strictly with K on a generic model
    assert e_md[1] > e_md[0] + 1e-6, e_md
    for a, b in zip(e_md, e_tok):
        assert a >= b - TOL, (e_md, e_tok)
    _, tp, _, _ = tm.exact("block", V, 1, L, seed)
    assert abs(tm.expected_tau(tp) - e_md[0]) < TOL
    assert tm.expected_tau(tp) >= e_tok[0] - TOL


@pytest.mark.parametrize("V,K,L,seed", [(3, 2, 2, 0), (3, 3, 2, 1), (2, 3, 3, 2), (2, 4, 2, 3)])
def test_token_mode_matches_independent_rrs(V, K, L, seed):
    """The oracle's per-position multi-draft mode (sample space, uniforms,
    trie) against the same rule written in probability space."""
    _, tp, P, Q = tm.exact("token", V, K, L, seed)
    assert abs(tm.expected_tau(tp) - tm.rrs_expected_tau(P, Q, V, K, L)) < TOL


@pytest.mark.parametrize("seed", [0, 4])
def test_multidraft_K1_is_block_verification(seed):
    V, L = 3, 3
    sp1, tp1, _, _ = tm.exact("multidraft", V, 1, L, seed)
    sp2, tp2, _, _ = tm.exact("block", V, 1, L, seed)
    assert np.max(np.abs(sp1 - sp2)) < TOL
    assert np.max(np.abs(tp1 - tp2)) < TOL


@pytest.mark.parametrize("seed", [0, 1, 5])
def test_block_tail_identity(seed):
    """P(tau >= i) = E_X[p_i(X)] for greedy block verification."""
    V, L = 3, 3
    _, tp, P, Q = tm.exact("block", V, 1, L, seed)
    ep = tm.gbv_expected_p(P, Q, V, L)
    tail = np.cumsum(tp[::-1])[::-1]
    assert np.max(np.abs(tail[1:] - ep[1:])) < TOL


def _fixed_problem(V, K, L, seed, T=1.0, dtype="f32"):
    rng = np.random.default_rng(seed)
    tgt = rng.normal(0, 1.5, (1, K, L + 1, V)).astype(np.float32)
    dft = (tgt[:, :, :L] + rng.normal(0, 1.0, (1, K, L, V))).astype(np.float32)
    tok = rng.integers(0, V, (1, K, L)).astype(np.int32)
    au = np.zeros((1, K, L))
    su = np.zeros((1, K, L + 1))
    return oracle.Problem(tgt, dft, tok, None, au, su, T), tgt, dft, tok


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_token_closed_form_fixed_draft(seed):
    """K = 1, fixed draft: P(tau = i, token = x) =
    prod_{j<i} r_j * (1 - r_i) * res_i(x) for i < L and prod_j r_j * P_L(x)
    for i = L, with r_j = min(1, P_j(X)/Q_j(X)), res = norm(max(P - Q, 0))."""
    V, L, T = 5, 3, 1.0
    prob, tgt, dft, tok = _fixed_problem(V, 1, L, seed, T)
    ex = oracle.exact_outcomes("token", prob)
    P = tm.softmax_rows(tgt[0, 0], T)
    Q = tm.softmax_rows(dft[0, 0], T)
    r = [min(1.0, P[j, tok[0, 0, j]] / Q[j, tok[0, 0, j]]) for j in range(L)]
    want = np.zeros((L + 1, V))
    for i in range(L + 1):
        head = np.prod(r[:i])
        if i < L:
            res = np.maximum(P[i] - Q[i], 0.0)
            want[i] = head * (1 - r[i]) * res / res.sum()
        else:
            want[i] = head * P[L]
    assert np.max(np.abs(ex[:, 0, :] - want)) < TOL


@pytest.mark.parametrize("seed", [0, 3])
def test_block_closed_form_fixed_draft(seed):
    """GBV with a fixed draft: P(tau = i) = h_i * prod_{m>i} (1 - h_m) and the
    correction given tau = i < L follows norm(max(p_i P_i - Q_i, 0))."""
    V, L, T = 4, 3, 0.8
    prob, tgt, dft, tok = _fixed_problem(V, 1, L, seed, T)
    ex = oracle.exact_outcomes("block", prob)
    P = tm.softmax_rows(tgt[0, 0], T)
    Q = tm.softmax_rows(dft[0, 0], T)
    X = tok[0, 0]
    p = [1.0]
    for i in range(1, L + 1):
        p.append(min(p[-1] * P[i - 1, X[i - 1]] / Q[i - 1, X[i - 1]], 1.0))
    h = [1.0] * (L + 1)
    for i in range(1, L):
        S = np.maximum(p[i] * P[i] - Q[i], 0).sum()
        h[i] = S / (S + 1 - p[i])
    h[L] = p[L]
    for i in range(L + 1):
        pt = (h[i] if i > 0 else 1.0) * np.prod([1 - h[m] for m in range(i + 1, L + 1)])
        if i < L:
            res = np.maximum(p[i] * P[i] - Q[i], 0)
            want = pt * res / res.sum()
        else:
            want = pt * P[L]
        assert np.max(np.abs(ex[i, 0] - want)) < TOL


def test_rrs_two_draws_closed_form():
    """Recursive rejection sampling at the root with two drafts and L = 1:
    draw 1 accepted w.p. a1 = min(1, P(y1)/Q(y1)); after a rejection the
    residual r1 = norm(max(P - Q, 0)) accepts y2 w.p. min(1, r1(y2)/Q(y2));
    after two rejections the correction comes from norm(max(r1 - Q, 0))."""
    V, K, L, T = 4, 2, 1, 1.0
    for seed in range(4):
        prob, tgt, dft, tok = _fixed_problem(V, K, L, seed, T)
        tok[0, 1, 0] = (tok[0, 0, 0] + 1) % V  # distinct tokens
        prob = oracle.Problem(tgt, dft, tok, None, prob.accept_u, prob.sample_u, T)
        ex = oracle.exact_outcomes("token", prob)
        P = tm.softmax_rows(tgt[0, 0, 0], T)
        Q = tm.softmax_rows(dft[0, 0, 0], T)
        y1, y2 = tok[0, 0, 0], tok[0, 1, 0]
        a1 = min(1.0, P[y1] / Q[y1])
        r1 = np.maximum(P - Q, 0)
        r1 /= r1.sum()
        a2 = min(1.0, r1[y2] / Q[y2])
        r2 = np.maximum(r1 - Q, 0)
        assert abs(ex[1, 0].sum() - a1) < TOL
        assert abs(ex[1, 1].sum() - (1 - a1) * a2) < TOL
        if r2.sum() > 0:
            want = (1 - a1) * (1 - a2) * r2 / r2.sum()
            assert np.max(np.abs(ex[0, 0] - want)) < TOL


@pytest.mark.parametrize("mode", ["block", "multidraft"])
def test_full_weight_with_tiny_residual_accepts(mode):
    # GBV (and SpecTr-GBV at K = 1): h = S / (S + 1 - p).  With p = 1 the
    # test accepts for any S > 0, however small: here the depth-0 ratio
    # P(X)/Q(X) is 1, so p_1 = 1, and the depth-1 residual lives on one
    # token whose target probability is about 1.5e-16 (below half an ulp
    # of 1 in double) while the draft's is about 1e-35.
    V, K, L = 2, 1, 2
    tgt = np.zeros((1, K, L + 1, V), np.float32)
    dft = np.zeros((1, K, L, V), np.float32)
    tgt[0, 0, 1] = [0.0, np.log(1.5e-16)]
    dft[0, 0, 1] = [0.0, -80.0]
    tok = np.zeros((1, K, L), np.int32)
    prob = oracle.Problem(tgt, dft, tok, None, np.zeros((1, K, L)), np.zeros((1, K, L + 1)), 1.0)
    out = oracle.verify(mode, prob)
    assert out["rc"] == 0
    assert out["accept_prob"][0, 0, 0] == 1.0  # h at depth 1
    assert 1e-16 < out["residual_mass"][0] < 1e-15 or out["accept_len"][0] == L


@pytest.mark.parametrize("mode,K", [("token", 1), ("token", 3), ("block", 1), ("multidraft", 3)])
def test_identical_models_accept_everything(mode, K):
    V, L = 4, 3
    rng = np.random.default_rng(7)
    tgt = rng.normal(0, 2, (1, K, L + 1, V)).astype(np.float32)
    dft = tgt[:, :, :L].copy()
    tok = rng.integers(0, V, (1, K, L)).astype(np.int32)
    for k in range(1, K):  # same prefix => same rows
        tgt[0, k, 0] = tgt[0, 0, 0]
        dft[0, k, 0] = dft[0, 0, 0]
    prob = oracle.Problem(tgt, dft, tok, None, np.zeros((1, K, L)), np.zeros((1, K, L + 1)), 1.0)
    ex = oracle.exact_outcomes(mode, prob)
    assert abs(ex[L].sum() - 1.0) < 1e-12
    # bonus token ~ the first draft's last target row
    P = tm.softmax_rows(tgt[0, 0, L], 1.0)
    assert np.max(np.abs(ex[L, 0] - P)) < 1e-12


@pytest.mark.parametrize("mode,K", [("token", 1), ("token", 2), ("block", 1), ("multidraft", 2)])
def test_disjoint_supports_reject_at_root(mode, K):
    V, L = 6, 2
    rng = np.random.default_rng(11)
    tgt = rng.normal(0, 1, (1, K, L + 1, V)).astype(np.float32)
    dft = rng.normal(0, 1, (1, K, L, V)).astype(np.float32)
    tgt[..., 3:] = -np.inf   # target lives on {0,1,2}
    dft[..., :3] = -np.inf   # draft lives on {3,4,5}
    tok = rng.integers(3, 6, (1, K, L)).astype(np.int32)
    for k in range(1, K):
        tgt[0, k, 0] = tgt[0, 0, 0]
        dft[0, k, 0] = dft[0, 0, 0]
    prob = oracle.Problem(tgt, dft, tok, None, np.zeros((1, K, L)), np.zeros((1, K, L + 1)), 1.0)
    ex = oracle.exact_outcomes(mode, prob)
    P0 = tm.softmax_rows(tgt[0, 0, 0], 1.0)
    assert abs(ex[0].sum() - 1.0) < 1e-12
    assert np.max(np.abs(ex[0, 0] - P0)) < 1e-12


@pytest.mark.parametrize("mode", ["token", "block", "multidraft", "greedy"])
def test_empty_draft_samples_context_row(mode):
    V, K = 5, 1
    rng = np.random.default_rng(3)
    tgt = rng.normal(0, 1, (1, K, 1, V)).astype(np.float32)
    dft = np.zeros((1, K, 0, V), np.float32)
    tok = np.zeros((1, K, 0), np.int32)
    prob = oracle.Problem(tgt, dft, tok, None, np.zeros((1, K, 0)), np.zeros((1, K, 1)), 1.0)
    ex = oracle.exact_outcomes(mode, prob)
    if mode == "greedy":
        want = np.zeros(V)
        want[np.argmax(tgt[0, 0, 0])] = 1
    else:
        want = tm.softmax_rows(tgt[0, 0, 0], 1.0)
    assert np.max(np.abs(ex[0, 0] - want)) < 1e-12


@pytest.mark.parametrize("seed", range(6))
def test_greedy_matches_target_greedy_decode(seed):
    """Greedy T = 0: the emitted stream is the target's own greedy decode for
    tau + 1 tokens, and no draft matches that decode for longer than tau."""
    V, K, L = 3, 3, 3
    tgt_tab, dft_tab, P, Q = tm.make(V, L, seed)
    rng = np.random.default_rng(100 + seed)
    drafts = rng.integers(0, V, (K, L))
    drafts[1, :2] = drafts[0, :2]  # shared prefixes exercise the trie
    tgt = np.zeros((1, K, L + 1, V), np.float32)
    dft = np.zeros((1, K, L, V), np.float32)
    for k in range(K):
        for j in range(L + 1):
            tgt[0, k, j] = tgt_tab[oracle.prefix_index(drafts[k, :j], V)]
        for j in range(L):
            dft[0, k, j] = dft_tab[oracle.prefix_index(drafts[k, :j], V)]
    for mode in ("greedy", "token", "multidraft"):
        prob = oracle.Problem(tgt, dft, drafts[None].astype(np.int32), None,
                              np.zeros((1, K, L)), np.zeros((1, K, L + 1)), 0.0)
        o = oracle.verify(mode, prob)
        # the target's greedy decode (first maximal logit)
        dec = []
        for i in range(L + 1):
            dec.append(int(np.argmax(tgt_tab[oracle.prefix_index(dec, V)])))
        match = [next((m for m in range(L) if drafts[k, m] != dec[m]), L) for k in range(K)]
        tau = o["accept_len"][0]
        assert tau == max(match)
        assert o["accept_draft"][0] == match.index(max(match))
        assert o["out_token"][0] == dec[tau]


def test_sampler_inverse_cdf_intervals():
    """The inverse-CDF draw maps u to the first token whose running sum
    exceeds u*S: the token intervals tile [0, 1) in index order with widths
    equal to the normalised weights."""
    V, L = 6, 0
    rng = np.random.default_rng(5)
    tgt = rng.normal(0, 1, (1, 1, 1, V)).astype(np.float32)
    tgt[0, 0, 0, 2] = -np.inf  # a zero-mass token is never drawn
    P = tm.softmax_rows(tgt[0, 0, 0], 1.0)
    edges = np.concatenate([[0.0], np.cumsum(P)])
    for u in np.linspace(0, 1, 97, endpoint=False):
        prob = oracle.Problem(tgt, np.zeros((1, 1, 0, V), np.float32), np.zeros((1, 1, 0), np.int32),
                              None, np.zeros((1, 1, 0)), np.full((1, 1, 1), u), 1.0)
        o = oracle.verify("token", prob)
        x = o["out_token"][0]
        assert P[x] > 0
        assert edges[x] - 1e-12 <= u < edges[x + 1] + 1e-12


# --------------------------------------------------------------------------
# Sensitivity: plant plausible mistakes in a copy of the oracle and check
# that the pins above catch each one.

MUTANTS = {
    "drop_minus_p_in_D": ("D = 1.0 - p + S;", "D = 1.0 + S;"),
    "drop_D_in_acceptance": ("double denom = D * r->Q[y];", "double denom = r->Q[y];"),
    "residual_from_P_each_draw": ("r->R[x] = fmax(r->R[x] - D * r->Q[x], 0.0);",
                                  "r->R[x] = fmax(p * r->P[x] - D * r->Q[x], 0.0);"),
    "h_sign_flip": ("r->h[j][o] = D > 0.0 ? S / D : 1.0;", "r->h[j][o] = S / (1.0 + p + S);"),
    "gbv_h_denominator": ("h[i] = S + (1.0 - p[i]) > 0.0 ? S / (S + (1.0 - p[i])) : 1.0;",
                          "h[i] = S / (S + 1.0);"),
    "gbv_residual_without_p": ("r->R[x] = fmax(p[tau] * r->P[x] - r->Q[x], 0.0);",
                               "r->R[x] = fmax(r->P[x] - r->Q[x], 0.0);"),
    "correction_from_target": ("S = eval_node(r, ej, eo, p);\n        w = S > 0.0 ? r->R : r->P;",
                               "S = eval_node(r, ej, eo, p);\n        w = r->P;"),
    "leaf_bonus_from_stale_residual": ("S = p;\n        w = r->P;", "S = p;\n        w = r->R;"),
    "no_trie_merge": ("o = k2;\n                    break;", "break;"),
    "merge_only_at_root": ("for (int k2 = 0; k2 < k; ++k2) {", "for (int k2 = 0; k2 < k && j == 0; ++k2) {"),
    "child_weight_from_wrong_level": ("return j == 0 ? 1.0 : r->a[j - 1][o];",
                                      "return j == 0 ? 1.0 : (j >= 2 ? r->a[j - 2][o] : 1.0);"),
}


def _build_mutant(tmpdir, name):
    here = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle")
    src = open(os.path.join(here, "sdv_oracle.c")).read()
    old, new = MUTANTS[name]
    assert src.count(old) == 1, name
    d = os.path.join(tmpdir, name)
    os.makedirs(d)
    open(os.path.join(d, "sdv_oracle.c"), "w").write(src.replace(old, new))
    shutil.copy(os.path.join(here, "sdv_oracle.h"), d)
    shutil.copy(os.path.join(here, "exact.c"), d)
    so = os.path.join(d, "libm.so")
    subprocess.run(["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-o", so,
                    os.path.join(d, "sdv_oracle.c"), os.path.join(d, "exact.c"), "-lm"], check=True)
    return so


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, monkeypatch):
    with tempfile.TemporaryDirectory() as tmp:
        so = _build_mutant(tmp, name)
        mlib = ctypes.CDLL(so)
        mlib.sdvo_exact_streams.restype = ctypes.c_int
        monkeypatch.setattr(oracle, "_lib", mlib)
        caught = []
        for mode, K, L, V in [("multidraft", 3, 2, 3), ("multidraft", 1, 3, 3), ("token", 3, 2, 3),
                              ("block", 1, 3, 3), ("multidraft", 2, 2, 2)]:
            for seed in (0, 2):
                try:
                    sp, tp, P, Q = tm.exact(mode, V, K, L, seed)
                except RuntimeError:
                    caught.append((mode, "error"))
                    continue
                if tm.completed_stream_error(sp, P, V, L) > 1e-9:
                    caught.append((mode, K))
        # acceptance invariants under the same mutant; the per-position
        # reference comes from the independent probability-space recursion
        for seed in (0, 1, 2):
            try:
                e = {K: tm.expected_tau(tm.exact("multidraft", 3, K, 2, seed)[1]) for K in (1, 2, 3)}
                et = {K: tm.expected_tau(tm.exact("token", 3, K, 2, seed)[1]) for K in (1, 2, 3)}
            except RuntimeError:
                caught.append("error")
                continue
            _, _, P, Q = tm.make(3, 2, seed)
            ref = {K: tm.rrs_expected_tau(P, Q, 3, K, 2) for K in (1, 2, 3)}
            if not (e[2] > e[1] + 1e-6 and e[3] >= e[2] - TOL
                    and all(e[K] >= ref[K] - TOL and abs(et[K] - ref[K]) < 1e-9 for K in (1, 2, 3))):
                caught.append(("invariant", seed))
        assert caught, f"mutant {name} not caught by the stream-validity pin"


@pytest.mark.parametrize("mode,K", [("token", 1), ("token", 3), ("block", 1), ("multidraft", 3), ("kseq", 3),
                                    ("greedy", 2)])
@pytest.mark.parametrize("seed", [0, 4])
def test_exact_accept_len_is_the_outcome_marginal(mode, K, seed):
    """sdvo_exact_accept_len integrates over the accept uniforms alone: its
    P(tau = i) equals the marginal of the full exact outcome law, and the
    token rule at K = 1 gives the closed-form tail prod_{j<i} r_j."""
    V, L, T = 4, 3, 0.8
    prob, tgt, dft, tok = _fixed_problem(V, K, L, seed, T)
    ex = oracle.exact_outcomes(mode, prob)
    tau = oracle.exact_accept_len(mode, prob)
    assert abs(tau.sum() - 1.0) < TOL
    assert np.max(np.abs(tau - ex.sum(axis=(1, 2)))) < TOL
    if mode == "token" and K == 1:
        P = tm.softmax_rows(tgt[0, 0], T)
        Q = tm.softmax_rows(dft[0, 0], T)
        r = [min(1.0, P[j, tok[0, 0, j]] / Q[j, tok[0, 0, j]]) for j in range(L)]
        tail = [np.prod(r[:i]) for i in range(L + 1)]
        assert np.max(np.abs(np.cumsum(tau[::-1])[::-1] - tail)) < TOL


def test_expected_accept_len_over_requests():
    """expected_accept_len: per request E[tau] = sum_i i P(tau = i), one
    request at a time on host threads."""
    V, K, L, T = 4, 2, 3, 1.0
    probs = [_fixed_problem(V, K, L, s, T)[0] for s in range(3)]
    for mode in ("token", "multidraft"):
        for p in probs:
            want = float(np.dot(np.arange(L + 1), oracle.exact_accept_len(mode, p)))
            got = oracle.expected_accept_len(mode, p, threads=2)
            assert got.shape == (1,) and abs(got[0] - want) < TOL
