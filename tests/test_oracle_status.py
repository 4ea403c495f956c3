"""Oracle host logic: argument checks, per-request data status, unread rows."""
import numpy as np
import pytest

import oracle


def _problem(B=3, K=2, L=3, V=7, seed=0, T=1.0):
    rng = np.random.default_rng(seed)
    tgt = rng.normal(0, 2, (B, K, L + 1, V)).astype(np.float32)
    dft = (tgt[:, :, :L] + rng.normal(0, 1, (B, K, L, V))).astype(np.float32)
    tok = rng.integers(0, V, (B, K, L)).astype(np.int32)
    if K > 1:
        tok[:, 1, 0] = tok[:, 0, 0]      # drafts 0 and 1 share their first token
        tgt[:, 1, :2] = tgt[:, 0, :2]    # ... hence their rows up to depth 1
        dft[:, 1, :2] = dft[:, 0, :2]
    au = rng.random((B, K, L))
    su = rng.random((B, K, L + 1))
    lengths = np.array([L, 1, 2][:B], np.int32)
    return dict(target=tgt, draft=dft, tokens=tok, lengths=lengths, accept_u=au, sample_u=su, temperature=T)


def _run(mode, d):
    return oracle.verify(mode, oracle.Problem(**d))


MODES = ["token", "greedy", "multidraft"]


@pytest.mark.parametrize("mode", MODES)
def test_nan_in_used_row_flags_only_that_request(mode):
    d = _problem()
    base = _run(mode, d)
    assert (base["req_status"] == 0).all()
    d["target"][1, 0, 0, 3] = np.nan
    o = _run(mode, d)
    assert o["req_status"][1] == oracle.REQ_NONFINITE
    assert o["out_token"][1] == -1 and o["accept_len"][1] == 0
    for b in (0, 2):
        assert o["req_status"][b] == 0
        assert o["out_token"][b] == base["out_token"][b]
        assert o["accept_len"][b] == base["accept_len"][b]


@pytest.mark.parametrize("value", [np.inf, np.nan])
def test_nonfinite_draft_row(value):
    d = _problem()
    d["draft"][0, 0, 1, 2] = value
    o = _run("token", d)
    assert o["req_status"][0] == oracle.REQ_NONFINITE
    # greedy never reads draft rows
    assert _run("greedy", d)["req_status"][0] == 0


def test_all_minus_inf_row_is_invalid_but_partial_minus_inf_is_fine():
    d = _problem()
    d["target"][2, 0, 1, :3] = -np.inf
    assert _run("token", d)["req_status"][2] == 0
    d["target"][2, 0, 1, :] = -np.inf
    assert _run("token", d)["req_status"][2] == oracle.REQ_NONFINITE


@pytest.mark.parametrize("mode", MODES)
def test_unread_rows_never_matter(mode):
    """Rows past a request's length, duplicate-prefix copies and row padding
    are never read: poisoning them changes nothing."""
    d = _problem()
    base = _run(mode, d)
    # request 1 has length 1: rows 2.. of target and 1.. of draft are unused
    d["target"][1, :, 2:] = np.nan
    d["draft"][1, :, 1:] = np.nan
    # draft 1 shares depth 0 and 1 with draft 0: its copies are unread
    d["target"][:, 1, :2] = np.nan
    d["draft"][:, 1, :2] = np.nan
    # tokens past the length are padding
    d["tokens"][1, :, 1:] = 99999
    o = _run(mode, d)
    assert (o["req_status"] == 0).all()
    for key in ("accept_len", "accept_draft", "out_token"):
        np.testing.assert_array_equal(o[key], base[key])


def test_padding_columns_are_not_read():
    d = _problem(V=7)
    base = _run("multidraft", d)
    for key in ("target", "draft"):
        a = d[key]
        pad = np.full(a.shape[:-1] + (3,), np.nan, np.float32)
        d[key] = np.concatenate([a, pad], axis=-1)
    o = oracle.verify("multidraft", oracle.Problem(**d, V=7))
    assert (o["req_status"] == 0).all()
    np.testing.assert_array_equal(o["out_token"], base["out_token"])


def test_bad_tokens_and_lengths():
    d = _problem()
    d["tokens"][0, 1, 2] = 7          # == V, at a used position of request 0
    d["lengths"][2] = 4               # > L
    o = _run("token", d)
    assert o["req_status"][0] == oracle.REQ_BAD_TOKEN
    assert o["req_status"][1] == 0
    assert o["req_status"][2] == oracle.REQ_BAD_LENGTH
    d["lengths"][2] = -1
    assert _run("token", d)["req_status"][2] == oracle.REQ_BAD_LENGTH


@pytest.mark.parametrize("field,value", [("temperature", -0.5), ("temperature", float("nan")),
                                         ("temperature", float("inf"))])
def test_invalid_arguments(field, value):
    d = _problem()
    d[field] = value
    assert _run("token", d)["rc"] == 1


def test_block_requires_single_draft():
    assert _run("block", _problem(K=2))["rc"] == 1
    assert _run("block", _problem(K=1))["rc"] == 0


def test_zero_temperature_is_greedy_in_every_mode():
    d = _problem(T=0.0)
    g = _run("greedy", d)
    for mode in ("token", "multidraft"):
        o = _run(mode, d)
        for key in ("accept_len", "accept_draft", "out_token", "accept_prob"):
            np.testing.assert_array_equal(o[key], g[key])


def test_bf16_is_decoded_exactly():
    d = _problem()
    # values exactly representable in bf16: decoding must not change them
    for key in ("target", "draft"):
        a = d[key]
        bits = (a.view(np.uint32) >> 16).astype(np.uint16)
        d[key + "_bits"] = bits
        d[key] = (bits.astype(np.uint32) << 16).view(np.float32)
    f = oracle.verify("multidraft", oracle.Problem(d["target"], d["draft"], d["tokens"], d["lengths"],
                                                   d["accept_u"], d["sample_u"], 1.0))
    b = oracle.verify("multidraft", oracle.Problem(d["target_bits"], d["draft_bits"], d["tokens"],
                                                   d["lengths"], d["accept_u"], d["sample_u"], 1.0))
    for key in ("accept_len", "accept_draft", "out_token", "accept_prob", "residual_mass"):
        np.testing.assert_array_equal(f[key], b[key])


def _leaves(d, b):
    """Drafts owning a leaf of request b (no lower draft has its first L_b tokens)."""
    Lb = int(d["lengths"][b])
    tok = d["tokens"][b, :, :Lb]
    return [k for k in range(tok.shape[0]) if not any((tok[k2] == tok[k]).all() for k2 in range(k))]


@pytest.mark.parametrize("mode,K", [("token", 2), ("multidraft", 2), ("block", 1)])
def test_leaf_row_is_read_only_by_its_bonus_draw(mode, K):
    """A leaf's target row enters only the bonus draw when the decision ends
    there (its residual is p P, of mass p, whatever P is).  With accept_u = 0
    every test passes: the decision ends at draft 0's leaf.  Poisoning the
    other leaves changes nothing; poisoning that one invalidates the request
    alone."""
    d = _problem(K=K)
    d["accept_u"][:] = 0.0
    base = _run(mode, d)
    assert (base["req_status"] == 0).all()
    np.testing.assert_array_equal(base["accept_len"], d["lengths"])
    np.testing.assert_array_equal(base["accept_draft"], 0)
    for b in range(3):
        for k in _leaves(d, b)[1:]:
            d["target"][b, k, d["lengths"][b], 1] = np.nan
    o = _run(mode, d)
    assert (o["req_status"] == 0).all()
    for key in ("accept_len", "accept_draft", "out_token", "accept_prob", "residual_mass"):
        np.testing.assert_array_equal(o[key], base[key])
    d["target"][2, 0, d["lengths"][2], 4] = np.inf
    o = _run(mode, d)
    assert o["req_status"].tolist() == [0, 0, oracle.REQ_NONFINITE]
    assert o["accept_len"][2] == 0 and o["accept_draft"][2] == 0 and o["out_token"][2] == -1
    assert o["residual_mass"][2] == 0.0 and (o["accept_prob"][2] == 0).all()
    for key in ("accept_len", "out_token", "accept_prob"):
        np.testing.assert_array_equal(o[key][:2], base[key][:2])


@pytest.mark.parametrize("mode,K", [("token", 2), ("multidraft", 2), ("block", 1)])
def test_leaf_rows_are_unread_when_a_draft_position_is_rejected(mode, K):
    """With accept_u near 1 almost every test fails; a request that stops
    short of its length never reads a leaf row."""
    d = _problem(K=K, seed=4)
    d["accept_u"][:] = 0.999
    base = _run(mode, d)
    short = [b for b in range(3) if base["accept_len"][b] < d["lengths"][b]]
    assert short, "the fixture should stop short somewhere"
    for b in short:
        for k in range(K):
            d["target"][b, k, d["lengths"][b]] = np.nan
    o = _run(mode, d)
    assert (o["req_status"] == 0).all()
    for key in ("accept_len", "accept_draft", "out_token", "accept_prob", "residual_mass"):
        np.testing.assert_array_equal(o[key], base[key])


def test_greedy_reads_a_leaf_row_only_where_the_decision_ends():
    """Greedy's matches use the inner nodes' argmaxes; a leaf's argmax is the
    correction only when the decision ends there.  Draft 0 follows its rows'
    argmax path, so every request ends at draft 0's leaf: the other leaves
    are never read, and poisoning draft 0's leaf invalidates that request
    alone."""
    d = _problem(K=3)
    for b in range(3):
        for j in range(d["lengths"][b]):
            d["tokens"][b, 0, j] = np.argmax(d["target"][b, 0, j])
        d["tokens"][b, 1, 0] = d["tokens"][b, 0, 0]  # the fixture's shared first token
    base = _run("greedy", d)
    assert (base["req_status"] == 0).all()
    np.testing.assert_array_equal(base["accept_len"], d["lengths"])
    np.testing.assert_array_equal(base["accept_draft"], 0)
    for b in range(3):
        np.testing.assert_equal(base["out_token"][b], np.argmax(d["target"][b, 0, d["lengths"][b]]))
        for k in _leaves(d, b)[1:]:
            d["target"][b, k, d["lengths"][b], 1] = np.nan
    o = _run("greedy", d)
    assert (o["req_status"] == 0).all()
    for key in ("accept_len", "accept_draft", "out_token", "accept_prob"):
        np.testing.assert_array_equal(o[key], base[key])
    d["target"][2, 0, d["lengths"][2], 4] = np.inf
    o = _run("greedy", d)
    assert o["req_status"].tolist() == [0, 0, oracle.REQ_NONFINITE]
    assert o["accept_len"][2] == 0 and o["accept_draft"][2] == 0 and o["out_token"][2] == -1
    assert (o["accept_prob"][2] == 0).all()
    for key in ("accept_len", "out_token", "accept_prob"):
        np.testing.assert_array_equal(o[key][:2], base[key][:2])


def test_greedy_that_stops_short_reads_no_leaf():
    d = _problem(K=2, seed=5)
    base = _run("greedy", d)
    short = [b for b in range(3) if base["accept_len"][b] < d["lengths"][b]]
    assert short, "the fixture should stop short somewhere"
    for b in short:
        d["target"][b, :, d["lengths"][b]] = np.nan
    o = _run("greedy", d)
    assert (o["req_status"] == 0).all()
    for key in ("accept_len", "accept_draft", "out_token", "accept_prob"):
        np.testing.assert_array_equal(o[key], base[key])
