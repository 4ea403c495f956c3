"""Pins of the oracle's LM head (oracle.lm_head_logits) and of its f64 logit
rows, which together define greedy verification fused into the LM head.

The target model's pass ends in its LM head: logits = hidden . W^T, one row
of W per vocabulary entry ("Speculative Decoding: Performance or Illusion?",
section 3.2, where verification is the target model's pass).  The greedy
rule on those logits is the one the verification oracle already implements;
the fused form only changes where the logits come from.  These tests fix the
LM head against exact integer arithmetic, a closed form and an independent
numpy product, and fix the f64 row decoding against the f32 one.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle


def _bf16(a):
    return torch.as_tensor(np.asarray(a, np.float32)).to(torch.bfloat16)


def test_integer_inputs_give_the_exact_integer_products():
    # small integers are exact in bf16; M != V and an odd d catch a transposed
    # operand, a dropped term or an index off by one
    rng = np.random.default_rng(11)
    M, V, d = 5, 7, 13
    h = rng.integers(-8, 9, size=(M, d))
    w = rng.integers(-8, 9, size=(V, d))
    got = oracle.lm_head_logits(_bf16(h), _bf16(w))
    want = [[sum(int(h[r, i]) * int(w[x, i]) for i in range(d)) for x in range(V)] for r in range(M)]
    assert got.shape == (M, V)
    assert got.tolist() == want


def test_one_hot_hidden_reads_one_column_of_the_head():
    rng = np.random.default_rng(12)
    V, d = 9, 6
    w = _bf16(rng.standard_normal((V, d)))
    wd = w.double().numpy()
    for i in range(d):
        h = np.zeros((1, d), np.float32)
        h[0, i] = -2.0
        got = oracle.lm_head_logits(_bf16(h), w)
        assert np.array_equal(got[0], -2.0 * wd[:, i])


def test_matches_an_independent_float64_product():
    rng = np.random.default_rng(13)
    h = _bf16(rng.standard_normal((4, 3, 96)))
    w = _bf16(rng.standard_normal((301, 96)) * 0.1)
    got = oracle.lm_head_logits(h, w)
    want = np.einsum("abi,xi->abx", h.double().numpy(), w.double().numpy())
    assert got.shape == (4, 3, 301)
    assert np.max(np.abs(got - want)) <= 1e-12 * np.max(np.abs(want))


def test_columns_past_V_are_not_written(oracle_lib):
    h = _bf16(np.ones((2, 8))).view(torch.int16).numpy()
    w = _bf16(np.ones((3, 8))).view(torch.int16).numpy()
    out = np.full((2, 5), 7.5)
    rc = oracle_lib.sdvo_lm_head_logits(ctypes.c_int(2), ctypes.c_int(3), ctypes.c_int(8),
                                        h.ctypes.data_as(ctypes.c_void_p), w.ctypes.data_as(ctypes.c_void_p),
                                        out.ctypes.data_as(ctypes.c_void_p), ctypes.c_longlong(5))
    assert rc == 0
    assert out[:, :3].tolist() == [[8.0] * 3] * 2
    assert out[:, 3:].tolist() == [[7.5, 7.5]] * 2


def test_bad_arguments_are_rejected(oracle_lib):
    x = np.zeros(16, np.uint16)
    o = np.zeros(16)
    p = x.ctypes.data_as(ctypes.c_void_p)
    q = o.ctypes.data_as(ctypes.c_void_p)
    f = oracle_lib.sdvo_lm_head_logits
    assert f(ctypes.c_int(1), ctypes.c_int(4), ctypes.c_int(0), p, p, q, ctypes.c_longlong(4)) != 0
    assert f(ctypes.c_int(1), ctypes.c_int(4), ctypes.c_int(2), p, p, q, ctypes.c_longlong(3)) != 0
    assert f(ctypes.c_int(-1), ctypes.c_int(4), ctypes.c_int(2), p, p, q, ctypes.c_longlong(4)) != 0
    assert f(ctypes.c_int(0), ctypes.c_int(4), ctypes.c_int(2), None, None, None, ctypes.c_longlong(4)) == 0


def _problem(target, tokens, lengths=None):
    B, K, L1, V = target.shape
    return oracle.Problem(target, None, tokens, lengths, None, None, 0.0, V=V)


@pytest.mark.parametrize("mode", ["greedy", "token", "multidraft"])
def test_f64_rows_decode_like_f32_rows(mode):
    # the same values as f32 and as f64 give the same results in every rule
    rng = np.random.default_rng(14)
    B, K, L, V = 3, 3, 4, 37
    t32 = (rng.standard_normal((B, K, L + 1, V)) * 2).astype(np.float32)
    d32 = (t32[:, :, :L] + rng.standard_normal((B, K, L, V)).astype(np.float32)).astype(np.float32)
    tokens = rng.integers(0, V, size=(B, K, L)).astype(np.int32)
    tokens[:, 1, :2] = tokens[:, 0, :2]  # a shared prefix
    au = rng.random((B, K, L))
    su = rng.random((B, K, L + 1))
    T = 0.0 if mode == "greedy" else 0.8
    p32 = oracle.Problem(t32, d32, tokens, None, au, su, T, V=V)
    p64 = oracle.Problem(t32.astype(np.float64), d32.astype(np.float64), tokens, None, au, su, T, V=V)
    assert p64.dtype == oracle.F64
    a = oracle.verify(mode, p32)
    b = oracle.verify(mode, p64)
    for key in ("accept_len", "accept_draft", "out_token", "accept_prob", "req_status"):
        assert np.array_equal(a[key], b[key]), key


def test_f64_rows_keep_differences_f32_would_lose():
    # logits 1 and 1 + 2^-40 tie in f32 (lowest index wins); in f64 the
    # second is the argmax
    V = 4
    t = np.zeros((1, 1, 2, V))
    t[..., 0] = 1.0
    t[..., 2] = 1.0 + 2.0 ** -40
    tokens = np.array([[[2]]], np.int32)
    r64 = oracle.verify("greedy", _problem(t, tokens))
    r32 = oracle.verify("greedy", _problem(t.astype(np.float32), tokens))
    assert (r64["accept_len"][0], r64["out_token"][0]) == (1, 2)
    assert (r32["accept_len"][0], r32["out_token"][0]) == (0, 0)


def test_fused_greedy_by_brute_force():
    # tiny integer LM head: exact logits, the greedy rule written out here
    # (longest run of drafted tokens equal to the row argmax, lowest draft on
    # ties; correction = argmax at the end row)
    rng = np.random.default_rng(15)
    B, K, L, V, d = 6, 3, 3, 11, 5
    w = rng.integers(-3, 4, size=(V, d))
    hidden = rng.integers(-3, 4, size=(B, K, L + 1, d))
    tokens = np.zeros((B, K, L), np.int32)
    am = np.zeros((B, K, L + 1), np.int64)
    for j in range(L + 1):  # depth by depth: drafts with a common prefix share its row
        for b in range(B):
            for k in range(K):
                for k2 in range(k):
                    if np.array_equal(tokens[b, k, :j], tokens[b, k2, :j]):
                        hidden[b, k, j] = hidden[b, k2, j]
                        break
        am[:, :, j] = np.argmax(hidden[:, :, j] @ w.T, axis=-1)  # first maximum
        if j < L:
            tokens[:, :, j] = np.where(rng.random((B, K)) < 0.7, am[:, :, j], rng.integers(0, 3, size=(B, K)))
    logits = oracle.lm_head_logits(_bf16(hidden), _bf16(w))
    assert logits.tolist() == (hidden @ w.T).tolist()
    lengths = rng.integers(0, L + 1, size=B).astype(np.int32)
    got = oracle.verify("greedy", _problem(logits, tokens, lengths))
    for b in range(B):
        best, bk = -1, 0
        for k in range(K):
            m = 0
            while m < lengths[b] and tokens[b, k, m] == am[b, k, m]:
                m += 1
            if m > best:
                best, bk = m, k
        assert got["accept_len"][b] == best
        assert got["accept_draft"][b] == bk
        assert got["out_token"][b] == am[b, bk, best]
