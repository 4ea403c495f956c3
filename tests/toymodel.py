"""Prefix-consistent toy language models for the oracle's exact pins.

A toy model assigns a target and a draft logit row to every prefix of length
0..n over a vocabulary of V tokens (rows indexed like
``oracle.prefix_index``).  Probabilities are computed here with numpy, in
float64, from the float32 logits the oracle sees; nothing here calls the
oracle's arithmetic.
"""
import itertools

import numpy as np

import oracle


def softmax_rows(logits_f32, T):
    a = logits_f32.astype(np.float64) / T
    e = np.exp(a - a.max(axis=-1, keepdims=True))
    return e / e.sum(axis=-1, keepdims=True)


def make(V, n, seed, T=1.0, scale=1.5, noise=1.0):
    """Tables for prefixes of length 0..n: (tgt_logits, dft_logits, P, Q)."""
    rng = np.random.default_rng(seed)
    rows = oracle.n_prefixes(n, V)
    tgt = rng.normal(0.0, scale, (rows, V)).astype(np.float32)
    dft = (tgt + rng.normal(0.0, noise, (rows, V))).astype(np.float32)
    return tgt, dft, softmax_rows(tgt, T), softmax_rows(dft, T)


def target_prob(P, s, V):
    """Target probability of the string s under the toy model."""
    pr = 1.0
    for i in range(len(s)):
        pr *= P[oracle.prefix_index(s[:i], V), s[i]]
    return pr


def completed_stream_error(stream_prob, P, V, L):
    """Largest |P(completed stream starts with s) - P_target(s)| over |s| = L+1.

    The completed stream is the emitted stream (accepted prefix plus the
    correction token) followed by tokens drawn from the target; speculative
    verification is valid iff it is distributed as the target."""
    err = 0.0
    for s in itertools.product(range(V), repeat=L + 1):
        truth = target_prob(P, s, V)
        got = 0.0
        for m in range(1, L + 2):
            cont = 1.0
            for i in range(m, L + 1):
                cont *= P[oracle.prefix_index(s[:i], V), s[i]]
            got += stream_prob[oracle.prefix_index(s[:m], V)] * cont
        err = max(err, abs(got - truth))
    return err


def exact(mode, V, K, L, seed, T=1.0, **kw):
    """Exact (stream_prob, tau_prob, P, Q) for a toy model."""
    tgt, dft, P, Q = make(V, L, seed, T, **kw)
    sp, tp = oracle.exact_streams(mode, V, K, L, T, tgt, dft, Q)
    return sp, tp, P, Q


def expected_tau(tau_prob):
    return float(np.dot(tau_prob, np.arange(len(tau_prob))))


def gbv_expected_p(P, Q, V, L):
    """E over single drafts X ~ Q of p_i(X) for i = 1..L, with p_0 = 1 and
    p_i = min(p_{i-1} P(X_i | X_<i) / Q(X_i | X_<i), 1)."""
    out = np.zeros(L + 1)
    out[0] = 1.0
    for i in range(1, L + 1):
        acc = 0.0
        for x in itertools.product(range(V), repeat=i):
            w, p = 1.0, 1.0
            for t in range(i):
                r = oracle.prefix_index(x[:t], V)
                w *= Q[r, x[t]]
                p = min(p * P[r, x[t]] / Q[r, x[t]], 1.0)
            acc += w * p
        out[i] = acc
    return out


def _rrs_from_node(P, Q, V, drafts, ks, depth, L):
    """Expected further accepted length of recursive rejection sampling at
    the node reached by the drafts ``ks`` (all sharing their first ``depth``
    tokens), computed in probability space: draw j is the first accepted
    with probability prod_{i<j}(1 - a_i) a_j, where a_j = min(1, r(y_j)/Q(y_j))
    and r is renormalised to max(r - Q, 0) after each rejection; the
    accepted token's node carries on with every draft that shares it."""
    if depth == L:
        return 0.0
    row = oracle.prefix_index(list(drafts[ks[0], :depth]), V)
    r = P[row].copy()
    q = Q[row]
    e, reach = 0.0, 1.0
    for k in ks:
        y = drafts[k, depth]
        a = min(1.0, r[y] / q[y]) if q[y] > 0 else 1.0
        child = [k2 for k2 in ks if drafts[k2, depth] == y]
        e += reach * a * (1.0 + _rrs_from_node(P, Q, V, drafts, child, depth + 1, L))
        reach *= 1.0 - a
        r = np.maximum(r - q, 0.0)
        if r.sum() > 0:
            r = r / r.sum()
    return e


def rrs_expected_tau(P, Q, V, K, L):
    """E[tau] of per-position multi-draft verification (recursive rejection
    sampling over the draft trie), averaged over i.i.d. drafts from Q."""
    total = 0.0
    for tup in itertools.product(range(V), repeat=K * L):
        drafts = np.array(tup, dtype=np.int64).reshape(K, L)
        w = 1.0
        for k in range(K):
            for j in range(L):
                w *= Q[oracle.prefix_index(list(drafts[k, :j]), V), drafts[k, j]]
        if w > 0:
            total += w * _rrs_from_node(P, Q, V, drafts, list(range(K)), 0, L)
    return total
