"""GPU-versus-oracle comparison rules.

Bar (per request): accept_len, accept_draft and out_token equal the
oracle's, except where some decision on the oracle's path had a margin
|u - threshold| (or distance of u to its CDF interval's ends) below 1e-5.
Such mismatches are counted per workload (every mode and temperature of it
together, in LEDGER) and must stay below 1e-4 of that workload's decisions
(the decisions the oracle took: accept tests and inverse-CDF draws; one per
request for greedy matching, which has none).  accept_prob within 1e-5
absolute everywhere (for K-SEQ, see KSEQ_FLAT); residual_mass within 1e-5
where the end node agrees.  Requests
the oracle marks invalid must come back invalid with the same status bit.
"""
import numpy as np
import torch

import draft_verification_row_gb300 as sdv
import oracle

TOL = 1e-5
MARGIN = 1e-5
# K-SEQ's acceptance probabilities min(1, P(y) / (rho Q(y))) carry rho from
# a search whose tests gamma(beta(rho)) <= rho take beta, a vocabulary sum,
# in fp32 on the GPU and in fp64 in the oracle.  Both test the same dyadic
# points; where a tested point's two sides lie within KSEQ_FLAT of each
# other (relative), the fp32 sum's rounding settles the test, and the two
# searches may branch apart and end at different rho.  Any rho that passes
# the test keeps the emitted token distributed as P.  Such a node's
# acceptance probabilities are compared with the rho the GPU chose, which
# must pass the test in fp64; the node is counted (LEDGER "kseq_flat_zone").
KSEQ_FLAT = 1e-5


def pad8(a):
    """Pad the last (vocabulary) axis with NaN columns to a multiple of 8:
    the library's row stride rule; the padding must never be read."""
    a = np.asarray(a, np.float32)
    extra = (-a.shape[-1]) % 8 or 8
    pad = np.full(a.shape[:-1] + (extra,), np.nan, np.float32)
    return np.concatenate([a, pad], axis=-1)


def gpu_run(mode, batch, **kw):
    out = sdv.verify(mode, batch.target, batch.draft, batch.tokens, batch.lengths, batch.accept_u,
                     batch.sample_u, batch.temperature, V=batch.V, **kw)
    torch.cuda.synchronize()
    return {k: (None if v is None else v.cpu().numpy()) for k, v in out.items()}


# Per workload: comparisons, requests, decisions, near-margin decisions
# (|u - threshold| < MARGIN) and mismatches, over every comparison made
# with that workload label in this test session.  conftest.py prints it at
# the end and fails the session if a workload's mismatches reach 1e-4 of
# its decisions.
LEDGER = {}
SMALL = "small cases"


def ledger_violations():
    """Workloads whose mismatches are not below 1e-4 of their decisions."""
    return {k: v for k, v in LEDGER.items() if v["mismatches"] and not v["mismatches"] < 1e-4 * v["decisions"]}


def oracle_run(mode, batch, requests=None, residual_out=False):
    """Oracle on all requests, or on the listed ones (host copies of their
    slabs), spread over the host's cores."""
    idx = list(range(batch.B)) if requests is None else list(requests)
    if requests is None:
        take = lambda t: None if t is None else t.cpu()
    else:
        sel = torch.as_tensor(idx, dtype=torch.long, device=batch.target.device)
        take = lambda t: None if t is None else t.index_select(0, sel).cpu()
    prob = oracle.Problem(take(batch.target), take(batch.draft), take(batch.tokens), take(batch.lengths),
                          take(batch.accept_u), take(batch.sample_u), batch.temperature, V=batch.V)
    ref = oracle.verify_threads(mode, prob, residual_out=residual_out)
    ref["mode"] = mode
    ref["requests"] = idx
    ref["prob"] = prob
    return ref


def _softmax64(row, T):
    x = np.asarray(row, np.float64) / T
    x = np.exp(x - x.max())
    return x / x.sum()


def kseq_gamma(beta, n):
    beta = min(max(float(beta), 0.0), 1.0)
    return -np.expm1(n * np.log1p(-beta)) / beta if beta > 0 else float(n)


def kseq_reachable(P, Q, n, eps=KSEQ_FLAT):
    """Every rho the K-SEQ search (as include/sdv.h states it: rho = 1 if
    gamma(1) <= 1, else 10 rounds over [lo, hi] = [1, n] testing
    lo + (hi - lo) i / 4, i = 1..3, keeping the quarter that ends at the
    first point to pass, the last quarter if none does; rho = the final hi)
    can end at when a test whose two sides lie within eps of each other
    (relative) may go either way.  fp64; returns a sorted list."""
    seen = {}

    def outcomes(r):
        if r not in seen:
            g = kseq_gamma(np.minimum(Q, P / r).sum(), n)
            seen[r] = {True, False} if abs(g - r) < eps * r else {bool(g <= r)}
        return seen[r]

    ends = set()
    if True in outcomes(1.0):
        ends.add(1.0)
    if False not in outcomes(1.0):
        return sorted(ends)
    states = {(1.0, float(n))}
    for _ in range(10):
        nxt = set()
        for lo, hi in states:
            pts = [lo + (hi - lo) * i / 4.0 for i in (1, 2, 3)]
            for i, r in enumerate(pts):
                res = outcomes(r)
                if True in res:
                    nxt.add((lo if i == 0 else pts[i - 1], r))
                if False not in res:
                    break
            else:
                nxt.add((pts[2], hi))
        states = nxt
    return sorted(ends | {hi for _, hi in states})


def _kseq_node_ok(prob, i, j, ks, a_gpu, what):
    """A K-SEQ node whose acceptance probabilities differ from the oracle's:
    they must all follow, within TOL, from one rho the search can end at
    when its tests within KSEQ_FLAT of their threshold go either way."""
    T, V = prob.temperature, prob.V
    o = ks[0]
    row = lambda a, jj: (a[i, o, jj, :V].view(np.uint16).astype(np.uint32) << 16).view(np.float32) \
        if prob.dtype == oracle.BF16 else a[i, o, jj, :V]
    P, Q = _softmax64(row(prob.target, j), T), _softmax64(row(prob.draft, j), T)
    ys = [int(prob.tokens[i, k, j]) for k in ks]
    ends = kseq_reachable(P, Q, len(ks))
    err = lambda rho: max(abs(a - (min(1.0, P[y] / (rho * Q[y])) if Q[y] > 0 else 1.0)) for y, a in zip(ys, a_gpu))
    best = min(ends, key=err)
    assert err(best) <= TOL, f"{what}: no search end explains the GPU's values (best rho {best}, off {err(best):.3g})"


def _kseq_nodes(gpu, ref, i, b, what):
    """Compare one K-SEQ request's acceptance probabilities node by node;
    returns the flat-zone nodes found (see KSEQ_FLAT)."""
    prob = ref["prob"]
    tok = prob.tokens[i]
    Lb = int(prob.lengths[i]) if prob.lengths is not None else prob.L
    flat = set()
    for j in range(Lb):
        groups = {}
        for k in range(prob.K):
            o = min(k2 for k2 in range(prob.K) if (tok[k2, :j] == tok[k, :j]).all())
            groups.setdefault(o, []).append(k)
        for o, ks in groups.items():
            a_gpu = [float(gpu["accept_prob"][b, k, j]) for k in ks]
            a_ref = [float(ref["accept_prob"][i, k, j]) for k in ks]
            if max(abs(x - y) for x, y in zip(a_gpu, a_ref)) > TOL:
                _kseq_node_ok(prob, i, j, ks, a_gpu, f"{what} request {b} node ({j}, {o})")
                flat.add((j, o))
    return flat


def compare(gpu, ref, what="", workload=SMALL):
    """Check the GPU's outputs against the oracle's (bar in the module
    docstring) and add the comparison to LEDGER[workload].  Returns the
    number of near-margin mismatches."""
    idx = ref["requests"]
    kseq = ref.get("mode") == "kseq"
    mism = flat_nodes = 0
    status_or = 0
    for i, b in enumerate(idx):
        st = int(ref["req_status"][i])
        status_or |= st
        if st:
            assert gpu["out_token"][b] == -1 and gpu["accept_len"][b] == 0, f"{what} request {b}: status {st}"
            continue
        flat = _kseq_nodes(gpu, ref, i, b, what) if kseq and gpu.get("accept_prob") is not None else set()
        flat_nodes += len(flat)
        same = (gpu["accept_len"][b] == ref["accept_len"][i] and gpu["accept_draft"][b] == ref["accept_draft"][i]
                and gpu["out_token"][b] == ref["out_token"][i])
        if not same:
            assert ref["margin"][i] < MARGIN, (
                f"{what} request {b}: gpu ({gpu['accept_len'][b]}, {gpu['accept_draft'][b]}, "
                f"{gpu['out_token'][b]}) oracle ({ref['accept_len'][i]}, {ref['accept_draft'][i]}, "
                f"{ref['out_token'][i]}) margin {ref['margin'][i]:.3g}")
            mism += 1
        elif gpu.get("residual_mass") is not None and (int(gpu["accept_len"][b]), int(gpu["accept_draft"][b])) \
                not in flat:
            d = abs(float(gpu["residual_mass"][b]) - float(ref["residual_mass"][i]))
            assert d <= TOL, f"{what} request {b}: residual_mass off by {d:.3g}"
        if gpu.get("accept_prob") is not None and not kseq:
            d = np.max(np.abs(gpu["accept_prob"][b] - ref["accept_prob"][i]), initial=0.0)
            assert d <= TOL, f"{what} request {b}: accept_prob off by {d:.3g}"
    if len(idx) == len(gpu["out_token"]):
        assert int(gpu["device_status"][0]) == status_or, f"{what}: device status {gpu['device_status'][0]}"
    # a decision within 1e-5 of its threshold is settled by fp32 rounding
    # (the kernel's summation order): such mismatches are counted against
    # the workload's decisions
    e = LEDGER.setdefault(workload, dict(comparisons=0, requests=0, decisions=0, near_margin=0, mismatches=0,
                                         kseq_flat_zone=0))
    e["kseq_flat_zone"] += flat_nodes
    e["comparisons"] += 1
    e["requests"] += len(idx)
    e["decisions"] += int(np.maximum(ref["decisions"], 1).sum()) if len(idx) else 0
    e["near_margin"] += int(ref["near_margin"].sum()) if len(idx) else 0
    e["mismatches"] += mism
    return mism


def compare_residual_rows(gpu, ref, what=""):
    """residual_out: the normalised distribution each request's correction
    was drawn from, element by element within TOL (fp32 against the
    oracle's fp64), where the decision agrees (else the rows belong to
    different end nodes); an invalid request's row is zero.  Returns the
    largest difference seen and the number of rows compared."""
    worst, n = 0.0, 0
    rows = gpu["residual_out"]
    for i, b in enumerate(ref["requests"]):
        if int(ref["req_status"][i]):
            assert not np.any(rows[b]), f"{what} request {b}: an invalid request's row is not zero"
            continue
        if not (gpu["accept_len"][b] == ref["accept_len"][i] and gpu["accept_draft"][b] == ref["accept_draft"][i]):
            continue
        d = float(np.max(np.abs(rows[b].astype(np.float64) - ref["residual_out"][i]), initial=0.0))
        worst = max(worst, d)
        n += 1
        assert d <= TOL, f"{what} request {b}: residual_out off by {d:.3g}"
    return worst, n


def pattern_row(kind, V):
    """Degenerate logit rows (kinds 0..6) for the online-maximum and masking
    paths; a float32 tensor of V logits."""
    x = np.arange(V, dtype=np.float64)
    if kind == 0:      # every logit equal: the maximum ties everywhere
        r = np.full(V, 1.5)
    elif kind == 1:    # ascending: every chunk holds a new maximum
        r = 8.0 * x / V
    elif kind == 2:    # descending: the maximum at index 0
        r = 8.0 - 8.0 * x / V
    elif kind == 3:    # flat with one spike at the last index
        r = np.zeros(V)
        r[-1] = 6.0
    elif kind == 4:    # two equal maxima far apart, a wavy floor
        r = np.sin(x * 0.37)
        r[3] = r[-5] = 5.0
    elif kind == 5:    # the first half masked to -inf, as a filtered vocabulary
        r = np.sin(x * 0.11) * 2.0
        r[: V // 2] = -np.inf
    else:              # top-3 filtering: three finite logits, the rest -inf
        r = np.full(V, -np.inf)
        r[[V // 7, V // 2, V - 2]] = [1.0, 2.5, 0.5]
    return torch.as_tensor(r, dtype=torch.float32)
