"""GPU-versus-oracle comparison rules.

Bar (per request): accept_len, accept_draft and out_token equal the
oracle's, except where some decision on the oracle's path had a margin
|u - threshold| (or distance of u to its CDF interval's ends) below 1e-5;
such mismatches are counted and must stay at one per comparison or under
1e-4 of all decisions, whichever is larger.
accept_prob within 1e-5 absolute everywhere (1e-4 for K-SEQ, whose rho
comes from a search; see TOL_KSEQ); residual_mass within 1e-5 where the
end node agrees.  Requests the oracle marks invalid must come back
invalid with the same status bit.
"""
import numpy as np
import torch

import draft_verification_row_gb300 as sdv
import oracle

TOL = 1e-5
MARGIN = 1e-5
# K-SEQ's acceptance probabilities min(1, P(y) / (rho Q(y))) carry rho from
# a search whose test gamma(beta(rho)) <= rho is evaluated with an fp32
# vocabulary sum on the GPU (relative error ~1e-6) and in fp64 by the
# oracle.  Both test the same dyadic points, but near the crossing the two
# can decide differently and end on opposite sides of it; rho then differs
# by the width of that zone, about 1e-6 / |1 - d gamma / d rho|, which a
# flat crossing widens.  The emitted token follows P for either rho.
TOL_KSEQ = 1e-4


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


def oracle_run(mode, batch, requests=None):
    """Oracle on all requests, or on the listed ones (host copies of their slabs)."""
    idx = list(range(batch.B)) if requests is None else list(requests)
    sel = torch.as_tensor(idx, dtype=torch.long, device=batch.target.device)

    def take(t):
        return None if t is None else t.index_select(0, sel).cpu()

    prob = oracle.Problem(take(batch.target), take(batch.draft), take(batch.tokens), take(batch.lengths),
                          take(batch.accept_u), take(batch.sample_u), batch.temperature, V=batch.V)
    ref = oracle.verify(mode, prob, trace_cap=1 << 20)
    ref["mode"] = mode
    ref["decisions"] = len(ref["trace"]) + len(idx)
    ref["requests"] = idx
    return ref


def compare(gpu, ref, what=""):
    idx = ref["requests"]
    ap_tol = TOL_KSEQ if ref.get("mode") == "kseq" else TOL
    mism = 0
    status_or = 0
    for i, b in enumerate(idx):
        st = int(ref["req_status"][i])
        status_or |= st
        if st:
            assert gpu["out_token"][b] == -1 and gpu["accept_len"][b] == 0, f"{what} request {b}: status {st}"
            continue
        same = (gpu["accept_len"][b] == ref["accept_len"][i] and gpu["accept_draft"][b] == ref["accept_draft"][i]
                and gpu["out_token"][b] == ref["out_token"][i])
        if not same:
            assert ref["margin"][i] < MARGIN, (
                f"{what} request {b}: gpu ({gpu['accept_len'][b]}, {gpu['accept_draft'][b]}, "
                f"{gpu['out_token'][b]}) oracle ({ref['accept_len'][i]}, {ref['accept_draft'][i]}, "
                f"{ref['out_token'][i]}) margin {ref['margin'][i]:.3g}")
            mism += 1
        elif gpu.get("residual_mass") is not None:
            d = abs(float(gpu["residual_mass"][b]) - float(ref["residual_mass"][i]))
            assert d <= TOL, f"{what} request {b}: residual_mass off by {d:.3g}"
        if gpu.get("accept_prob") is not None:
            d = np.max(np.abs(gpu["accept_prob"][b] - ref["accept_prob"][i]), initial=0.0)
            assert d <= ap_tol, f"{what} request {b}: accept_prob off by {d:.3g}"
    # a decision within 1e-5 of its threshold is decided by fp32 rounding
    # (the kernel's summation order): one such flip per comparison is
    # allowed, or 1e-4 of the decisions on large ones
    assert mism <= max(1.0, 1e-4 * ref["decisions"]), f"{what}: {mism} near-margin mismatches of {ref['decisions']}"
    if len(idx) == len(gpu["out_token"]):
        assert int(gpu["device_status"][0]) == status_or, f"{what}: device status {gpu['device_status'][0]}"
    return mism


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
