"""GPU LM head and greedy verification fused into it (through the C-ABI),
against the oracle.

The oracle computes the target model's logits = hidden . W^T in double and
applies the greedy rule to them ("Speculative Decoding: Performance or
Illusion?", section 3.2: the target model's pass is the verification step).
The GPU sums the d products of each logit in fp32 on the tensor cores, in
the hardware's order, so a logit may differ from the exact sum by at most
the classic bound for a sum of d terms, gamma_d * sum_i |h_i w_i| with
gamma_d ~ d * 2^-24; the tests allow four times that, ERR = d * 2^-22.
Where floating point decides an integer (a row's argmax), a decision is
compared only where it is unique: the oracle's top two logits of every row
the request reads lie more than twice the error allowance apart.
Integer-valued inputs make every logit exact on both sides, so those cases
(including ties, lowest index first) must match bit for bit.
"""
import numpy as np
import pytest
import torch

import draft_verification_row_gb300 as sdv
import oracle
from draft_verification_row_gb300 import workloads as W

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
WL = W.LM_HEAD_HEADLINE


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


@pytest.fixture(autouse=True, params=["cta_pair", "one_cta"])
def lm_form(request):
    """Every test runs on both forms of the LM-head kernel: CTA pairs
    (tcgen05 cta_group::2, the default where a cluster of two CTAs fits) and
    one CTA per tile (the fallback), chosen through the library's test hook."""
    from draft_verification_row_gb300 import binding
    h = binding.lib()
    assert h.sdv_testing_set_lm_head_single_cta(1 if request.param == "one_cta" else 0) == 0
    yield request.param
    h.sdv_testing_set_lm_head_single_cta(0)


def _err_bound(hidden, lm_head):
    """Per-logit error allowance d * 2^-22 * sum_i |h_i w_i| (numpy, float64)."""
    h = np.abs(hidden.to(torch.float64).numpy())
    w = np.abs(lm_head.to(torch.float64).numpy())
    return h.shape[-1] * 2.0 ** -22 * np.einsum("...i,xi->...x", h, w)


def _hw(M, V, d, seed, integer=0, scale=1.0):
    g = torch.Generator(device=DEV)
    g.manual_seed(seed)
    if integer:
        h = torch.randint(-integer, integer + 1, (M, d), generator=g, device=DEV)
        w = torch.randint(-integer, integer + 1, (V, d), generator=g, device=DEV)
    else:
        h = torch.randn((M, d), generator=g, device=DEV)
        w = torch.randn((V, d), generator=g, device=DEV) * scale
    return h.to(torch.bfloat16).contiguous(), w.to(torch.bfloat16).contiguous()


# ------------------------------------------------------------------ the LM head

@pytest.mark.parametrize("M,V,d", [(1, 8, 8), (130, 1000, 136), (300, 3001, 200), (257, 513, 64), (64, 300, 1032)])
def test_lm_head_logits_within_the_error_bound(M, V, d):
    h, w = _hw(M, V, d, seed=M + V + d, scale=3.0 / d ** 0.5)
    stride = (V + 3) // 4 * 4 + 4
    out = torch.full((M, stride), float("nan"), device=DEV)
    logits, status = sdv.lm_head_logits(h, w, logits=out)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    got = logits.cpu().numpy()
    ref = oracle.lm_head_logits(h.cpu(), w.cpu())
    bound = _err_bound(h.cpu(), w.cpu())
    err = np.abs(got[:, :V].astype(np.float64) - ref)
    assert (err <= bound).all(), f"max err {err.max()} (bound there {bound.flat[err.argmax()]})"
    assert np.isnan(got[:, V:]).all(), "columns past V were written"


def test_lm_head_logits_exact_on_integers():
    # integer inputs: every partial sum is an integer below 2^24, exact in fp32
    M, V, d = 300, 1000, 136
    h, w = _hw(M, V, d, seed=3, integer=8)
    logits, status = sdv.lm_head_logits(h, w)
    torch.cuda.synchronize()
    ref = oracle.lm_head_logits(h.cpu(), w.cpu())
    assert int(status.item()) == 0
    assert np.array_equal(logits.cpu().numpy().astype(np.float64), ref)


def test_lm_head_logits_empty_and_bad_arguments():
    h, w = _hw(4, 16, 8, seed=4)
    logits, status = sdv.lm_head_logits(h[:0], w)
    torch.cuda.synchronize()
    assert logits.shape == (0, 16) and int(status.item()) == 0
    with pytest.raises(sdv.SDVError):  # d not a multiple of 8
        hh, ww = _hw(4, 16, 12, seed=5)
        sdv.lm_head_logits(hh, ww)
    with pytest.raises(sdv.SDVError):  # row stride not a multiple of 4
        sdv.lm_head_logits(h, w, logits=torch.empty((4, 18), device=DEV)[:, :17])


# ------------------------------------------------------------- fused greedy

def _read_rows(tokens, lengths, L):
    """[B][K][L+1] mask of the rows a request reads: depths 0..L_b, the
    lowest draft of each distinct prefix."""
    B, K = tokens.shape[:2]
    m = np.zeros((B, K, L + 1), bool)
    for b in range(B):
        if not 0 <= lengths[b] <= L:
            continue
        for j in range(lengths[b] + 1):
            for k in range(K):
                m[b, k, j] = not any((tokens[b, k2, :j] == tokens[b, k, :j]).all() for k2 in range(k))
    return m


def _oracle(batch, exact=False):
    """Oracle greedy outputs on the exact logits, and per request whether
    every row it reads has a unique argmax under the error allowance."""
    host = batch.to("cpu")
    lg = oracle.lm_head_logits(host.hidden, host.lm_head)
    ref = oracle.verify("greedy", oracle.Problem(lg, None, host.tokens, host.lengths, None, None, 0.0, V=host.V))
    unique = np.ones(batch.B, bool)
    if not exact:
        bound = _err_bound(host.hidden, host.lm_head)
        top2 = np.sort(np.nan_to_num(lg, nan=-np.inf), axis=-1)[..., -2:]
        with np.errstate(invalid="ignore", over="ignore"):  # NaN or Inf rows
            ok = top2[..., 1] - top2[..., 0] > 2 * np.nan_to_num(bound, nan=0.0).max(axis=-1)  # [B][K][L+1]
        ok |= ~np.isfinite(lg).all(axis=-1)  # an unusable row decides by its status, not its argmax
        read = _read_rows(host.tokens.numpy(), host.lengths.numpy(), batch.L)
        unique = (ok | ~read).all(axis=(1, 2))
    return ref, unique


def _compare(batch, got, ref, unique, what):
    keys = ("accept_len", "accept_draft", "out_token")
    g = {k: got[k].cpu().numpy() for k in keys + ("accept_prob",)}
    for b in range(batch.B):
        same = all(g[k][b] == ref[k][b] for k in keys) and np.array_equal(g["accept_prob"][b], ref["accept_prob"][b])
        assert same or not unique[b], f"{what}: request {b} differs: " + str(
            {k: (g[k][b], ref[k][b]) for k in keys})
    assert (~unique).sum() <= max(1, 1e-3 * batch.B), f"{what}: {(~unique).sum()} ambiguous requests"


def _run(batch):
    out = sdv.verify_greedy_lm_head(batch.hidden, batch.lm_head, batch.tokens, batch.lengths)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("B,K,L,V,d", [(8, 4, 4, 3001, 200), (3, 1, 5, 257, 64), (16, 8, 3, 1500, 72)])
def test_fused_greedy_matches_the_oracle(B, K, L, V, d):
    batch = W.make_lm_head(WL, DEV, B=B, K=K, L=L, V=V, d=d, poison_unread=True)
    got = _run(batch)
    ref, unique = _oracle(batch)
    assert int(got["device_status"].item()) == 0
    _compare(batch, got, ref, unique, f"B{B} K{K} L{L} V{V} d{d}")


def test_fused_greedy_at_the_maximum_sizes():
    # K = 16 drafts of L = 16 tokens: up to 272 trie nodes per request
    batch = W.make_lm_head(WL, DEV, B=4, K=16, L=16, V=1000, d=64, agree=0.9, poison_unread=True)
    got = _run(batch)
    ref, unique = _oracle(batch)
    assert int(got["device_status"].item()) == 0
    _compare(batch, got, ref, unique, "K16 L16")
    assert (got["accept_len"].cpu().numpy() > 4).any()  # long accepted runs happen


def test_fused_greedy_ties_across_tiles_take_the_lowest_index():
    # integer logits in -64..64 over 1500 entries: the maximum repeats in about
    # a quarter of the rows, mostly in different 256-wide vocabulary tiles;
    # several 128-row tiles of nodes
    batch = W.make_lm_head(WL, DEV, B=40, K=4, L=4, V=1500, d=64, integer=1, agree=0.8)
    got = _run(batch)
    ref, unique = _oracle(batch, exact=True)
    host = batch.to("cpu")
    lg = oracle.lm_head_logits(host.hidden, host.lm_head)
    assert ((lg == lg.max(axis=-1, keepdims=True)).sum(axis=-1) > 1).mean() > 0.15  # ties are common
    assert int(got["device_status"].item()) == 0
    _compare(batch, got, ref, unique, "integer ties")


def test_fused_greedy_edge_cases():
    V, d = 700, 64
    # lengths 0 (only the context row is read) and L = 0
    batch = W.make_lm_head(WL, DEV, B=5, K=3, L=3, V=V, d=d, lengths=[0, 3, 1, 0, 2], poison_unread=True)
    ref, unique = _oracle(batch)
    _compare(batch, _run(batch), ref, unique, "zero lengths")
    batch = W.make_lm_head(WL, DEV, B=4, K=2, L=0, V=V, d=d)
    ref, unique = _oracle(batch)
    got = _run(batch)
    _compare(batch, got, ref, unique, "L = 0")
    assert (got["accept_len"].cpu().numpy() == 0).all()
    # B = 0
    batch = W.make_lm_head(WL, DEV, B=0, K=2, L=2, V=V, d=d)
    got = _run(batch)
    assert int(got["device_status"].item()) == 0
    # invalid requests leave the others alone
    batch = W.make_lm_head(WL, DEV, B=6, K=2, L=3, V=V, d=d, lengths=[3, 3, 3, 2, 3, 1])
    batch.lengths[2] = 4                    # bad length
    batch.tokens[3, 1, 0] = V               # bad token
    batch.hidden[4, 0, 0, 5] = float("nan")  # the context row of request 4
    got = _run(batch)
    st = int(got["device_status"].item())
    assert st == 1 | 2 | 4
    al, ot = got["accept_len"].cpu().numpy(), got["out_token"].cpu().numpy()
    assert (ot[[2, 3, 4]] == -1).all() and (al[[2, 3, 4]] == 0).all()
    keep = [0, 1, 5]
    sub = W.LmHeadBatch(name="sub", B=3, K=2, L=3, V=V, d=d, hidden=batch.hidden[keep], lm_head=batch.lm_head,
                        tokens=batch.tokens[keep], lengths=batch.lengths[keep])
    ref, unique = _oracle(sub)
    for i, b in enumerate(keep):
        if unique[i]:
            assert (al[b], ot[b]) == (ref["accept_len"][i], ref["out_token"][i])


def test_fused_greedy_reads_only_the_leaves_it_ends_at():
    # leaves are computed only where the decision ends there: poisoning the
    # others changes nothing; poisoning those makes just their requests invalid
    V, d = 1000, 64
    batch = W.make_lm_head(WL, DEV, B=12, K=3, L=3, V=V, d=d, agree=0.6, poison_unread=True)
    clean = {k: v.cpu().numpy() for k, v in _run(batch).items() if v is not None}
    lens = batch.lengths.cpu().numpy()
    tok = batch.tokens.cpu().numpy()
    ends = []  # requests whose decision ends at a leaf, with that leaf's draft
    for b in range(batch.B):
        if clean["accept_len"][b] == lens[b]:
            ks = int(clean["accept_draft"][b])
            ends.append((b, min(k2 for k2 in range(batch.K) if (tok[b, k2, :lens[b]] == tok[b, ks, :lens[b]]).all())))
    assert 0 < len(ends) < batch.B
    end_set = set(ends)
    for b in range(batch.B):
        for k in range(batch.K):
            if (b, k) not in end_set:
                batch.hidden[b, k, lens[b]] = float("nan")
    got = _run(batch)
    assert int(got["device_status"].item()) == 0
    for key in ("accept_len", "accept_draft", "out_token", "accept_prob"):
        assert np.array_equal(got[key].cpu().numpy(), clean[key]), key
    for b, k in ends:
        batch.hidden[b, k, lens[b], 3] = float("inf")
    got = _run(batch)
    ref, unique = _oracle(batch)
    _compare(batch, got, ref, unique, "poisoned end leaves")
    assert int(got["device_status"].item()) == 4
    ot = got["out_token"].cpu().numpy()
    for b in range(batch.B):
        assert (ot[b] == -1) == (b in {e[0] for e in ends})


def test_fused_greedy_is_deterministic():
    batch = W.make_lm_head(WL, DEV, B=16, K=4, L=4, V=2000, d=128)
    a = {k: v.cpu() for k, v in _run(batch).items() if v is not None}
    for _ in range(3):
        b = {k: v.cpu() for k, v in _run(batch).items() if v is not None}
        for k in a:
            assert torch.equal(a[k], b[k]), k


def test_fused_greedy_full_size_sampled():
    # the bench's workload at full size; one request of length 1 against the
    # oracle (its 2 * K rows in double cost ~10 s on one core), the rest by
    # properties that hold at any size
    batch = W.make_lm_head(WL, DEV)
    got = _run(batch)
    assert int(got["device_status"].item()) == 0
    lens = batch.lengths.cpu().numpy()
    al, ad, ot = (got[k].cpu().numpy() for k in ("accept_len", "accept_draft", "out_token"))
    assert ((al >= 0) & (al <= lens)).all() and ((ad >= 0) & (ad < batch.K)).all()
    assert ((ot >= 0) & (ot < batch.V)).all()
    assert 0 < al.mean() < lens.mean()  # drafts agree often, not always
    b = int(np.flatnonzero(lens == 1)[0])
    sub = W.LmHeadBatch(name="sub", B=1, K=batch.K, L=1, V=batch.V, d=batch.d,
                        hidden=batch.hidden[b:b + 1, :, :2].contiguous(), lm_head=batch.lm_head,
                        tokens=batch.tokens[b:b + 1, :, :1].contiguous(), lengths=batch.lengths[b:b + 1])
    host = sub.to("cpu")
    lg = oracle.lm_head_logits(host.hidden, host.lm_head)
    ref = oracle.verify("greedy", oracle.Problem(lg, None, host.tokens, host.lengths, None, None, 0.0, V=sub.V))
    # the GPU's own logits of these rows, as the fused kernel sums them
    gl, _ = sdv.lm_head_logits(sub.hidden.view(-1, sub.d), sub.lm_head)
    gl = gl.cpu().numpy().astype(np.float64).reshape(lg.shape)
    err = np.abs(gl - lg).max(axis=-1)
    top2 = np.sort(lg, axis=-1)[..., -2:]
    unique = (top2[..., 1] - top2[..., 0] > 2 * err).all()
    if unique:
        assert (al[b], ad[b], ot[b]) == (ref["accept_len"][0], ref["accept_draft"][0], ref["out_token"][0])
    # whatever the margins: the fused decision is the greedy rule on the GPU's own logits
    am = gl.argmax(axis=-1)[0]  # [K][2], first maximum
    best = max(range(batch.K), key=lambda k: (int(sub.tokens[0, k, 0].item()) == am[k, 0], -k))
    m = int(int(sub.tokens[0, best, 0].item()) == am[best, 0])
    assert (al[b], ad[b], ot[b]) == (m, best, am[best, m])


def test_trie_logits_for_the_sampling_rules():
    # every trie node's row, leaves included, written once in bf16 into the
    # verification layout: within bf16 rounding (2^-9 relative) of the fp32
    # sum, itself within the summation allowance of the exact logits; every
    # other row and the padding stay untouched
    B, K, L, V, d = 7, 4, 3, 1003, 136
    batch = W.make_lm_head(WL, DEV, B=B, K=K, L=L, V=V, d=d, poison_unread=True)
    batch.lengths[6] = L + 1  # an invalid request: its rows are not written
    target, status = sdv.lm_head_trie_logits(batch.hidden, batch.lm_head, batch.tokens, batch.lengths)
    torch.cuda.synchronize()
    assert int(status.item()) == 1
    host = batch.to("cpu")
    ref = oracle.lm_head_logits(host.hidden, host.lm_head)
    bound = _err_bound(host.hidden, host.lm_head)
    got = target.float().cpu().numpy()
    assert np.isnan(got[..., V:]).all()
    read = _read_rows(host.tokens.numpy(), host.lengths.numpy(), L)
    assert not read[6].any() and read.sum() > B * 2
    for b in range(B):
        for k in range(K):
            for j in range(L + 1):
                g = got[b, k, j, :V]
                if not read[b, k, j]:
                    assert np.isnan(g).all(), (b, k, j)
                    continue
                tol = bound[b, k, j] + 2.0 ** -8 * np.abs(ref[b, k, j]) + 1e-30
                assert (np.abs(g - ref[b, k, j]) <= tol).all(), (b, k, j)
