"""CUDA path against the oracle through the C-ABI (needs a GB300)."""
import os

import numpy as np
import pytest
import torch

import draft_verification_row_gb300 as sdv
from draft_verification_row_gb300 import binding
from draft_verification_row_gb300 import workloads as W
from tests import goldens
from tests import parity as P

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
MODES_K1 = ["token", "block", "multidraft", "greedy"]
MODES_K = ["token", "multidraft", "greedy"]


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _modes(batch):
    return MODES_K1 if batch.K == 1 else MODES_K


GOLDEN = goldens.cases()


@pytest.mark.parametrize("case", GOLDEN, ids=[c["name"] for c in GOLDEN])
def test_worked_examples(case):
    dev = torch.device(DEV)
    t = lambda a: None if a is None else torch.as_tensor(a).to(dev)
    out = P.sdv.verify(case["mode"], t(P.pad8(case["target"])), t(P.pad8(case["draft"])), t(case["tokens"]),
                       t(case["lengths"]), t(case["accept_u"]), t(case["sample_u"]), case["T"],
                       V=case["V"])
    torch.cuda.synchronize()
    e = case["expected"]
    assert int(out["device_status"][0]) == 0
    assert int(out["accept_len"][0]) == e["accept_len"]
    assert int(out["accept_draft"][0]) == e["accept_draft"]
    assert int(out["out_token"][0]) == e["out_token"]
    np.testing.assert_allclose(out["accept_prob"][0].cpu().numpy(), np.asarray(e["accept_prob"]), atol=1e-6)
    assert abs(float(out["residual_mass"][0]) - e["residual_mass"]) < 1e-6


# small shapes of every workload: several tiles, a ragged vocabulary tail
SMALL = [
    ("token-B4-K1-L4-V1024-f32", dict(B=6, V=1021), None),
    ("token-greedy-B64-K1-L5-V32000-bf16", dict(B=6, V=3001), 1.0),
    ("token-greedy-B64-K1-L5-V32000-bf16", dict(B=6, V=3001), 0.0),
    ("block-B128-K1-L5-V128256-bf16", dict(B=6, V=12829), None),
    ("multidraft-B32-K4-L4-V32000-f32", dict(B=6, V=3203), 0.1),
    ("multidraft-B32-K4-L4-V32000-f32", dict(B=6, V=3203), 0.7),
    ("mixed-B256-K8-L8-V151936-bf16", dict(B=6, V=15197), None),
]


# Without accept_prob the block rules skip the last sweep of a node whose
# test must fail (and of the root): every comparison of those rules is also
# made without it.
LAZY = ("block", "multidraft")


def _compare_both(mode, batch, ref, what, **kw):
    P.compare(P.gpu_run(mode, batch), ref, what, **kw)
    if mode in LAZY:
        P.compare(P.gpu_run(mode, batch, accept_prob=False), ref, what + " (no accept_prob)", **kw)


@pytest.mark.parametrize("name,kw,T", SMALL)
def test_small_parity(name, kw, T):
    batch = W.make(name, DEV, temperature=T, **kw)
    # (K-SEQ at low temperature: test_kseq_low_temperature_rho_is_valid)
    for mode in _modes(batch) + (["kseq"] if batch.temperature >= 0.4 else []):
        _compare_both(mode, batch, P.oracle_run(mode, batch), f"{name}/{mode}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("V", [1, 2, 7, 8, 9, 33, 1000, 4097])
def test_vocabulary_edges(dtype, V):
    batch = W.make("multidraft-B32-K4-L4-V32000-f32", DEV, B=4, K=3, L=3, V=V, dtype=dtype, temperature=0.9)
    for mode in MODES_K + ["kseq"]:
        _compare_both(mode, batch, P.oracle_run(mode, batch), f"V={V}/{mode}")


def test_max_drafts_and_length():
    batch = W.make("mixed-B256-K8-L8-V151936-bf16", DEV, B=3, K=16, L=16, V=2053, temperature=1.5)
    for mode in MODES_K + ["kseq"]:
        _compare_both(mode, batch, P.oracle_run(mode, batch), f"K16L16/{mode}")


@pytest.mark.parametrize("lengths", [[0, 0, 0], [0, 3, 1], [3, 3, 3]])
def test_ragged_and_empty_lengths(lengths):
    batch = W.make("multidraft-B32-K4-L4-V32000-f32", DEV, B=3, K=4, L=3, V=999, lengths=lengths,
                   temperature=0.7)
    for mode in MODES_K:
        P.compare(P.gpu_run(mode, batch), P.oracle_run(mode, batch), f"{lengths}/{mode}")


def test_empty_draft_dimension():
    batch = W.make("token-B4-K1-L4-V1024-f32", DEV, B=5, L=0, V=777)
    for mode in MODES_K1:
        P.compare(P.gpu_run(mode, batch), P.oracle_run(mode, batch), f"L=0/{mode}")


def test_empty_batch():
    batch = W.make("token-B4-K1-L4-V1024-f32", DEV, B=0)
    out = P.gpu_run("token", batch)
    assert out["accept_len"].shape == (0,)
    assert int(out["device_status"][0]) == 0


@pytest.mark.parametrize("name", ["mixed-B256-K8-L8-V151936-bf16", "multidraft-B32-K4-L4-V32000-f32"])
def test_unread_rows_are_never_read(name):
    """Rows past a request's length, duplicate-prefix copies, stride padding
    and padding tokens hold NaN / -1: the outputs must not change."""
    kw = dict(B=5, V=4001, stride_pad=8)
    clean = W.make(name, DEV, **kw)
    dirty = W.make(name, DEV, poison_unread=True, **kw)
    for mode in MODES_K:
        a, b = P.gpu_run(mode, clean), P.gpu_run(mode, dirty)
        assert int(b["device_status"][0]) == 0
        for key in ("accept_len", "accept_draft", "out_token", "accept_prob", "residual_mass"):
            np.testing.assert_array_equal(a[key], b[key])


def test_invalid_requests_are_isolated():
    batch = W.make("multidraft-B32-K4-L4-V32000-f32", DEV, B=6, K=3, L=3, V=1500, temperature=0.7)
    batch.target[1, 0, 0, 17] = float("nan")          # used row of request 1
    batch.draft[2, 0, 0, 3] = float("inf")            # used draft row of request 2
    batch.tokens[3, 1, 0] = batch.V                   # used token out of range
    batch.lengths[4] = 4                              # length > L
    batch.target[5, 0, 0, :] = float("-inf")          # no finite value
    for mode in MODES_K:
        ref = P.oracle_run(mode, batch)
        _compare_both(mode, batch, ref, f"invalid/{mode}")
        gpu = P.gpu_run(mode, batch)
        st = ref["req_status"]
        assert st[0] == 0 and st[3] == 2 and st[4] == 1
        assert st[1] == 4 and st[5] == 4
        assert st[2] == (0 if mode == "greedy" else 4)


@pytest.mark.parametrize("name,K", [("multidraft-B32-K4-L4-V32000-f32", 3), ("block-B128-K1-L5-V128256-bf16", 1)])
def test_leaf_rows_are_read_only_by_the_bonus_draw(name, K):
    """A leaf's target row enters only the bonus draw, made when the decision
    ends there.  Requests 0-2 accept everything (accept_u = 0: the decision
    ends at draft 0's leaf); the others mostly stop short (accept_u = 0.999;
    a draw still passes where a = 1).  Every leaf row is poisoned except
    draft 0's in requests 0 and 1.  A request whose clean decision stops
    short of its leaves must come back unchanged; one that ends at a leaf,
    invalid.  Greedy, too, reads a leaf only where its decision ends."""
    lengths = [3, 2, 3, 3, 1, 2, 3, 3, 2, 3]
    batch = W.make(name, DEV, B=len(lengths), K=K, L=3, V=2003, lengths=lengths, temperature=0.8)
    batch.accept_u[:3] = 0.0
    batch.accept_u[3:] = 0.999
    modes = ["token", "multidraft", "greedy", "kseq"] if K > 1 else ["token", "block", "greedy", "kseq"]
    clean = {mode: P.oracle_run(mode, batch) for mode in modes}
    for b, Lb in enumerate(lengths):
        for k in range(K):
            if b in (0, 1) and k == 0:
                continue
            batch.target[b, k, Lb, (7 * b + 3 * k) % batch.V] = float("nan") if k % 2 == 0 else float("inf")
    for mode in modes:
        gpu = P.gpu_run(mode, batch)
        ref = P.oracle_run(mode, batch)
        _compare_both(mode, batch, ref, f"leaves/{mode}")
        st, c = ref["req_status"], clean[mode]
        assert (c["req_status"] == 0).all()
        if mode == "greedy":
            # greedy ends at a leaf only where a draft matches to its end,
            # and reads that leaf alone
            tok = batch.tokens.cpu().numpy()
            ended = 0
            for b, Lb in enumerate(lengths):
                if c["accept_len"][b] < Lb:
                    assert st[b] == 0
                    for key in ("accept_len", "accept_draft", "out_token"):
                        assert ref[key][b] == c[key][b], (mode, b, key)
                else:
                    ended += 1
                    ks = int(c["accept_draft"][b])
                    owner = min(k2 for k2 in range(K) if (tok[b, k2, :Lb] == tok[b, ks, :Lb]).all())
                    assert st[b] == (0 if b in (0, 1) and owner == 0 else 4), (b, owner)
            continue
        assert st[0] == 0 and st[1] == 0 and st[2] == 4
        assert gpu["accept_len"][0] == 3 and gpu["accept_len"][1] == 2
        short = [b for b in range(3, len(lengths)) if c["accept_len"][b] < lengths[b]]
        assert short, "the fixture should stop short somewhere"
        for b in range(3, len(lengths)):
            if b in short:
                assert st[b] == 0
                for key in ("accept_len", "accept_draft", "out_token"):
                    assert ref[key][b] == c[key][b], (mode, b, key)
            else:
                assert st[b] == 4
        for b in np.nonzero(st)[0]:
            assert gpu["residual_mass"][b] == 0.0 and (gpu["accept_prob"][b] == 0).all()


def test_concurrent_calls_on_two_streams():
    # two calls with their own outputs and workspaces, queued on two streams
    # without a synchronisation between them, give what they give alone: a
    # node kernel's CTAs take work only while running, so a parent is always
    # held by a running CTA whatever share of the GPU the other call has
    a = W.make("mixed-B256-K8-L8-V151936-bf16", DEV, B=24, V=15197, seed=71)
    b = W.make("block-B128-K1-L5-V128256-bf16", DEV, B=24, seed=72)
    jobs = [(a, "multidraft"), (b, "block"), (a, "token"), (b, "token")]
    alone = [P.gpu_run(m, x) for x, m in jobs]
    outs = [binding.Outputs(m, x.B, x.K, x.L, x.V, x.target.device) for x, m in jobs]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    torch.cuda.synchronize()
    for i, (x, m) in enumerate(jobs):
        with torch.cuda.stream(streams[i % 2]):
            sdv.verify(m, x.target, x.draft, x.tokens, x.lengths, x.accept_u, x.sample_u, x.temperature, V=x.V,
                       out=outs[i])
    torch.cuda.synchronize()
    for i, (x, m) in enumerate(jobs):
        got = {k: (None if v is None else v.cpu().numpy()) for k, v in outs[i].as_dict().items()}
        for k, v in alone[i].items():
            if v is None:
                continue
            np.testing.assert_array_equal(got[k], v, err_msg=f"job {i} ({m}): {k}")


def test_deterministic():
    batch = W.make("mixed-B256-K8-L8-V151936-bf16", DEV, B=8, V=30011)
    for mode, kw in (("token", {}), ("multidraft", {}), ("multidraft", dict(accept_prob=False))):
        a, b = P.gpu_run(mode, batch, **kw), P.gpu_run(mode, batch, **kw)
        for key in a:
            if a[key] is not None:
                np.testing.assert_array_equal(a[key], b[key])


def test_full_size_calls_repeat_bit_for_bit():
    """The headline batch at full size, in the launch configuration the bench
    times (the decision kernel overlapping the node kernel's tail, nodes
    handed out by a global counter): repeated calls on the same inputs give
    the same bits, in every rule that runs the node kernel.  A dependence on
    which CTA took which node, or on the timing of the weights' flags and
    the node counts, would show here."""
    batch = W.make("mixed-B256-K8-L8-V151936-bf16", DEV)
    stream = torch.cuda.current_stream()
    for mode, ap in (("multidraft", False), ("multidraft", True), ("token", True), ("kseq", True)):
        out = binding.Outputs(mode, batch.B, batch.K, batch.L, batch.V, DEV, accept_prob=ap)
        ref = None
        for _ in range(8):
            sdv.verify(mode, batch.target, batch.draft, batch.tokens, batch.lengths, batch.accept_u, batch.sample_u,
                       batch.temperature, V=batch.V, out=out, stream=stream)
            torch.cuda.synchronize()
            got = {k: v.cpu().numpy().copy() for k, v in out.as_dict().items() if v is not None}
            assert int(got["device_status"][0]) == 0, mode
            if ref is None:
                ref = got
            else:
                for k in ref:
                    np.testing.assert_array_equal(ref[k], got[k], err_msg=f"{mode} accept_prob={ap} {k}")


@pytest.mark.parametrize("name,kw,T", SMALL[3:])
def test_skipping_last_sweeps_keeps_every_output(name, kw, T):
    """Without accept_prob the block rules skip the last sweep of nodes whose
    test must fail and of the root: every other output is bit for bit the
    one of the call with accept_prob, except residual_mass where the end
    node is the root (summed in another order by the draw pass)."""
    batch = W.make(name, DEV, temperature=T, **kw)
    for mode in ("block", "multidraft") if batch.K == 1 else ("multidraft",):
        full, lazy = P.gpu_run(mode, batch), P.gpu_run(mode, batch, accept_prob=False)
        for key in ("accept_len", "accept_draft", "out_token", "device_status"):
            np.testing.assert_array_equal(full[key], lazy[key], err_msg=key)
        at_root = full["accept_len"] == 0
        np.testing.assert_array_equal(full["residual_mass"][~at_root], lazy["residual_mass"][~at_root])
        np.testing.assert_allclose(full["residual_mass"][at_root], lazy["residual_mass"][at_root], atol=1e-6, rtol=0)


# The node kernel streams rows in chunks of 768 16-byte units (6144 bf16 or
# 3072 fp32 logits: 12 consumer warps of 64 contiguous units each):
# vocabularies at and around those boundaries, a tail chunk that only some
# warps reach, and a tail unit that only part of a warp's lanes reach; and
# the same around the 8192-logit boundary of 16-warp chunks, which now fall
# inside a chunk.
@pytest.mark.parametrize("V,dtype", [(6143, "bf16"), (6144, "bf16"), (6145, "bf16"), (6144 + 64 * 8, "bf16"),
                                     (6144 + 40 * 8 + 3, "bf16"), (12288, "bf16"), (12288 + 11 * 64 * 8 + 5, "bf16"),
                                     (3071, "f32"), (3072, "f32"), (3073, "f32"), (3072 + 64 * 4 + 1, "f32"),
                                     (8191, "bf16"), (8192, "bf16"), (8193, "bf16"), (4096, "f32")])
def test_chunk_boundaries(V, dtype):
    batch = W.make("mixed-B256-K8-L8-V151936-bf16", DEV, B=4, K=4, L=3, V=V, dtype=dtype)
    for mode in ("token", "multidraft"):
        _compare_both(mode, batch, P.oracle_run(mode, batch), f"V={V}/{dtype}/{mode}")


# Seeds on which an earlier build drifted from the oracle beyond 1e-5:
# a node weight below the complement's resolution raised again down the
# chain (block seed 100, multi-draft seed 110 at T = 0.1), and a ratio
# P(x)/Q(x) within 6e-8 of 1 whose complement was dropped (block seed 318
# at T = 0.1).  Every request, with and without accept_prob.
@pytest.mark.parametrize("name,seed,T,mode", [
    ("block-B128-K1-L5-V128256-bf16", 100, 0.7, "block"),
    ("block-B128-K1-L5-V128256-bf16", 318, 0.1, "block"),
    ("multidraft-B32-K4-L4-V32000-f32", 110, 0.1, "multidraft"),
])
def test_numerically_hard_seeds(name, seed, T, mode):
    batch = W.make(name, DEV, seed=seed, temperature=T)
    _compare_both(mode, batch, P.oracle_run(mode, batch), f"{name}/seed {seed}/T={T}/{mode}",
                  workload=f"{name} (hard seeds)")


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("V", [262143, 262144])
def test_largest_vocabulary(dtype, V):
    # the library's largest vocabulary (SDV_MAX_V) and a ragged one below it
    batch = W.make("multidraft-B32-K4-L4-V32000-f32", DEV, B=3, K=3, L=2, V=V, dtype=dtype, temperature=0.8)
    for mode in MODES_K + ["kseq"]:
        _compare_both(mode, batch, P.oracle_run(mode, batch), f"V={V}/{dtype}/{mode}")


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_degenerate_rows(dtype):
    """Rows whose maximum ties across lanes and chunks, moves every chunk,
    or sits at either end, and rows filtered to -inf (half the vocabulary,
    or all but three tokens): the online normaliser's set-aside and exact
    paths, against the oracle."""
    V = 40007
    batch = W.make("mixed-B256-K8-L8-V151936-bf16", DEV, B=14, K=3, L=3, V=V, dtype=dtype)
    for b in range(batch.B):
        t = P.pattern_row(b % 7, V).to(batch.target.dtype).to(DEV)
        d = P.pattern_row((b // 7 + b + 2) % 7, V).to(batch.draft.dtype).to(DEV)
        batch.target[b, :, :, :V] = t
        batch.draft[b, :, :, :V] = d
    for mode in ("token", "multidraft"):
        _compare_both(mode, batch, P.oracle_run(mode, batch), f"degenerate/{dtype}/{mode}")


@pytest.mark.parametrize("mode,K,ap", [("token", 1, True), ("token", 2, True), ("block", 1, True),
                                       ("multidraft", 2, True), ("block", 1, False), ("multidraft", 2, False)])
def test_sampled_outputs_follow_exact_law(mode, K, ap):
    """Chi-square of the GPU's (tau, k*, token) over many requests sharing
    logits and drafts but not uniforms, against the exact law the oracle
    integrates (tiny vocabulary)."""
    from scipy.stats import chi2
    import oracle
    V, L, N = 4, 2, 200000
    rng = np.random.default_rng(17)
    tgt = rng.normal(0, 1.2, (1, K, L + 1, V)).astype(np.float32)
    dft = (tgt[:, :, :L] + rng.normal(0, 1.0, (1, K, L, V))).astype(np.float32)
    tok = rng.integers(0, V, (1, K, L)).astype(np.int32)
    if K > 1:
        tgt[:, 1:, 0] = tgt[:, :1, 0]
        dft[:, 1:, 0] = dft[:, :1, 0]
    law = oracle.exact_outcomes(mode, oracle.Problem(tgt, dft, tok, None, np.zeros((1, K, L)),
                                                     np.zeros((1, K, L + 1)), 1.0)).ravel()
    dev = torch.device(DEV)
    rep = lambda a: torch.as_tensor(a).to(dev).expand((N,) + a.shape[1:]).contiguous()
    g = torch.Generator(device=dev).manual_seed(5)
    out = P.sdv.verify(mode, rep(P.pad8(tgt)), rep(P.pad8(dft)), rep(tok), None,
                       torch.rand((N, K, L), generator=g, device=dev),
                       torch.rand((N, K, L + 1), generator=g, device=dev), 1.0, V=V, accept_prob=ap)
    torch.cuda.synchronize()
    code = ((out["accept_len"].long() * K + out["accept_draft"].long()) * V + out["out_token"].long())
    counts = torch.bincount(code, minlength=law.size).cpu().numpy()
    keep = law * N >= 5
    assert counts[~keep].sum() <= max(10, 3 * law[~keep].sum() * N + 3)
    exp = law[keep] * N
    stat = float(((counts[keep] - exp) ** 2 / exp).sum())
    assert chi2.sf(stat, keep.sum() - 1) > 1e-3, (stat, keep.sum())


FULL = [
    ("token-B4-K1-L4-V1024-f32", [None]),
    ("token-greedy-B64-K1-L5-V32000-bf16", [0.0, 1.0]),
    ("block-B128-K1-L5-V128256-bf16", [None]),
    ("multidraft-B32-K4-L4-V32000-f32", [0.1, 0.4, 0.7]),
    ("mixed-B256-K8-L8-V151936-bf16", [None]),
]


def test_kseq_low_temperature_rho_is_valid():
    """K-SEQ at T = 0.1.  Where P and Q are both nearly one-hot on the same
    token, gamma(beta(rho)) - rho stays within ~1e-6 over a range of rho, so
    an fp32 search and the oracle's fp64 search stop at different points of
    that range.  Check instead that the GPU's rho, recovered from its
    acceptance probabilities (a = P(y) / (rho Q(y)) when a < 1), qualifies
    in fp64: gamma(beta(rho)) <= rho to within 1e-6 (the emitted token then
    follows P up to that clamp)."""
    batch = W.make("multidraft-B32-K4-L4-V32000-f32", DEV, B=6, V=3203, temperature=0.1)
    gpu = P.gpu_run("kseq", batch)
    assert int(gpu["device_status"][0]) == 0
    T, V = batch.temperature, batch.V
    checked = 0
    for b in range(batch.B):
        Lb = int(batch.lengths[b])
        tok = batch.tokens[b].cpu().numpy()
        for j in range(Lb):
            for k in range(batch.K):
                if any((tok[k2, :j] == tok[k, :j]).all() for k2 in range(k)):
                    continue  # not the node's owner
                n = sum(1 for k2 in range(batch.K) if (tok[k2, :j] == tok[k, :j]).all())
                lt = batch.target[b, k, j, :V].double().cpu().numpy()
                ld = batch.draft[b, k, j, :V].double().cpu().numpy()
                Pd = np.exp((lt - lt.max()) / T); Pd /= Pd.sum()
                Qd = np.exp((ld - ld.max()) / T); Qd /= Qd.sum()
                y = int(tok[k, j])
                a = float(gpu["accept_prob"][b, k, j])
                if not (1e-6 < a < 1.0) or n == 1:
                    continue
                rho = Pd[y] / (a * Qd[y])
                beta = np.minimum(Qd, Pd / rho).sum()
                gamma = -np.expm1(n * np.log1p(-min(beta, 1.0))) / beta
                assert 1.0 - 1e-6 <= rho <= n * (1 + 1e-6), (b, j, k, rho)
                assert gamma <= rho + 1e-6, (b, j, k, rho, gamma - rho)
                checked += 1
    assert checked > 0


def test_kseq_full_size():
    """K-SEQ on the mixed batch at full size (the launch configuration the
    bench times), every request against the oracle."""
    batch = W.make(W.HEADLINE, DEV)
    P.compare(P.gpu_run("kseq", batch), P.oracle_run("kseq", batch), "mixed/kseq", workload=W.HEADLINE + " (K-SEQ)")


@pytest.mark.parametrize("name,temps", FULL)
def test_full_size_parity(name, temps):
    """The workloads at their full sizes, in the launch configuration the
    bench times; the oracle checks every request of every mode and
    temperature, and the workload's near-margin mismatches together must
    stay below 1e-4 of its decisions."""
    before = dict(P.LEDGER.get(name, {}))
    for T in temps:
        batch = W.make(name, DEV, temperature=T)
        for mode in _modes(batch):
            _compare_both(mode, batch, P.oracle_run(mode, batch), f"{name}/T={T}/{mode}", workload=name)
        del batch
        torch.cuda.empty_cache()
    e = {k: v - before.get(k, 0) for k, v in P.LEDGER[name].items()}
    print(f"{name}: {e['requests']} requests, {e['decisions']} decisions, {e['near_margin']} near-margin, "
          f"{e['mismatches']} mismatched")
    assert e["mismatches"] == 0 or e["mismatches"] < 1e-4 * e["decisions"], e


@pytest.mark.parametrize("mode", ["multidraft", "token", "greedy", "kseq"])
def test_copy_read_rows_is_all_verification_needs(mode):
    """Copy only the rows verification reads (sdv_copy_read_rows) from host
    memory into NaN-filled device tensors: the results equal those of the
    fully copied batch, bit for bit."""
    import dataclasses
    import draft_verification_row_gb300 as sdv
    batch = W.make("mixed-B256-K8-L8-V151936-bf16", DEV, B=16, V=9001)
    full = P.gpu_run(mode, batch)
    ht, hd = batch.target.cpu().pin_memory(), batch.draft.cpu().pin_memory()
    tok, lens = batch.tokens.cpu(), batch.lengths.cpu()
    t2 = torch.full_like(batch.target, float("nan"))
    d2 = torch.full_like(batch.draft, float("nan"))
    n = sdv.copy_read_rows(ht, hd, tok, lens, t2, d2, V=batch.V)
    torch.cuda.synchronize()
    assert n == sdv.read_rows_bytes(tok, lens, batch.V, batch.stride, batch.target.dtype)
    assert n < batch.target.numel() * 2 + batch.draft.numel() * 2
    part = P.gpu_run(mode, dataclasses.replace(batch, target=t2, draft=d2))
    assert int(part["device_status"][0]) == 0
    for key in ("accept_len", "accept_draft", "out_token", "accept_prob", "residual_mass"):
        np.testing.assert_array_equal(full[key], part[key])


def test_gather_read_rows_matches_the_copy():
    """The GPU-side gather of the rows verification reads (from pinned,
    device-mapped host tensors) writes exactly the rows the host-side copy
    does; verification from them equals the full batch's."""
    import dataclasses
    import draft_verification_row_gb300 as sdv
    batch = W.make("mixed-B256-K8-L8-V151936-bf16", DEV, B=16, V=9001)
    ht, hd = batch.target.cpu().pin_memory(), batch.draft.cpu().pin_memory()
    a_t, a_d = torch.full_like(batch.target, float("nan")), torch.full_like(batch.draft, float("nan"))
    b_t, b_d = torch.full_like(batch.target, float("nan")), torch.full_like(batch.draft, float("nan"))
    sdv.copy_read_rows(ht, hd, batch.tokens.cpu(), batch.lengths.cpu(), a_t, a_d, V=batch.V)
    sdv.gather_read_rows(ht, hd, batch.tokens, batch.lengths, b_t, b_d, V=batch.V)
    torch.cuda.synchronize()
    # NaN == NaN for the untouched rows: compare the bits
    assert torch.equal(a_t.view(torch.int16), b_t.view(torch.int16))
    assert torch.equal(a_d.view(torch.int16), b_d.view(torch.int16))
    full = P.gpu_run("multidraft", batch)
    part = P.gpu_run("multidraft", dataclasses.replace(batch, target=b_t, draft=b_d))
    for key in ("accept_len", "accept_draft", "out_token", "accept_prob", "residual_mass"):
        np.testing.assert_array_equal(full[key], part[key])


@pytest.mark.parametrize("mode", ["multidraft", "token", "greedy", "kseq"])
def test_inner_rows_with_leaves_read_from_the_host(mode):
    """sdv_gather_inner_rows brings every row but the leaves' target rows;
    sdv_verify_leaves_apart reads the leaf rows the decisions end at from the
    pinned host tensor itself.  The results equal the full batch's, bit for
    bit, and the device tensor's leaf rows (NaN here) are never read."""
    import draft_verification_row_gb300 as sdv
    lengths = [3, 1, 2, 3, 0, 3, 2, 1, 3, 3, 2, 3]
    batch = W.make("mixed-B256-K8-L8-V151936-bf16", DEV, B=len(lengths), K=4, L=3, V=9001, lengths=lengths)
    batch.accept_u[:4] = 0.0  # these requests accept everything: their decisions end at leaves
    ht, hd = batch.target.cpu().pin_memory(), batch.draft.cpu().pin_memory()
    t = torch.full_like(batch.target, float("nan"))
    d = torch.full_like(batch.draft, float("nan"))
    sdv.gather_read_rows(ht, hd, batch.tokens, batch.lengths, t, d, V=batch.V, leaves=False)
    torch.cuda.synchronize()
    for b, Lb in enumerate(lengths):  # no leaf row was brought
        assert torch.isnan(t[b, :, Lb].float()).all()
    full = P.gpu_run(mode, batch)
    out = sdv.verify(mode, t, d, batch.tokens, batch.lengths, batch.accept_u, batch.sample_u, batch.temperature,
                     V=batch.V, leaf_target=ht)
    torch.cuda.synchronize()
    assert int(out["device_status"].item()) == 0
    for key in ("accept_len", "accept_draft", "out_token", "accept_prob", "residual_mass"):
        np.testing.assert_array_equal(full[key], out[key].cpu().numpy(), err_msg=key)
    ends_at_leaf = int((full["accept_len"] == np.array(lengths)).sum())
    assert ends_at_leaf >= (1 if mode == "greedy" else 4)  # greedy: at least the length-0 request
