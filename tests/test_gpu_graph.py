"""Verification and sampling calls captured in a CUDA graph and replayed.

A serving loop verifies one batch per step with the same shapes, so it can
capture the call once and replay it: the library's calls are asynchronous,
allocate nothing and never synchronise, so every launch and memset lands in
the graph.  Each test captures a call on one batch, replays it, refills the
captured input tensors with a second batch and replays again: both replays
must equal direct calls on the same inputs, bit for bit.
"""
import ctypes

import numpy as np
import pytest
import torch

import draft_verification_row_gb300 as sdv
from draft_verification_row_gb300 import binding
from draft_verification_row_gb300 import workloads as W

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
FIELDS = ("target", "draft", "tokens", "lengths", "accept_u", "sample_u")


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _capture(fn):
    # one call outside the capture first (as torch asks of captured code)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        fn()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    return g


def _host(d):
    return {k: None if v is None else v.cpu().numpy().copy() for k, v in d.items()}


def _same(a, b, what):
    for k in a:
        if a[k] is None:
            assert b[k] is None, f"{what}: {k}"
            continue
        np.testing.assert_array_equal(a[k], b[k], err_msg=f"{what}: {k}")


def _inputs(batch):
    return {k: None if getattr(batch, k) is None else getattr(batch, k).clone() for k in FIELDS}


def _refill(inp, batch):
    for k in FIELDS:
        if inp[k] is not None:
            inp[k].copy_(getattr(batch, k))


@pytest.mark.parametrize("name,mode,ap", [
    ("mixed-B256-K8-L8-V151936-bf16", "multidraft", False),
    ("mixed-B256-K8-L8-V151936-bf16", "multidraft", True),
    ("mixed-B256-K8-L8-V151936-bf16", "token", True),
    ("mixed-B256-K8-L8-V151936-bf16", "greedy", True),
    ("mixed-B256-K8-L8-V151936-bf16", "kseq", True),
    ("block-B128-K1-L5-V128256-bf16", "block", False),
    ("multidraft-B32-K4-L4-V32000-f32", "multidraft", True),
])
def test_verification_replays_like_direct_calls(name, mode, ap):
    small = dict(B=16, V=15197) if name.startswith("mixed") else dict(B=12)
    a = W.make(name, DEV, seed=31, **small)
    b = W.make(name, DEV, seed=32, **small)
    inp = _inputs(a)
    out = binding.Outputs(mode, a.B, a.K, a.L, a.V, a.target.device, accept_prob=ap)

    def call():
        sdv.verify(mode, inp["target"], inp["draft"], inp["tokens"], inp["lengths"], inp["accept_u"],
                   inp["sample_u"], a.temperature, V=a.V, out=out, accept_prob=ap)

    g = _capture(call)
    for batch, what in ((a, "first batch"), (b, "refilled inputs")):
        _refill(inp, batch)
        g.replay()
        torch.cuda.synchronize()
        got = _host(out.as_dict())
        ref = _host(sdv.verify(mode, batch.target, batch.draft, batch.tokens, batch.lengths, batch.accept_u,
                               batch.sample_u, batch.temperature, V=batch.V, accept_prob=ap))
        torch.cuda.synchronize()
        _same(got, ref, f"{name}/{mode}/{what}")
        assert int(got["device_status"][0]) == 0


def test_sampling_replays_like_direct_calls():
    a = W.make(W.HEADLINE, DEV, seed=31, B=16)
    b = W.make(W.HEADLINE, DEV, seed=32, B=16)
    rows = a.draft[:, :, 0, :].reshape(a.B * a.K, a.stride).contiguous()
    g0 = torch.Generator(device=DEV)
    g0.manual_seed(5)
    u = torch.rand((rows.shape[0], 3), generator=g0, device=DEV)
    tokens = torch.empty((rows.shape[0], 3), dtype=torch.int32, device=DEV)
    status = torch.empty(1, dtype=torch.int32, device=DEV)

    def call():
        sdv.sample_rows(rows, 3, u, a.temperature, V=a.V, tokens=tokens, device_status=status)

    g = _capture(call)
    for batch in (a, b):
        rows.copy_(batch.draft[:, :, 0, :].reshape(batch.B * batch.K, batch.stride))
        g.replay()
        torch.cuda.synchronize()
        got = tokens.cpu().numpy().copy()
        ref, st = sdv.sample_rows(rows.clone(), 3, u, batch.temperature, V=batch.V)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(got, ref.cpu().numpy())
        assert int(status.item()) == 0 and int(st.item()) == 0


def test_non_allocating_entry_replays_like_direct_calls():
    h = sdv.lib()
    fn = h.sdv_verify_multidraft_static
    fn.restype = ctypes.c_int
    fn.argtypes = ([ctypes.c_int] * 4 + [ctypes.c_longlong, ctypes.c_int, ctypes.c_float]
                   + [ctypes.c_void_p] * 6 + [ctypes.c_void_p] * 6 + [ctypes.c_void_p])
    a = W.make("multidraft-B32-K4-L4-V32000-f32", DEV, seed=31, B=12)
    b = W.make("multidraft-B32-K4-L4-V32000-f32", DEV, seed=32, B=12)
    inp = _inputs(a)
    out = {k: torch.empty(s, dtype=dt, device=DEV) for k, s, dt in (
        ("accept_len", (a.B,), torch.int32), ("accept_draft", (a.B,), torch.int32),
        ("out_token", (a.B,), torch.int32), ("accept_prob", (a.B, a.K, a.L), torch.float32),
        ("residual_mass", (a.B,), torch.float32), ("device_status", (1,), torch.int32))}
    p = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())

    def call():
        stream = torch.cuda.current_stream(DEV)
        rc = fn(a.B, a.K, a.L, a.V, a.stride, 1 if a.dtype == "bf16" else 0, a.temperature,
                p(inp["target"]), p(inp["draft"]), p(inp["tokens"]), p(inp["lengths"]), p(inp["accept_u"]),
                p(inp["sample_u"]), p(out["accept_len"]), p(out["accept_draft"]), p(out["out_token"]),
                p(out["accept_prob"]), p(out["residual_mass"]), p(out["device_status"]),
                ctypes.c_void_p(stream.cuda_stream))
        assert rc == 0

    g = _capture(call)
    for batch, what in ((a, "first batch"), (b, "refilled inputs")):
        _refill(inp, batch)
        g.replay()
        torch.cuda.synchronize()
        got = _host(out)
        ref = _host(sdv.verify("multidraft", batch.target, batch.draft, batch.tokens, batch.lengths,
                               batch.accept_u, batch.sample_u, batch.temperature, V=batch.V))
        torch.cuda.synchronize()
        _same(got, ref, f"static/{what}")
