"""The non-allocating SpecTr-GBV entry point, sdv_verify_multidraft_static.

Some callers cannot allocate device memory: a plugin whose host framework
owns all device memory and hands it only input and output buffers, code
running inside a device allocator's own hooks, or a serving loop that
forbids cudaMalloc because it can synchronise the device.  For them the
library takes the scratch from a fixed array of its own.  These tests call
that entry point through the C-ABI twice in a row, on two differently
shaped batches (so the second call finds the first call's leftovers in the
shared array), and check each result against sdv_verify_multidraft run
with a workspace the caller allocated.
"""
import ctypes

import numpy as np
import pytest
import torch

from draft_verification_row_gb300 import workloads as W

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
SDV_ERR_WORKSPACE = 5


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    import draft_verification_row_gb300 as sdv
    h = sdv.lib()
    fn = h.sdv_verify_multidraft_static
    fn.restype = ctypes.c_int
    fn.argtypes = ([ctypes.c_int] * 4 + [ctypes.c_longlong, ctypes.c_int, ctypes.c_float]
                   + [ctypes.c_void_p] * 6 + [ctypes.c_void_p] * 6 + [ctypes.c_void_p])
    return h


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _static_call(h, batch):
    dev = batch.target.device
    out = {
        "accept_len": torch.full((batch.B,), -7, dtype=torch.int32, device=dev),
        "accept_draft": torch.full((batch.B,), -7, dtype=torch.int32, device=dev),
        "out_token": torch.full((batch.B,), -7, dtype=torch.int32, device=dev),
        "accept_prob": torch.full((batch.B, batch.K, batch.L), -1.0, dtype=torch.float32, device=dev),
        "residual_mass": torch.full((batch.B,), -1.0, dtype=torch.float32, device=dev),
        "device_status": torch.full((1,), -1, dtype=torch.int32, device=dev),
    }
    stream = torch.cuda.current_stream(dev)
    rc = h.sdv_verify_multidraft_static(
        batch.B, batch.K, batch.L, batch.V, batch.stride, 1 if batch.dtype == "bf16" else 0, batch.temperature,
        _p(batch.target), _p(batch.draft), _p(batch.tokens), _p(batch.lengths), _p(batch.accept_u),
        _p(batch.sample_u), _p(out["accept_len"]), _p(out["accept_draft"]), _p(out["out_token"]),
        _p(out["accept_prob"]), _p(out["residual_mass"]), _p(out["device_status"]),
        ctypes.c_void_p(stream.cuda_stream))
    assert rc == 0, f"sdv_verify_multidraft_static returned {rc}"
    return out


def _workspace_call(batch):
    import draft_verification_row_gb300 as sdv
    return sdv.verify("multidraft", batch.target, batch.draft, batch.tokens, batch.lengths, batch.accept_u,
                      batch.sample_u, batch.temperature, V=batch.V)


def _same(a, b):
    # the same kernels on the same inputs: bit for bit, floats included
    torch.cuda.synchronize()
    a = {k: v.cpu().numpy() for k, v in a.items() if v is not None}
    b = {k: v.cpu().numpy() for k, v in b.items() if v is not None}
    for key in ("accept_len", "accept_draft", "out_token", "device_status", "accept_prob", "residual_mass"):
        np.testing.assert_array_equal(a[key], b[key], err_msg=key)


def test_matches_workspace_entry_point_on_two_calls(lib):
    first = W.make("mixed-B256-K8-L8-V151936-bf16", DEV, B=6, K=4, L=4, V=5003)
    second = W.make("multidraft-B32-K4-L4-V32000-f32", DEV, B=5, K=3, L=3, V=3001, temperature=0.4)
    got1 = _static_call(lib, first)
    got2 = _static_call(lib, second)
    _same(got1, _workspace_call(first))
    _same(got2, _workspace_call(second))


def test_rejects_problems_beyond_the_fixed_scratch(lib):
    """A batch whose scratch would not fit the fixed array is refused before
    anything is launched (no pointer is touched, so NULLs are fine)."""
    import draft_verification_row_gb300 as sdv
    B, K, L, V = 20000, 16, 16, 1024
    assert sdv.workspace_bytes("multidraft", B, K, L, V) > 4 << 20
    args = [B, K, L, V, V, 0, 1.0] + [None] * 12 + [None]
    assert lib.sdv_verify_multidraft_static(*args) == SDV_ERR_WORKSPACE
